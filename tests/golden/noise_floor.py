"""Writes tests/golden/noise_floor.json: the oracle's own sensitivity to the
rounding that fp32 accumulation adds, for every multi-layer bf16 workload
the GPU parity tests compare.

Why: the bf16 model keeps its activations in bf16 and normalises them at
every layer (RMSNorm on the residual, QK-RMSNorm).  A single intermediate
value rounded to the neighbouring bf16 value changes the RMS of its row,
which shifts every normalised element of that row and flips the bf16
rounding of some of them; those flips spread the same way through the next
layer.  Any implementation whose GEMMs accumulate in fp32 instead of exactly
rounds a few outputs differently from the float64 oracle, so after a few
random-init layers its outputs differ from the oracle's by an amount set by
this spreading, not by the size of the first difference.

Measured here: the oracle run twice over the same rows, once as it is and
once with every Linear product (QKV, o_proj, gate_up, down, lm_head)
accumulated in fp32 -- numpy's float32 matmul on the same bf16 operands,
the row-parallel shard partials added in fp32 -- before the one rounding to
bf16.  That is what a tensor-core GEMM does; nothing else in the oracle
changes.  The recorded floor per workload: max and mean |difference| of the
logits and of the final hidden state over the rows the GPU test compares,
and the fraction of rows whose greedy argmax agrees.

Only oracle/ and the seeded input generators are used (no CUDA path).
Run from the repository root:

    python tests/golden/noise_floor.py [--workers 4] [--only NAME ...]
"""
from __future__ import annotations

import argparse
import json
import multiprocessing as mp
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

OUT = os.path.join(ROOT, "tests", "golden", "noise_floor.json")


# ----------------------------------------------------------------------------
# the perturbation: every Linear product accumulated in fp32
# ----------------------------------------------------------------------------

def _perturb(on: bool):
    import numpy as np
    import oracle as O
    import oracle.qwen3 as Q
    if not hasattr(Q, "_exact_linear"):
        Q._exact_linear, Q._exact_row = Q.linear, Q.row_parallel_linear
    if not on:
        Q.linear, Q.row_parallel_linear = Q._exact_linear, Q._exact_row
        return

    def linear(x, w, dtype):
        acc = np.asarray(x, dtype=np.float32) @ np.asarray(w, dtype=np.float32).T
        return O.round_to(acc.astype(np.float64), dtype)

    def row_parallel_linear(x_shards, w_full, tp, dtype):
        k_l = w_full.shape[1] // tp
        acc = None
        for r in range(tp):
            part = np.asarray(x_shards[r], dtype=np.float32) @ np.asarray(
                w_full[:, r * k_l:(r + 1) * k_l], dtype=np.float32).T
            acc = part if acc is None else acc + part
        return O.round_to(acc.astype(np.float64), dtype)
    Q.linear, Q.row_parallel_linear = linear, row_parallel_linear


def _both(fn):
    """(exact result, perturbed result) of fn() -> (hidden rows, logits rows)."""
    _perturb(False)
    a = fn()
    _perturb(True)
    try:
        b = fn()
    finally:
        _perturb(False)
    return a, b


# ----------------------------------------------------------------------------
# work units (each returns exact and perturbed (hidden, logits) of its rows)
# ----------------------------------------------------------------------------

_WEIGHTS = {}


def _weights(m, key):
    import oracle as O
    if key not in _WEIGHTS:
        _WEIGHTS.clear()
        _WEIGHTS[key] = O.load_weights(m)
    return _WEIGHTS[key]


def unit_small(name, over, seq_lens, steps, phases):
    """run_oracle on a small model (all sequences, the given phases)."""
    import numpy as np
    import seeded_inputs as si
    from tests.model_parity import forced_tokens, run_oracle
    m = si.QWEN3_0_6B.replace(**over)
    forced = forced_tokens(m, steps, len(seq_lens))
    w = _weights(m, name)

    def fn():
        t = run_oracle(m, seq_lens, steps, forced=forced, weights=w)
        return (np.concatenate([t.hidden[p] for p in phases]), np.concatenate([t.logits[p] for p in phases]))
    return _both(fn)


def unit_c4(b):
    """One sequence of the 64-sequence decode step, with its own cache history."""
    import numpy as np
    import torch
    import seeded_inputs as si
    from tests.model_parity import oracle_decode_layerwise
    w = si.workload("model_decode")
    m = w.model
    ctx_lens = si.decode_context_lens(0, w.batch, w.ctx_low, w.ctx_high)
    batch = si.decode_batch(m, ctx_lens)
    L = ctx_lens[b]
    slots = torch.arange(int(batch.seq_base[b]), int(batch.seq_base[b]) + L - 1)
    hist = [(si.kv_history(m, l, "k", slots).double().numpy(), si.kv_history(m, l, "v", slots).double().numpy())
            for l in range(m.n_layers)]

    def history(l):
        k = np.zeros((L, m.n_kv_heads, m.head_dim))
        v = np.zeros_like(k)
        k[:L - 1], v[:L - 1] = hist[l]
        return k, v
    ow = _weights(m, "qwen3_0_6b")

    def fn():
        return oracle_decode_layerwise(m, ow, batch.ids.numpy()[b:b + 1], np.array([L - 1]), np.array([L]),
                                       np.array([L - 1]), np.array([0]), L, history)
    return _both(fn)


def unit_c5_seq(b):
    """One sequence of the 8 x 2048 prefill + 128 forced decode steps, as one causal
    prefill of prompt + forced tokens: rows at the last prompt token and at decode
    steps 0, 63 and 127."""
    import numpy as np
    import seeded_inputs as si
    from tests.model_parity import forced_tokens, oracle_prefill_layerwise
    w = si.workload("model_prefill_decode")
    m, seq_lens, S = w.model, list(w.seq_lens), w.decode_steps
    forced = forced_tokens(m, S, len(seq_lens))
    prompt = si.prefill_batch(m, seq_lens, extra_capacity=S).ids.numpy()
    cu = np.concatenate([[0], np.cumsum(seq_lens)])
    ids = np.concatenate([prompt[cu[b]:cu[b + 1]], forced[:, b].numpy()])
    rows = np.array([seq_lens[b] - 1 + k for k in (0, 1, 64, 128)])
    ow = _weights(m, "qwen3_0_6b")
    return _both(lambda: oracle_prefill_layerwise(m, ow, ids, [len(ids)], rows))


def unit_c5_decode_path():
    """Sequence 0 through the oracle's decode path: the prefill, then all 128 steps."""
    import numpy as np
    import oracle as O
    import seeded_inputs as si
    from tests.model_parity import forced_tokens
    w = si.workload("model_prefill_decode")
    m, seq_lens, S = w.model, list(w.seq_lens), w.decode_steps
    forced = forced_tokens(m, S, len(seq_lens))
    prompt = si.prefill_batch(m, seq_lens, extra_capacity=S).ids.numpy()
    L0 = seq_lens[0]
    ow = _weights(m, "qwen3_0_6b")
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)

    def fn():
        cache = O.KVCache(m.n_layers, L0 + S, m.n_kv_heads, m.head_dim, m.tp)
        ctx = O.AttnContext(True, np.arange(L0), cu_seqlens=np.array([0, L0]))
        hh = O.model_forward(m, ow, prompt[:L0], np.arange(L0), ctx, cache, cos_sin)
        hs, ls = [hh[-1:]], [O.compute_logits(m, ow.embed, hh, m.tp, np.array([0, L0]))]
        for s in range(S):
            pos = L0 + s
            dctx = O.AttnContext(False, np.array([pos]), seq_base=np.array([0]), context_lens=np.array([pos + 1]))
            hh = O.model_forward(m, ow, forced[s].numpy()[:1], np.array([pos]), dctx, cache, cos_sin)
            hs.append(hh)
            ls.append(O.compute_logits(m, ow.embed, hh, m.tp))
        return np.concatenate(hs), np.concatenate(ls)
    return _both(fn)


SMALL3 = dict(vocab=8192, n_layers=3, gamma_sigma=0.1)
FUSED2 = dict(vocab=4096, n_layers=2, gamma_sigma=0.1)

# name -> list of (unit function, args); rows of all units are pooled per name
WORKLOADS = {
    # tests/test_gpu_model.py::test_small_bf16_model_prefill_and_decode: prefill and 3 decode steps
    "small3_tp1": [(unit_small, ("small3_tp1", dict(SMALL3, tp=1), [37, 130, 1, 64], 3, [0, 1, 2, 3]))],
    "small3_tp2": [(unit_small, ("small3_tp2", dict(SMALL3, tp=2), [37, 130, 1, 64], 3, [0, 1, 2, 3]))],
    # tests/test_gpu_decode_step.py::test_decode_step_against_oracle: the decode steps
    "fused2_gqa2_tp2_b5": [(unit_small, ("fused2_gqa2_tp2_b5", dict(FUSED2, tp=2), [37, 130, 1, 64, 300], 2,
                                         [1, 2]))],
    "fused2_gqa2_tp1_b1": [(unit_small, ("fused2_gqa2_tp1_b1", dict(FUSED2, tp=1), [1], 3, [1, 2, 3]))],
    "fused2_gqa1_tp2_b3": [(unit_small, ("fused2_gqa1_tp2_b3", dict(FUSED2, n_heads=8, n_kv_heads=8,
                                                                    intermediate=1024, tp=2), [20, 700, 129], 2,
                                         [1, 2]))],
    "fused2_gqa4_tp2_b16": [(unit_small, ("fused2_gqa4_tp2_b16", dict(FUSED2, n_heads=16, n_kv_heads=4, tp=2),
                                          [3 + 37 * i for i in range(16)], 2, [1, 2]))],
    # tests/test_gpu_fullsize.py
    "model_decode_64": [(unit_c4, (b,)) for b in range(64)],
    "model_prefill_decode": [(unit_c5_seq, (b,)) for b in range(8)] + [(unit_c5_decode_path, ())],
}


def _run(task):
    fn, args = task
    t0 = time.time()
    (h0, l0), (h1, l1) = fn(*args)
    return h0, l0, h1, l1, time.time() - t0


def main(argv=None):
    import numpy as np
    import oracle as O
    ap = argparse.ArgumentParser()
    ap.add_argument("--workers", type=int, default=4)
    ap.add_argument("--only", nargs="*", default=None)
    args = ap.parse_args(argv)
    names = args.only or list(WORKLOADS)
    result = {}
    if os.path.exists(OUT):
        with open(OUT) as f:
            result = json.load(f).get("workloads", {})
    ctx = mp.get_context("spawn")
    with ctx.Pool(args.workers) as pool:
        for name in names:
            t0 = time.time()
            parts = pool.map(_run, WORKLOADS[name], chunksize=1)
            h0 = np.concatenate([p[0] for p in parts])
            l0 = np.concatenate([p[1] for p in parts])
            h1 = np.concatenate([p[2] for p in parts])
            l1 = np.concatenate([p[3] for p in parts])
            dl, dh = np.abs(l1 - l0), np.abs(h1 - h0)
            agree = float(np.mean(O.greedy(l0) == O.greedy(l1)))
            result[name] = {"rows": int(l0.shape[0]), "logits_max": float(dl.max()), "logits_mean": float(dl.mean()),
                            "hidden_max": float(dh.max()), "hidden_mean": float(dh.mean()), "argmax_agreement": agree}
            print(name, result[name], f"{time.time() - t0:.0f} s", flush=True)
            with open(OUT, "w") as f:
                json.dump({"what": "oracle vs oracle with every Linear product accumulated in fp32 (float32 matmul) "
                                   "before its bf16 rounding (written by tests/golden/noise_floor.py)",
                           "workloads": result}, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main()
