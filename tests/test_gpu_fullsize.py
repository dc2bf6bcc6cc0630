"""Parity at the workloads' full sizes (needs a GB300; slow).

* embedding + lm_head, vocab 151936 x 1024, 8192 tokens: the embedding is
  compared bit for bit on every row at 1/2/4 shards; the full [8192, 151936]
  logits on 64 rows spread over the batch (the oracle recomputes those rows).
* the 28-layer decode step for 64 sequences with synthetic cache history:
  every sequence through the oracle.
* the 28-layer two-shard model, prefill 8 x 2048 then 128 decode steps with
  forced decode inputs:
  - every sequence at the prefill and at decode steps 0, 63 and 127, the
    oracle running each sequence's 2048 prompt tokens plus its 128 forced
    tokens as one causal prefill (position 2048 + t of it is decode step t);
  - sequence 0 at every step through the oracle's own decode path;
  - the bench's CUDA-graph path (greedy feedback on the device) equal bit for
    bit to the same kernels launched one by one.

Tolerances are those of tests/test_gpu_model.py: the stated 2e-2, or twice the
model's fp32-accumulation noise floor over the same rows where that is
higher (28 layers of random-init weights: about 0.1 on the decode logits),
and greedy argmax agreement on at least 99 % of the decisive rows.
"""
import numpy as np
import pytest
import torch

import oracle as O
import seeded_inputs as si
from tests._util import assert_within_ulps, to_np
from tests.model_parity import forced_tokens, oracle_decode_layerwise, oracle_prefill_layerwise
from tests.test_gpu_model import Parity, check_bf16_step

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_transformer_forward_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def oracle_weights():
    """The 28-layer checkpoint as the oracle holds it (independent of the shard count)."""
    return O.load_weights(si.QWEN3_0_6B)


def test_embed_and_lm_head_full_size(oracle_weights):
    from qwen3_transformer_forward_gb300 import _lib as L
    w = si.workload("embed_lm_head")
    m = w.model
    table = si.checkpoint_tensor(m, "embed_tokens", device="cuda")
    ids = si.embed_ids(m, w.n_tokens, w.boundary_fraction)
    tab64 = oracle_weights.embed
    for tp in w.tps:
        out = torch.empty(w.n_tokens, m.hidden, dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        L.embed_vocab(ids.cuda(), table, tp, out, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert np.array_equal(to_np(out), O.vocab_parallel_embedding(ids.numpy(), tab64, tp)), tp
    hidden = si.normal(0, "embed_lm_head.hidden", (w.n_tokens, m.hidden), 1.0, "bf16")
    # 64 rows: both ends, the 128-row tile edges near them and rows spread over the batch
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 8063, 8064, 8190, 8191],
                                     np.linspace(2, 8189, 56).astype(np.int64)]))
    assert len(rows) == 64
    h = hidden.double().numpy()[rows]
    acc = 2.0 ** -18 * (np.abs(h) @ np.abs(tab64).T)
    for tp in w.tps:
        logits = torch.empty(w.n_tokens, m.vocab, dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(L.lm_head_workspace_size(w.n_tokens, m.vocab, m.hidden, tp, torch.bfloat16),
                         dtype=torch.uint8, device="cuda")
        L.lm_head(hidden.cuda(), None, w.n_tokens, table, tp, logits, None, ws)
        torch.cuda.synchronize()
        L.device_error()
        ref = O.compute_logits(m.replace(tp=tp), tab64, h, tp)
        got = to_np(logits[torch.from_numpy(rows).cuda()])
        assert_within_ulps(got, ref, 1.0, 0.9, f"lm_head tp{tp}", atol=acc)


def test_model_decode_64_sequences_full_size(oracle_weights):
    from qwen3_transformer_forward_gb300 import model as M
    from qwen3_transformer_forward_gb300 import _lib as L
    w = si.workload("model_decode")
    m = w.model
    ctx_lens = si.decode_context_lens(0, w.batch, w.ctx_low, w.ctx_high)
    batch = si.decode_batch(m, ctx_lens)
    params = M.load_params(m, device="cuda")
    kc = [torch.zeros(batch.num_slots, m.n_kv_heads, m.head_dim, dtype=torch.bfloat16, device="cuda")
          for _ in range(m.n_layers)]
    vc = [torch.zeros_like(kc[0]) for _ in range(m.n_layers)]
    hist = torch.cat([torch.arange(int(batch.seq_base[b]), int(batch.seq_base[b]) + ctx_lens[b] - 1)
                      for b in range(w.batch)]).cuda()
    for l in range(m.n_layers):
        kc[l][hist] = si.kv_history(m, l, "k", hist)
        vc[l][hist] = si.kv_history(m, l, "v", hist)
    fwd = M.Qwen3Forward(m, params, max_tokens=w.batch, num_slots=batch.num_slots, max_seqs=w.batch,
                         max_context=max(ctx_lens), kv_caches=(kc, vc))
    h = fwd.run_layers(M.to_device_decode(batch), decode=True).clone()
    logits, _ = fwd.compute_logits(h, None, w.batch)
    torch.cuda.synchronize()
    L.device_error()
    gh, gl = to_np(h), to_np(logits)
    del fwd, kc, vc
    torch.cuda.empty_cache()

    def history(l):
        # the seeded history generator, evaluated on the device for speed (its
        # values are bit-identical on CPU and GPU), then placed at its slots
        k = np.zeros((batch.num_slots, m.n_kv_heads, m.head_dim))
        v = np.zeros_like(k)
        rows = hist.cpu().numpy()
        k[rows] = si.kv_history(m, l, "k", hist).double().cpu().numpy()
        v[rows] = si.kv_history(m, l, "v", hist).double().cpu().numpy()
        return k, v

    oh, ol = oracle_decode_layerwise(m, oracle_weights, batch.ids.numpy(), batch.positions.numpy(),
                                     batch.context_lens.numpy(), batch.slot_mapping.numpy(),
                                     batch.seq_base.numpy(), batch.num_slots, history)
    par = Parity("model_decode_64")
    for b in range(w.batch):
        check_bf16_step(gl[b:b + 1], ol[b:b + 1], gh[b:b + 1], oh[b:b + 1], f"seq {b} ctx {ctx_lens[b]}", par)
    par.check()


def test_model_prefill_decode_full_size(oracle_weights):
    import bench
    from qwen3_transformer_forward_gb300 import model as M
    from qwen3_transformer_forward_gb300 import _lib as L
    wl = bench.Workload("cuda")
    m, seq_lens, S, B = wl.m, wl.seq_lens, wl.S, wl.B
    fwd = wl.fwd
    # (1) the kernels launched one by one, forced decode inputs
    forced = forced_tokens(m, S, B)
    hid, log = [], []
    h = fwd.run_layers(wl.pctx, decode=False)
    hid.append(to_np(h[wl.pctx.last_idx.long()]))
    lg, nt = fwd.compute_logits(h, wl.pctx.last_idx, B)
    log.append(to_np(lg))
    greedy0 = nt.clone()
    for s in range(S):
        ctx = M.DecodeContext(forced[s].cuda(), wl.dpos[s], wl.dcl[s], wl.dslots[s], wl.dbase, wl.max_context)
        h = fwd.run_layers(ctx, decode=True)
        hid.append(to_np(h))
        lg, _ = fwd.compute_logits(h, None, B)
        log.append(to_np(lg))
    torch.cuda.synchronize()
    L.device_error()
    # (2) the bench's graphs (greedy feedback) against the same kernels launched eagerly
    wl.capture()
    wl.step()
    torch.cuda.synchronize()
    gen_graph = wl.gen.clone()
    assert torch.equal(gen_graph[0], greedy0)
    y = fwd.run_layers(wl.pctx, decode=False)
    _, nt = fwd.compute_logits(y, wl.pctx.last_idx, B)
    eager = [nt.clone()]
    for s in range(S):
        ctx = M.DecodeContext(fwd.next_tokens[:B], wl.dpos[s], wl.dcl[s], wl.dslots[s], wl.dbase, wl.max_context)
        h = fwd.run_layers(ctx, decode=True)
        _, nt = fwd.compute_logits(h, None, B)
        eager.append(nt.clone())
    torch.cuda.synchronize()
    assert torch.equal(torch.stack(eager), gen_graph)
    del wl, fwd
    torch.cuda.empty_cache()

    ow = oracle_weights
    prompt = si.prefill_batch(m, seq_lens, extra_capacity=S).ids.numpy()
    cu = np.concatenate([[0], np.cumsum(seq_lens)])
    par = Parity("model_prefill_decode")
    # (3) every sequence: prompt + forced tokens as one causal prefill; its rows
    # at the last prompt token and at decode steps 0, 63 and 127
    steps = [0, 63, 127]
    ids = np.concatenate([np.concatenate([prompt[cu[b]:cu[b + 1]], forced[:, b].numpy()]) for b in range(B)])
    lens = [L0 + S for L0 in seq_lens]
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    rows = np.array([starts[b] + seq_lens[b] - 1 + k for b in range(B) for k in [0] + [1 + t for t in steps]])
    oh, ol = oracle_prefill_layerwise(m, ow, ids, lens, rows)
    for i, (b, k) in enumerate((b, k) for b in range(B) for k in [0] + [1 + t for t in steps]):
        what = f"seq {b} " + ("prefill" if k == 0 else f"decode step {k - 1}")
        check_bf16_step(log[k][b:b + 1], ol[i:i + 1], hid[k][b:b + 1], oh[i:i + 1], what, par)
    # (4) sequence 0 at every step through the oracle's decode path
    L0 = seq_lens[0]
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    cache = O.KVCache(m.n_layers, L0 + S, m.n_kv_heads, m.head_dim, m.tp)
    ctx = O.AttnContext(True, np.arange(L0), cu_seqlens=np.array([0, L0]))
    hh = O.model_forward(m, ow, prompt[:L0], np.arange(L0), ctx, cache, cos_sin)
    check_bf16_step(log[0][0:1], O.compute_logits(m, ow.embed, hh, m.tp, np.array([0, L0])), hid[0][0:1],
                    hh[-1:], "seq 0 prefill (decode path)", par)
    for s in range(S):
        pos = L0 + s
        dctx = O.AttnContext(False, np.array([pos]), seq_base=np.array([0]), context_lens=np.array([pos + 1]))
        hh = O.model_forward(m, ow, forced[s].numpy()[:1], np.array([pos]), dctx, cache, cos_sin)
        check_bf16_step(log[s + 1][0:1], O.compute_logits(m, ow.embed, hh, m.tp), hid[s + 1][0:1], hh,
                        f"seq 0 decode step {s} (decode path)", par)
    par.check()
