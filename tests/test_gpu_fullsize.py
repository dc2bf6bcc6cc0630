"""Parity at the workloads' full sizes (needs a GB300; slow).

* embedding + lm_head, vocab 151936 x 1024, 8192 tokens: the embedding is
  compared bit for bit on every row at 1/2/4 shards; the full [8192, 151936]
  logits on sampled rows (the oracle recomputes those rows one by one).
* the 28-layer decode step for 64 sequences with synthetic cache history:
  sampled sequences (shortest, longest, one in between) through the oracle.
* the 28-layer two-shard model, prefill 8 x 2048 then 128 decode steps:
  sequence 0 through the oracle with the same forced decode inputs, every
  step compared; and the bench's CUDA-graph path (greedy feedback on the
  device) equal bit for bit to the same kernels launched one by one.

Tolerances are those of tests/test_gpu_model.py (bf16 models, measured
against the oracle's own sensitivity to bf16 softmax weights).
"""
import numpy as np
import pytest
import torch

import oracle as O
import seeded_inputs as si
from tests._util import assert_within_ulps, to_np
from tests.model_parity import bf16_softmax_weights, forced_tokens
from tests.test_gpu_model import check_bf16_step

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
    rows = np.array([0, 1, 127, 128, 4095, 4096, 8000, 8191])
    for tp in w.tps:
        logits = torch.empty(w.n_tokens, m.vocab, dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(L.lm_head_workspace_size(w.n_tokens, m.vocab, m.hidden, tp, torch.bfloat16),
                         dtype=torch.uint8, device="cuda")
        L.lm_head(hidden.cuda(), None, w.n_tokens, table, tp, logits, None, ws)
        torch.cuda.synchronize()
        L.device_error()
        h = hidden.double().numpy()[rows]
        ref = O.compute_logits(m.replace(tp=tp), tab64, h, tp)
        got = to_np(logits[torch.from_numpy(rows).cuda()])
        acc = 2.0 ** -18 * (np.abs(h) @ np.abs(tab64).T)
        assert_within_ulps(got, ref, 1.0, 0.9, f"lm_head tp{tp}", atol=acc)


def _decode_fullsize_oracle(m, ow, b_idx, ctx_lens):
    """Oracle decode step for the sequences b_idx (each alone, with its own cache history)."""
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    batch = si.decode_batch(m, ctx_lens)
    outs = []
    for b in b_idx:
        L = ctx_lens[b]
        gslots = torch.arange(int(batch.seq_base[b]), int(batch.seq_base[b]) + L - 1, dtype=torch.int64)
        hist = [(si.kv_history(m, l, "k", gslots).double().numpy(), si.kv_history(m, l, "v", gslots).double().numpy())
                for l in range(m.n_layers)]
        ctx = O.AttnContext(False, np.array([L - 1]), seq_base=np.array([0]), context_lens=np.array([L]))
        res = []
        for rounded in (False, True):
            cache = O.KVCache(m.n_layers, L, m.n_kv_heads, m.head_dim, m.tp)
            for l in range(m.n_layers):
                cache.k[0][l][:L - 1], cache.v[0][l][:L - 1] = hist[l]
            if rounded:
                with bf16_softmax_weights():
                    h = O.model_forward(m, ow, batch.ids.numpy()[b:b + 1], np.array([L - 1]), ctx, cache, cos_sin)
            else:
                h = O.model_forward(m, ow, batch.ids.numpy()[b:b + 1], np.array([L - 1]), ctx, cache, cos_sin)
            res += [h[0], O.compute_logits(m, ow.embed, h, m.tp)[0]]
        outs.append(tuple(res))
    return outs


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
    order = np.argsort(ctx_lens)
    picks = [int(order[0]), int(order[len(order) // 2]), int(order[-1])]
    gh, gl = to_np(h), to_np(logits)
    for b, (oh, ol, nh, nl) in zip(picks, _decode_fullsize_oracle(m, oracle_weights, picks, ctx_lens)):
        check_bf16_step(gl[b:b + 1], ol[None], gh[b:b + 1], oh[None], nl[None], nh[None],
                        f"seq {b} ctx {ctx_lens[b]}")


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
    hid.append(h[wl.pctx.last_idx.long()].clone())
    lg, nt = fwd.compute_logits(h, wl.pctx.last_idx, B)
    log.append(lg.clone())
    greedy0 = nt.clone()
    for s in range(S):
        ctx = M.DecodeContext(forced[s].cuda(), wl.dpos[s], wl.dcl[s], wl.dslots[s], wl.dbase, wl.max_context)
        h = fwd.run_layers(ctx, decode=True)
        hid.append(h.clone())
        lg, _ = fwd.compute_logits(h, None, B)
        log.append(lg.clone())
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
    # (3) sequence 0 through the oracle with the same forced inputs
    ow = oracle_weights
    L0 = seq_lens[0]
    ids0 = si.prefill_batch(m, seq_lens, extra_capacity=S).ids.numpy()[:L0]
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)

    def run():
        cache = O.KVCache(m.n_layers, L0 + S, m.n_kv_heads, m.head_dim, m.tp)
        ctx = O.AttnContext(True, np.arange(L0), cu_seqlens=np.array([0, L0]))
        hh = O.model_forward(m, ow, ids0, np.arange(L0), ctx, cache, cos_sin)
        out_h = [hh[-1]]
        out_l = [O.compute_logits(m, ow.embed, hh, m.tp, np.array([0, L0]))[0]]
        for s in range(S):
            pos = L0 + s
            dctx = O.AttnContext(False, np.array([pos]), seq_base=np.array([0]), context_lens=np.array([pos + 1]))
            hh = O.model_forward(m, ow, forced[s].numpy()[:1], np.array([pos]), dctx, cache, cos_sin)
            out_h.append(hh[0])
            out_l.append(O.compute_logits(m, ow.embed, hh, m.tp)[0])
        return out_h, out_l
    oh, ol = run()
    with bf16_softmax_weights():
        nh, nl = run()
    for s in range(S + 1):
        check_bf16_step(to_np(log[s][0:1]), ol[s][None], to_np(hid[s][0:1]), oh[s][None], nl[s][None], nh[s][None],
                        f"step {s}")
