"""The one-kernel decode step (qw_decode_layers) against the oracle and
against the per-operation entry points (needs a GB300).

Shapes vary what the kernel partitions differently: GQA group sizes 1, 2
and 4, one and two tp shards, batches of 1, 5 and 16 tokens, contexts from
a single key (the token itself) to several attention chunks.  Tolerances
are those of tests/test_gpu_model.py (the stated bf16 bound, or twice the
model's fp32-accumulation noise floor where that is higher; argmax agreement
on decisive rows).
"""
import numpy as np
import pytest
import torch

import oracle as O
import seeded_inputs as si
from tests._util import assert_within_ulps, to_np
from tests.model_parity import forced_tokens, run_gpu, run_oracle
from tests.test_gpu_model import Parity, check_bf16_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_transformer_forward_gb300 import build
    build.build()


BASE = si.QWEN3_0_6B.replace(vocab=4096, n_layers=2, gamma_sigma=0.1)

CASES = {
    # name: (shape overrides, prefill lengths, decode steps)
    "gqa2_tp2_b5": (dict(tp=2), [37, 130, 1, 64, 300], 2),
    "gqa2_tp1_b1": (dict(tp=1), [1], 3),
    "gqa1_tp2_b3": (dict(n_heads=8, n_kv_heads=8, intermediate=1024, tp=2), [20, 700, 129], 2),
    "gqa4_tp2_b16": (dict(n_heads=16, n_kv_heads=4, tp=2), [3 + 37 * i for i in range(16)], 2),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_decode_step_against_oracle(case):
    over, seq_lens, steps = CASES[case]
    m = BASE.replace(**over)
    forced = forced_tokens(m, steps, len(seq_lens))
    fwds = []
    g = run_gpu(m, seq_lens, steps, forced=forced, fused_decode=True, fwd_out=fwds)
    assert fwds[0].fused_decode_ok(len(seq_lens)), "the fused path must be the one under test"
    o = run_oracle(m, seq_lens, steps, forced=forced, weights=O.load_weights(m))
    par = Parity(f"fused2_{case}")
    for s in range(1, steps + 1):
        check_bf16_step(g.logits[s], o.logits[s], g.hidden[s], o.hidden[s], f"{case} step {s}", par)
    par.check()


def test_decode_step_matches_per_operation_path():
    """Same inputs through both decode paths: hidden states agree to bf16
    rounding noise and the KV-cache rows each step writes agree (v as stored
    QKV outputs, k after norm + RoPE)."""
    m = BASE.replace(n_layers=3)
    seq_lens = [5, 90, 260, 33]
    steps = 2
    forced = forced_tokens(m, steps, len(seq_lens))
    fa, fb = [], []
    a = run_gpu(m, seq_lens, steps, forced=forced, fused_decode=True, fwd_out=fa)
    b = run_gpu(m, seq_lens, steps, forced=forced, fused_decode=False, fwd_out=fb)
    # Both paths round at the same points but add fp32 partial sums in
    # different orders (k-chunk order here, warp order in the per-operation
    # GEMV), so each rounding may land one bf16 step apart; through three
    # layers the mean gap stays within one bf16 ulp at 1.0 (2^-7).
    for s in range(1, steps + 1):
        d = np.abs(a.hidden[s] - b.hidden[s])
        assert d.max() <= 0.05 * max(1.0, np.abs(b.hidden[s]).max()), (s, d.max())
        assert d.mean() <= 2.0 ** -7, (s, d.mean())
    # layer 0 sees identical inputs in both paths: its new cache rows agree to
    # the rounding of one GEMV (v) or GEMV + norm + RoPE (k).  Deeper layers
    # see inputs that already carry the noise above: agreement to its scale.
    for l in range(m.n_layers):
        ka, kb = to_np(fa[0].k_cache[l]), to_np(fb[0].k_cache[l])
        va, vb = to_np(fa[0].v_cache[l]), to_np(fb[0].v_cache[l])
        if l == 0:
            assert_within_ulps(va, vb, 1.0, 0.95, "v cache layer 0", atol=2.0 ** -12)
            assert_within_ulps(ka, kb, 2.0, 0.9, "k cache layer 0", atol=2.0 ** -6)
        else:
            for name, x, y in (("v", va, vb), ("k", ka, kb)):
                d = np.abs(x - y)
                assert d.max() <= 2.0 ** -4 * np.abs(y).max(), (name, l, d.max())
                assert d.mean() <= 2.0 ** -10, (name, l, d.mean())


def test_decode_step_workspace_left_ready():
    """After a call the counters region is as the next call needs it: the grid
    barrier count a multiple of the CTA count, every other counter zero."""
    from qwen3_transformer_forward_gb300 import _lib as L
    m = BASE
    seq_lens = [10, 20]
    fwds = []
    run_gpu(m, seq_lens, 2, forced=forced_tokens(m, 2, 2), fused_decode=True, fwd_out=fwds)
    _, ws = fwds[0]._fused_state()
    torch.cuda.synchronize()
    L.device_error()
    head = ws[:64 * 1024].cpu()
    bar = int(head[:8].view(torch.int64).item())
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert bar > 0 and bar % n_sm == 0
    assert int(head[8:].to(torch.int64).abs().sum()) == 0


def test_decode_step_in_cuda_graph_equals_eager():
    """The kernel replayed from a CUDA graph gives the same bits as launched eagerly."""
    from qwen3_transformer_forward_gb300 import model as M
    m = BASE
    seq_lens = [40, 7, 300]
    B = len(seq_lens)
    params = M.load_params(m, device="cuda")
    b = si.prefill_batch(m, seq_lens, extra_capacity=1)
    fwd = M.Qwen3Forward(m, params, max_tokens=sum(seq_lens), num_slots=b.num_slots, max_seqs=B,
                         max_context=max(seq_lens) + 1)
    fwd.fused_decode = True
    fwd.run_layers(M.to_device_prefill(b), decode=False)
    from tests.model_parity import decode_meta
    pos, cl, slots, base = decode_meta(seq_lens, 0, 1)
    ctx = M.DecodeContext(forced_tokens(m, 1, B)[0].cuda(), torch.from_numpy(pos).cuda(),
                          torch.from_numpy(cl).cuda(), torch.from_numpy(slots).cuda(), torch.from_numpy(base).cuda(),
                          int(cl.max()))
    assert fwd.fused_decode_ok(B)
    eager = fwd.run_layers(ctx, decode=True).clone()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        out = fwd.run_layers(ctx, decode=True)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
