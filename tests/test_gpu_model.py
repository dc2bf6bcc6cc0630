"""End-to-end parity of the CUDA forward pass with the oracle (needs a GB300).

Tolerances (from the stated targets, read as explained here):
  * fp32 model: normwise relative error <= 1e-4 on the final hidden state and
    the logits (max |g - o| / max |o| per tensor).
  * bf16 models: |g - o| <= B + ulp(o) on the logits, where ulp(o) is the
    bf16 spacing at the oracle's value (the last rounding to bf16, taken
    independently on both sides, may land one step apart) and the budget
    B = max(2e-2, 2 * S).  S is the model's own bf16 sensitivity, measured
    in the test: the largest change of the oracle's output when the only
    change to it is rounding the softmax weights P to bf16 before the PV
    product, which every flash-style tensor-core kernel does.  On random-
    init weights that change alone reaches 0.026 on the logits 3 layers
    deep and 0.14 at 28 layers, above the 2e-2 target, so the target cannot
    be met literally by any bf16 flash-attention kernel.  The bulk of the
    error must match the noise floor closely: mean absolute errors at most
    max(one bf16 ulp at 1.0 (7.8e-3), 1.25x the sensitivity's mean).  The
    maximum over ~1.5e5 logits is a tail statistic of the same noise; the
    logits are projections of one perturbed 1024-wide hidden state, so the
    maxima of two noise draws differ by tens of percent even when their
    means agree (28 layers: means 7.05e-3 vs 6.77e-3, maxima 0.055 vs
    0.039): hence 2x on the maximum.
    On the final hidden state (RMS 1, |x| up to ~5) the same rule applies
    with the 2e-2 relative to max(1, |o|).
    Greedy argmax agreement >= 99 %, every disagreement a near-tie (the
    oracle's logits of the two tokens within the logit tolerance).
"""
import numpy as np
import pytest
import torch

import oracle as O
import seeded_inputs as si
from tests._util import bf16_ulp, normwise_rel_err
from tests.model_parity import argmax_agreement, bf16_softmax_weights, forced_tokens, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_transformer_forward_gb300 import build
    build.build()


def _report(name, g, o):
    d = np.abs(g - o)
    print(f"{name}: max abs {d.max():.3e} mean abs {d.mean():.3e} max|o| {np.abs(o).max():.3f}")
    return d


def test_tiny_fp32_model_prefill():
    w = si.workload("tiny_fp32_prefill")
    m = w.model
    g = run_gpu(m, w.seq_lens, 0)
    o = run_oracle(m, w.seq_lens, 0)
    assert normwise_rel_err(g.hidden[0], o.hidden[0]) <= 1e-4
    assert normwise_rel_err(g.logits[0], o.logits[0]) <= 1e-4
    assert np.array_equal(g.tokens[0], o.tokens[0])


def test_tiny_fp32_model_prefill_and_decode():
    m = si.TINY.replace(n_layers=2)
    seq_lens = [5, 16, 1]
    forced = forced_tokens(m, 4, 3)
    g = run_gpu(m, seq_lens, 4, forced=forced)
    o = run_oracle(m, seq_lens, 4, forced=forced)
    for s in range(5):
        assert normwise_rel_err(g.logits[s], o.logits[s]) <= 1e-4, s
        assert normwise_rel_err(g.hidden[s], o.hidden[s]) <= 1e-4, s


SMALL_BF16 = si.QWEN3_0_6B.replace(vocab=8192, n_layers=3, tp=2, gamma_sigma=0.1)


@pytest.mark.parametrize("tp,fused", [(1, True), (2, True), (2, False)])
def test_small_bf16_model_prefill_and_decode(tp, fused):
    """fused: decode steps through the one-kernel decode step (qw_decode_layers),
    else through the per-operation entry points."""
    m = SMALL_BF16.replace(tp=tp)
    seq_lens = [37, 130, 1, 64]
    steps = 3
    forced = forced_tokens(m, steps, len(seq_lens))
    g = run_gpu(m, seq_lens, steps, forced=forced, fused_decode=fused)
    w = O.load_weights(m)
    o = run_oracle(m, seq_lens, steps, forced=forced, weights=w)
    with bf16_softmax_weights():
        n = run_oracle(m, seq_lens, steps, forced=forced, weights=w)
    for s in range(steps + 1):
        check_bf16_step(g.logits[s], o.logits[s], g.hidden[s], o.hidden[s], n.logits[s], n.hidden[s], f"step {s}")


def check_bf16_step(gl, ol, gh, oh, nl, nh, what):
    """gl/gh: CUDA logits/hidden; ol/oh: oracle; nl/nh: oracle with bf16 softmax weights."""
    dl = _report(f"{what} logits", gl, ol)
    dh = _report(f"{what} hidden", gh, oh)
    sl = np.abs(nl - ol)
    sh = np.abs(nh - oh)
    print(f"{what} sensitivity: logits max {sl.max():.3e} mean {sl.mean():.3e}; hidden max {sh.max():.3e} "
          f"mean {sh.mean():.3e}")
    bl = max(LOGIT_TOL, 2.0 * float(sl.max()))
    bh = max(LOGIT_TOL, 2.0 * float(sh.max()))
    assert np.all(dl <= bl + bf16_ulp(ol)), what
    assert np.all(dh <= bh * np.maximum(1.0, np.abs(oh)) + bf16_ulp(oh)), what
    assert dl.mean() <= max(2.0 ** -7, 1.25 * sl.mean()), what
    assert dh.mean() <= max(2.0 ** -7, 1.25 * sh.mean()), what
    agree, bad = argmax_agreement(gl, ol, bl + float(bf16_ulp(np.abs(ol).max())))
    assert len(bad) == 0, what
    return agree


def test_single_layer_prefill_full_size():
    """One Qwen3-0.6B layer, two shards, prefill 4 x 512 from N(0,1) hidden inputs."""
    from qwen3_transformer_forward_gb300 import model as M
    from qwen3_transformer_forward_gb300 import _lib as L
    w = si.workload("layer_prefill")
    m = w.model
    b = si.prefill_batch(m, w.seq_lens)
    T = b.ids.shape[0]
    x = si.normal(0, "layer_prefill.hidden", (T, m.hidden), 1.0, "bf16")
    params = M.load_params(m, device="cuda")
    fwd = M.Qwen3Forward(m, params, max_tokens=T, num_slots=b.num_slots, max_seqs=len(w.seq_lens),
                         max_context=max(w.seq_lens))
    h, res = fwd.run_layers(M.to_device_prefill(b), decode=False, hidden_in=x.cuda(), final_norm=False)
    torch.cuda.synchronize()
    L.device_error()
    ow = O.load_weights(m, with_embed=False)
    cache = O.KVCache(1, b.num_slots, m.n_kv_heads, m.head_dim, m.tp)
    ctx = O.AttnContext(True, b.slot_mapping.numpy(), cu_seqlens=b.cu_seqlens.numpy())
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    oh, ores = O.decoder_layer(m, ow.layers[0], 0, b.positions.numpy(), x.double().numpy(), None, ctx, cache,
                               *cos_sin)
    # after the layer: residual = x + attention output, h = the MLP output
    for name, gv, ov in (("residual", res, ores), ("layer out", h, oh)):
        d = _report(name, gv.double().cpu().numpy(), ov)
        assert np.all(d <= LOGIT_TOL * np.maximum(1.0, np.abs(ov)) + bf16_ulp(ov)), name
        assert d.mean() <= 2.0 ** -7, name
    # KV cache contents after the layer: v bit-exact, k within 2 ulp
    kc = fwd.k_cache[0].double().cpu().numpy()
    vc = fwd.v_cache[0].double().cpu().numpy()
    kref = np.concatenate([cache.k[r][0] for r in range(m.tp)], axis=1)
    vref = np.concatenate([cache.v[r][0] for r in range(m.tp)], axis=1)
    # v depends on the QKV GEMM (one rounding), k on GEMM + norm + rope
    from tests._util import assert_within_ulps
    assert_within_ulps(vc, vref, 1.0, 0.95, "v cache", atol=1e-3)
    # k = rope(norm(k)): each output is a difference of two normalised O(1)
    # inputs, so a one-ulp difference in an input (ulp 2^-7 at 1.0) carries
    # into the output whatever its own size: absolute slack 2^-6 on top
    assert_within_ulps(kc, kref, 2.0, 0.9, "k cache", atol=2.0 ** -6)
