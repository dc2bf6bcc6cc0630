"""Per-kernel parity of the CUDA path with the CPU oracle (needs a GB300).

Every call goes through the C ABI (ctypes binding).  Inputs come from the
seeded generator; expected values come from the oracle only.  Sizes span
several tiles plus a ragged tail.

Tolerances:
  * integer/index/copy work (embedding, KV placement, v cache, argmax): bit-exact;
  * bf16 outputs of one rounding step: within 1 bf16 ulp of the oracle (the
    oracle rounds its float64 result once; the kernel rounds its fp32 result
    once, so they differ only where the two sit on opposite sides of a
    rounding midpoint); GEMMs add the fp32 accumulation error, at most
    (K/16) * 2^-24 * sum_k |a_k w_k| for K/16 sequential fp32 additions of
    16-term tensor-core products, taken as 2^-18 * sum_k |a_k w_k| (K <= 4096);
  * attention (prefill, and decode in bf16): P is rounded to bf16 before the
    PV product on the tensor cores, so |err| <= 2 ulp(|out|) + 2^-9 * max|v|
    (derived below);
  * fp32 paths: normwise relative error <= 1e-5.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import seeded_inputs as si
from tests._util import assert_within_ulps, bf16_ulp, normwise_rel_err, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_transformer_forward_gb300 import build
    build.build()
    from qwen3_transformer_forward_gb300 import _lib
    _lib.load()
    return _lib


def dev(t):
    return t.to("cuda")


def sync_ok(L):
    torch.cuda.synchronize()
    L.device_error()


# ----------------------------------------------------------------------------
# embedding
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("tp", [1, 2, 4])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_embed_vocab_bit_exact(L, tp, dtype):
    m = si.ModelShape(vocab=4096, hidden=1024 if dtype == "bf16" else 64, n_heads=1, n_kv_heads=1, head_dim=8,
                      intermediate=8, n_layers=0, dtype=dtype)
    table = si.checkpoint_tensor(m, "embed_tokens")
    ids = si.embed_ids(m, 1000, 0.05)
    ids[:8] = torch.tensor([0, 1023, 1024, 2047, 2048, 3071, 3072, 4095])
    ids[10] = -1          # out of range: zero row and one error count each
    ids[11] = 4096
    ids[12] = 10 ** 9
    out = torch.full((1000, m.hidden), 7.0, dtype=table.dtype, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.embed_vocab(dev(ids), dev(table), tp, out, err)
    sync_ok(L)
    ref = O.vocab_parallel_embedding(ids.numpy(), table.double().numpy(), tp)
    assert np.array_equal(to_np(out), ref)
    assert int(err.item()) == 3
    assert np.all(to_np(out)[[10, 11, 12]] == 0)


def test_embed_empty_is_noop(L):
    out = torch.full((1, 64), 3.0, device="cuda")
    L.embed_vocab(torch.zeros(0, dtype=torch.int64, device="cuda"), torch.zeros(8, 64, device="cuda"), 2, out[:0])
    sync_ok(L)
    assert torch.all(out == 3.0)


# ----------------------------------------------------------------------------
# add + RMSNorm
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,H", [("bf16", 1024), ("bf16", 2048), ("bf16", 64), ("f32", 64), ("f32", 1024)])
@pytest.mark.parametrize("with_res", [False, True])
def test_add_rmsnorm(L, dtype, H, with_res):
    T = 37
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = si.normal(0, "t.x", (T, H), 1.0, dtype)
    r = si.normal(0, "t.r", (T, H), 2.0, dtype)
    g = (si.normal(0, "t.g", (H,), 0.2, "f32") + 1.0).to(dt)
    y = torch.empty(T, H, dtype=dt, device="cuda")
    res_buf = dev(r.clone())
    L.add_rmsnorm(dev(x), res_buf if with_res else None, res_buf, dev(g), 1e-6, y)
    sync_ok(L)
    if with_res:
        ry, rres = O.add_rms_norm(x.double().numpy(), r.double().numpy(), g.double().numpy(), 1e-6, dtype)
    else:
        ry = O.rms_norm(x.double().numpy(), g.double().numpy(), 1e-6, dtype)
        rres = x.double().numpy()
    if dtype == "bf16":
        assert np.array_equal(to_np(res_buf), rres)          # residual add: one rounding of an exact sum
        assert_within_ulps(to_np(y), ry, 1.0, 0.98, "rmsnorm y")
    else:
        assert normwise_rel_err(to_np(res_buf), rres) <= 1e-6
        assert normwise_rel_err(to_np(y), ry) <= 1e-5


# ----------------------------------------------------------------------------
# QK-norm + RoPE + KV store
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,nh,nkv,hd,tp", [("bf16", 16, 8, 128, 2), ("bf16", 16, 8, 128, 1),
                                                ("bf16", 8, 2, 64, 2), ("f32", 4, 2, 16, 2)])
def test_qkv_norm_rope_store_kv(L, dtype, nh, nkv, hd, tp):
    T, num_slots = 45, 80
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    m = si.ModelShape(vocab=64, hidden=64, n_heads=nh, n_kv_heads=nkv, head_dim=hd, intermediate=64, n_layers=1,
                      tp=tp, dtype=dtype, max_position=3000)
    width = tp * (nh // tp + 2 * (nkv // tp)) * hd
    qkv = si.normal(0, "t.qkv", (T, width), 1.0, dtype)
    qg = (si.normal(0, "t.qg", (hd,), 0.2, "f32") + 1.0).to(dt)
    kg = (si.normal(0, "t.kg", (hd,), 0.2, "f32") + 1.0).to(dt)
    pos = si.uniform_int(0, "t.pos", (T,), 0, 2176)
    pos[0] = 0
    pos[1] = 2175
    perm = torch.randperm(num_slots, generator=torch.Generator().manual_seed(0))[:T]
    slots = perm.clone()
    slots[[3, 17, 40]] = -1
    sentinel = 5.0
    kc = torch.full((num_slots, nkv, hd), sentinel, dtype=dt, device="cuda")
    vc = torch.full((num_slots, nkv, hd), sentinel, dtype=dt, device="cuda")
    q_out = torch.empty(T, nh * hd, dtype=dt, device="cuda")
    cs = L.rope_cos_sin_table(m.max_position, hd, m.rope_theta)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.qkv_norm_rope_store_kv(dev(qkv), nh, nkv, hd, tp, dev(pos), dev(cs), dev(qg), dev(kg), m.eps, dev(slots),
                             kc, vc, q_out, err)
    sync_ok(L)
    assert int(err.item()) == 0
    # oracle: per shard, split the merged block, norm, rope, store
    cos_t, sin_t = O.rope_cos_sin(m.max_position, hd, m.rope_theta)
    nh_l, nkv_l = nh // tp, nkv // tp
    x = qkv.double().numpy()
    wr = (nh_l + 2 * nkv_l) * hd
    qs, ks, vs = [], [], []
    for r in range(tp):
        blk = x[:, r * wr:(r + 1) * wr]
        qs.append(blk[:, : nh_l * hd].reshape(T, nh_l, hd))
        ks.append(blk[:, nh_l * hd:(nh_l + nkv_l) * hd].reshape(T, nkv_l, hd))
        vs.append(blk[:, (nh_l + nkv_l) * hd:].reshape(T, nkv_l, hd))
    q = np.concatenate(qs, 1)
    k = np.concatenate(ks, 1)
    v = np.concatenate(vs, 1)
    q = O.apply_rope(O.rms_norm(q, qg.double().numpy(), m.eps, dtype), pos.numpy(), cos_t, sin_t, dtype)
    k = O.apply_rope(O.rms_norm(k, kg.double().numpy(), m.eps, dtype), pos.numpy(), cos_t, sin_t, dtype)
    cache = O.KVCache(1, num_slots, nkv, hd, 1)
    cache.k[0][0][:] = sentinel
    cache.v[0][0][:] = sentinel
    cache.store(0, 0, k, v, slots.numpy())
    kc_n, vc_n = to_np(kc), to_np(vc)
    assert np.array_equal(vc_n, cache.v[0][0])                  # placement + bit copy of v
    untouched = np.ones(num_slots, bool)
    untouched[slots.numpy()[slots.numpy() >= 0]] = False
    assert np.all(kc_n[untouched] == sentinel)                 # slots not in the mapping keep the sentinel
    if dtype == "bf16":
        # two roundings (norm, rope): a midpoint flip at the first can move the second by one ulp
        assert_within_ulps(kc_n, cache.k[0][0], 2.0, 0.97, "k cache")
        assert_within_ulps(to_np(q_out).reshape(T, nh, hd), q, 2.0, 0.97, "q")
    else:
        assert normwise_rel_err(kc_n, cache.k[0][0]) <= 1e-5
        assert normwise_rel_err(to_np(q_out).reshape(T, nh, hd), q) <= 1e-5


# ----------------------------------------------------------------------------
# GEMMs (tcgen05 for bf16, CUDA cores for f32)
# ----------------------------------------------------------------------------

def _gemm_abs_bound(A, W, mode, epi, tp):
    """2^-18 * sum_k |a_k||w_k| per output (for SiluAndMul: scaled by the gate/up sizes)."""
    a = np.abs(A.double().numpy())
    w = np.abs(W.double().numpy())
    if mode == 1:
        w = np.concatenate([w[r] for r in range(tp)], axis=1)
    s = a @ w.T
    if epi == 1:
        i_l = w.shape[0] // 2 // tp
        g = np.concatenate([s[:, r * 2 * i_l:r * 2 * i_l + i_l] for r in range(tp)], -1)
        u = np.concatenate([s[:, r * 2 * i_l + i_l:(r + 1) * 2 * i_l] for r in range(tp)], -1)
        s = (g + u) * (1.0 + g + u)
    return 2.0 ** -18 * s


def _gemm_ref(A, W, mode, epi, tp, dtype):
    a = A.double().numpy()
    w = W.double().numpy()
    if mode == 0:
        if epi == 0:
            return O.linear(a, w, dtype)
        N = w.shape[0]
        i_l = N // 2 // tp
        outs = []
        for r in range(tp):
            gu = O.linear(a, w[r * 2 * i_l:(r + 1) * 2 * i_l], dtype)
            outs.append(O.silu_and_mul(gu, dtype))
        return np.concatenate(outs, -1)
    # row reduce: W is [tp, N, K/tp] -> full [N, K]
    full = np.concatenate([w[r] for r in range(tp)], axis=1)
    k_l = full.shape[1] // tp
    return O.row_parallel_linear([a[:, r * k_l:(r + 1) * k_l] for r in range(tp)], full, tp, dtype)


GEMM_CASES = [
    # M,    N,    K,    tp, mode, epi
    (300, 784, 1024, 1, 0, 0),      # prefill path: 3 M tiles (ragged), 4 N tiles (last one 16 wide)
    (129, 4096, 1024, 2, 0, 0),
    (300, 1024, 2048, 2, 1, 0),     # row split, shard sum in the accumulator
    (257, 1024, 3072, 2, 1, 0),
    (200, 1536, 1024, 2, 0, 1),     # gate_up + SiluAndMul, I/tp = 384 (3 tiles per shard)
    (130, 1000 // 8 * 16, 1000, 1, 0, 0),   # K not a multiple of 64 (TMA zero fill)
    (1, 4096, 1024, 2, 0, 0),       # decode path (swapped operands, split K)
    (7, 1024, 2048, 2, 1, 0),
    (8, 1024, 3072, 2, 1, 0),       # decode down: staged activations, 16 weight rows per CTA in shared memory
    (5, 6144, 1024, 2, 0, 1),       # SiluAndMul on the staged path: gate and up rows side by side in shared memory
    (8, 2048, 1024, 1, 0, 0),       # column layout, narrow output, staged path
    (16, 6144, 1024, 2, 0, 1),
    (33, 1024, 3072, 2, 1, 0),
    (64, 4096, 1024, 1, 0, 0),
    (64, 6144, 1024, 1, 0, 1),
    (65, 1024, 2048, 2, 1, 0),      # first size on the prefill path
]


@pytest.mark.parametrize("M,N,K,tp,mode,epi", GEMM_CASES)
def test_gemm_bf16(L, M, N, K, tp, mode, epi):
    A = si.normal(0, f"g.A{M}.{K}", (M, K), 1.0, "bf16")
    if mode == 1:
        W = si.normal(0, f"g.W{N}.{K}", (tp, N, K // tp), 0.02, "bf16")
    else:
        W = si.normal(0, f"g.W{N}.{K}", (N, K), 0.02, "bf16")
    n_out = N // 2 if epi == 1 else N
    C = torch.full((M, n_out), 123.0, dtype=torch.bfloat16, device="cuda")
    ws_n = L.gemm_workspace_size(M, N, K, tp, mode, epi, torch.bfloat16)
    ws = torch.zeros(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    L.gemm(dev(A), dev(W), C, N, tp, mode, epi, ws)
    sync_ok(L)
    ref = _gemm_ref(A, W, mode, epi, tp, "bf16")
    # fp32 accumulation vs exact: one rounding each; SiluAndMul adds one more
    assert_within_ulps(to_np(C), ref, 1.0 if epi == 0 else 2.0, 0.9, f"gemm {M}x{N}x{K} mode{mode} epi{epi}",
                       atol=_gemm_abs_bound(A, W, mode, epi, tp))


@pytest.mark.parametrize("M,N,K,tp,epi,with_res", [(8, 4096, 1024, 2, 0, True), (8, 6144, 1024, 2, 1, True),
                                                    (1, 4096, 1024, 1, 0, False), (16, 6144, 1024, 2, 1, True),
                                                    (13, 1024, 2048, 2, 0, True), (5, 512, 96, 2, 1, False),
                                                    # 311 groups of 8 outputs: two per CTA, the last CTA half empty
                                                    (3, 4976, 256, 1, 1, True),
                                                    # two tokens per warp, K = 3072 (the down projection's width)
                                                    (16, 512, 3072, 1, 0, True),
                                                    # 32-row CTAs, the last one's second tile past N
                                                    (8, 4880, 1024, 1, 0, True),
                                                    # 8 weight rows per CTA (narrow output), rows in shared memory
                                                    (4, 1024, 2048, 2, 0, True)])
def test_add_rmsnorm_gemm(L, M, N, K, tp, epi, with_res):
    """Fused add + RMSNorm + column Linear (decode QKV / gate_up) against the
    oracle's add_rms_norm followed by the oracle Linear."""
    x = si.normal(0, f"ng.x{M}.{K}", (M, K), 1.0, "bf16")
    r = si.normal(0, f"ng.r{M}.{K}", (M, K), 2.0, "bf16")
    g = (si.normal(0, f"ng.g{K}", (K,), 0.2, "f32") + 1.0).to(torch.bfloat16)
    W = si.normal(0, f"ng.W{N}.{K}", (N, K), 0.02, "bf16")
    C = torch.full((M, N // 2 if epi == 1 else N), 123.0, dtype=torch.bfloat16, device="cuda")
    res_out = torch.full((M, K), 7.0, dtype=torch.bfloat16, device="cuda")
    L.add_rmsnorm_gemm(dev(x), dev(r) if with_res else None, res_out, dev(g), 1e-6, dev(W), C, N, tp, epi)
    sync_ok(L)
    if with_res:
        ry, rres = O.add_rms_norm(x.double().numpy(), r.double().numpy(), g.double().numpy(), 1e-6, "bf16")
    else:
        ry = O.rms_norm(x.double().numpy(), g.double().numpy(), 1e-6, "bf16")
        rres = x.double().numpy()
    assert np.array_equal(to_np(res_out), rres)   # residual add: one rounding of an exact sum
    y = torch.from_numpy(ry).to(torch.bfloat16)
    ref = _gemm_ref(y, W, 0, epi, tp, "bf16")
    # y itself may sit one bf16 step from the oracle's (rsqrt and summation
    # order): that step times sum_k |w_k| on top of the GEMM's own bound
    y_step = 2.0 ** -8 * (np.abs(ry) @ np.abs(W.double().numpy()).T)
    if epi == 1:
        i_l = N // 2 // tp
        y_step = np.concatenate([y_step[:, r_ * 2 * i_l:r_ * 2 * i_l + i_l] + y_step[:, r_ * 2 * i_l + i_l:(r_ + 1) * 2 * i_l]
                                 for r_ in range(tp)], -1) * 2.0
    assert_within_ulps(to_np(C), ref, 2.0, 0.9, f"add_rmsnorm_gemm {M}x{N}x{K} epi{epi}",
                       atol=_gemm_abs_bound(y, W, 0, epi, tp) + y_step)


@pytest.mark.parametrize("M,N,K,tp,mode,epi", [
    (300, 528, 192, 1, 0, 0),       # ragged M and N, one tile per CTA
    (200, 272, 256, 2, 1, 0),       # row split
    (333, 800, 128, 2, 0, 1),       # SiluAndMul, I/tp = 200: a half-filled last tile per shard
    (333, 512, 128, 2, 0, 1),       # SiluAndMul, I/tp = 128: tensor-store epilogue, ragged rows
    (4096, 4096, 64, 1, 0, 0),      # one k-block per tile: the ring spans tile boundaries
    (16384, 6144, 1024, 2, 0, 1),   # the 0.6B prefill gate_up: 20 tiles per CTA (256-row tiles by default)
    (2000, 5120, 256, 1, 0, 0),     # 256-row tiles: the last one's second half partly past M
    (1800, 5200, 128, 1, 0, 0),     # 256-row tiles: second half wholly past M, ragged N
    (2000, 4864, 512, 2, 1, 0),     # 256-row tiles, row split
    (2100, 8192, 256, 2, 0, 1),     # 256-row tiles, SiluAndMul
    (2560, 4000, 128, 2, 0, 1),     # 256-row tiles, SiluAndMul with I/tp = 1000 (ragged per shard)
])
def test_gemm_persistent_equals_one_tile_kernel(L, monkeypatch, M, N, K, tp, mode, epi):
    """The persistent prefill GEMM (QW_TC_PERSISTENT=1) accumulates each tile
    in the same k order as the default kernels (one 128- or 256-row tile per
    CTA), which the oracle tests above cover: the outputs must agree bit for bit."""
    g = torch.Generator(device="cuda").manual_seed(7)
    A = (torch.randn(M, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    W = (torch.randn(*((tp, N, K // tp) if mode == 1 else (N, K)), device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    n_out = N // 2 if epi == 1 else N
    out = {}
    for flag in ("0", "1"):
        monkeypatch.setenv("QW_TC_PERSISTENT", flag)
        C = torch.full((M, n_out), float("nan"), dtype=torch.bfloat16, device="cuda")
        L.gemm(A, W, C, N, tp, mode, epi)
        sync_ok(L)
        out[flag] = C
    assert not torch.isnan(out["1"].float()).any()
    assert torch.equal(out["0"], out["1"])


@pytest.mark.parametrize("M,N,K,tp,mode,epi", [(32, 128, 64, 2, 0, 0), (32, 64, 64, 2, 1, 0),
                                               (32, 256, 64, 2, 0, 1), (5, 512, 64, 1, 0, 0)])
def test_gemm_f32(L, M, N, K, tp, mode, epi):
    A = si.normal(0, "gf.A", (M, K), 1.0, "f32")
    W = si.normal(0, "gf.W", (tp, N, K // tp) if mode == 1 else (N, K), 0.02, "f32")
    n_out = N // 2 if epi == 1 else N
    C = torch.empty(M, n_out, dtype=torch.float32, device="cuda")
    L.gemm(dev(A), dev(W), C, N, tp, mode, epi)
    sync_ok(L)
    assert normwise_rel_err(to_np(C), _gemm_ref(A, W, mode, epi, tp, "f32")) <= 1e-5


def test_silu_mul(L):
    T, I, tp = 33, 3072, 2
    x = si.normal(0, "t.gu", (T, 2 * I), 2.0, "bf16")
    out = torch.empty(T, I, dtype=torch.bfloat16, device="cuda")
    L.silu_mul(dev(x), out, tp)
    sync_ok(L)
    xn = x.double().numpy()
    i_l = I // tp
    ref = np.concatenate([O.silu_and_mul(xn[:, r * 2 * i_l:(r + 1) * 2 * i_l], "bf16") for r in range(tp)], -1)
    assert_within_ulps(to_np(out), ref, 1.0, 0.98, "silu_mul")


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def _attn_tol(ref, v):
    # P in bf16 (relative error <= 2^-9 per weight) -> |sum p_j v_j| error <= 2^-9 * max|v|,
    # plus the final rounding of out (<= 1 ulp) and fp32 accumulation slack (1 ulp)
    return 2.0 * bf16_ulp(ref) + 2.0 ** -9 * np.max(np.abs(v)) + 1e-6


def _decode_tol(ref, v):
    # decode carries P as a bf16 pair hi + lo (relative error <= 2^-17 per weight);
    # with the fp32 exp2, softmax sum and accumulation over a few thousand keys
    # the pre-rounding error stays below 2^-14 * max|v|; the final rounding of out
    # may then land one bf16 step away from the oracle's
    return bf16_ulp(ref) + 2.0 ** -14 * np.max(np.abs(v)) + 1e-7


def _assert_decode_close(got, ref, v, what=""):
    err = np.abs(got - ref)
    assert np.all(err <= _decode_tol(ref, v)), (what, float(np.nanmax(err)))
    # most outputs round to the oracle's bf16 value exactly
    assert float(np.mean(got == ref)) >= 0.9, (what, float(np.mean(got == ref)))


@pytest.mark.parametrize("seq_lens,nh,nkv,poison", [
    ([1, 77, 200, 129], 16, 8, False),
    ([512, 512], 16, 8, False),
    ([3], 16, 8, False),
    ([1, 77, 200, 129], 16, 8, True),     # cache rows outside the sequences hold NaN
    ([300, 1000, 5], 8, 8, True),         # group size 1: two query tiles of one head per CTA
    ([129, 384], 6, 2, False),            # odd group size 3
    ([640, 33], 16, 4, False),            # group size 4
])
def test_attention_prefill_bf16_from_cache(L, seq_lens, nh, nkv, poison):
    hd = 128
    b = si.prefill_batch(si.QWEN3_0_6B, seq_lens, extra_capacity=5)
    T = sum(seq_lens)
    q = si.normal(0, "a.q", (T, nh, hd), 1.0, "bf16")
    k = si.normal(0, "a.k", (T, nkv, hd), 1.0, "bf16")
    v = si.normal(0, "a.v", (T, nkv, hd), 1.0, "bf16")
    fill = float("nan") if poison else 0.0
    kc = torch.full((b.num_slots, nkv, hd), fill, dtype=torch.bfloat16)
    vc = torch.full((b.num_slots, nkv, hd), fill, dtype=torch.bfloat16)
    kc[b.slot_mapping] = k
    vc[b.slot_mapping] = v
    out = torch.empty(T, nh * hd, dtype=torch.bfloat16, device="cuda")
    cu = dev(b.cu_seqlens)
    L.attention_prefill(dev(q), dev(kc), dev(vc), cu, cu, dev(b.seq_base), max(seq_lens), nh, nkv, hd,
                        hd ** -0.5, out)
    sync_ok(L)
    ref = O.attention_prefill(q.double().numpy(), k.double().numpy(), v.double().numpy(), b.cu_seqlens.numpy(),
                              hd ** -0.5, "bf16")
    got = to_np(out).reshape(T, nh, hd)
    err = np.abs(got - ref)
    assert np.all(err <= _attn_tol(ref, v.double().numpy())), float(np.nanmax(err))
    assert float(np.mean(err)) < 2e-3


def test_attention_prefill_growing_scores(L):
    """Keys whose norm grows along the sequence: each query's running max keeps
    rising from one key tile to the next, so the kernel's output must not
    depend on when (or whether) it re-bases its softmax accumulators."""
    nh, nkv, hd = 16, 8, 128
    seq_lens = [900, 260]
    b = si.prefill_batch(si.QWEN3_0_6B, seq_lens)
    T = sum(seq_lens)
    q = si.normal(0, "ag.q", (T, nh, hd), 2.0, "bf16")
    k = si.normal(0, "ag.k", (T, nkv, hd), 1.0, "f32")
    pos = b.positions.to(torch.float32)
    k = (k * (1.0 + pos / 64.0)[:, None, None]).to(torch.bfloat16)
    v = si.normal(0, "ag.v", (T, nkv, hd), 1.0, "bf16")
    out = torch.empty(T, nh * hd, dtype=torch.bfloat16, device="cuda")
    cu = dev(b.cu_seqlens)
    L.attention_prefill(dev(q), dev(k), dev(v), cu, cu, None, max(seq_lens), nh, nkv, hd, hd ** -0.5, out)
    sync_ok(L)
    ref = O.attention_prefill(q.double().numpy(), k.double().numpy(), v.double().numpy(), b.cu_seqlens.numpy(),
                              hd ** -0.5, "bf16")
    got = to_np(out).reshape(T, nh, hd)
    assert np.all(np.abs(got - ref) <= _attn_tol(ref, v.double().numpy()))


def test_attention_prefill_packed_and_prefix(L):
    # packed keys (no seq_base) and a query suffix over a longer key prefix
    nh, nkv, hd = 16, 8, 128
    Lk, Lq = [150, 40], [10, 40]
    k = si.normal(0, "a.pk", (sum(Lk), nkv, hd), 1.0, "bf16")
    v = si.normal(0, "a.pv", (sum(Lk), nkv, hd), 1.0, "bf16")
    q = si.normal(0, "a.pq", (sum(Lq), nh, hd), 1.0, "bf16")
    cu_k = torch.tensor([0, 150, 190], dtype=torch.int32)
    cu_q = torch.tensor([0, 10, 50], dtype=torch.int32)
    out = torch.empty(sum(Lq), nh * hd, dtype=torch.bfloat16, device="cuda")
    L.attention_prefill(dev(q), dev(k), dev(v), dev(cu_q), dev(cu_k), None, 40, nh, nkv, hd, hd ** -0.5, out)
    sync_ok(L)
    # the oracle's full causal attention over the whole key sequence, keeping the last Lq rows
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    refs = []
    for s in range(2):
        a, bq = int(cu_q[s]), int(cu_q[s + 1])
        ka, kb = int(cu_k[s]), int(cu_k[s + 1])
        qfull = np.zeros((kb - ka, nh, hd))
        qfull[(kb - ka) - (bq - a):] = qd[a:bq]
        o = O.attention_prefill(qfull, kd[ka:kb], vd[ka:kb], [0, kb - ka], hd ** -0.5, "bf16")
        refs.append(o[(kb - ka) - (bq - a):])
    ref = np.concatenate(refs)
    got = to_np(out).reshape(-1, nh, hd)
    assert np.all(np.abs(got - ref) <= _attn_tol(ref, vd))


def test_attention_prefill_f32(L):
    nh, nkv, hd = 4, 2, 16
    b = si.prefill_batch(si.TINY, [16, 16])
    T = 32
    q = si.normal(0, "af.q", (T, nh, hd), 1.0, "f32")
    k = si.normal(0, "af.k", (T, nkv, hd), 1.0, "f32")
    v = si.normal(0, "af.v", (T, nkv, hd), 1.0, "f32")
    out = torch.empty(T, nh * hd, dtype=torch.float32, device="cuda")
    cu = dev(b.cu_seqlens)
    L.attention_prefill(dev(q), dev(k), dev(v), cu, cu, dev(b.seq_base), 16, nh, nkv, hd, hd ** -0.5, out)
    sync_ok(L)
    ref = O.attention_prefill(q.double().numpy(), k.double().numpy(), v.double().numpy(), b.cu_seqlens.numpy(),
                              hd ** -0.5, "f32")
    assert normwise_rel_err(to_np(out).reshape(T, nh, hd), ref) <= 1e-5


@pytest.mark.parametrize("ctx", [[1, 63, 64, 65, 700], [2048] * 3 + [256], [2176] * 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_attention_decode(L, ctx, dtype):
    nh, nkv, hd = 16, 8, 128
    B = len(ctx)
    cap = [c + 3 for c in ctx]
    base = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int32)
    S = int(sum(cap))
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    kc = si.normal(0, "d.k", (S, nkv, hd), 1.0, dtype)
    vc = si.normal(0, "d.v", (S, nkv, hd), 1.0, dtype)
    q = si.normal(0, "d.q", (B, nh, hd), 1.0, dtype)
    out = torch.empty(B, nh * hd, dtype=dt, device="cuda")
    ws = torch.zeros(max(L.attention_decode_workspace_size(B, max(ctx), nh, hd), 16), dtype=torch.uint8,
                     device="cuda")
    L.attention_decode(dev(q), dev(kc), dev(vc), dev(torch.tensor(ctx, dtype=torch.int32)),
                       dev(torch.tensor(base)), max(ctx), nh, nkv, hd, hd ** -0.5, out, ws)
    sync_ok(L)
    kd, vd = kc.double().numpy(), vc.double().numpy()
    ref = O.attention_decode(q.double().numpy(), [kd[base[b]:base[b] + ctx[b]] for b in range(B)],
                             [vd[base[b]:base[b] + ctx[b]] for b in range(B)], hd ** -0.5, dtype)
    got = to_np(out).reshape(B, nh, hd)
    if dtype == "bf16":
        # the bf16 path runs QK^T and PV on the tensor cores with P as a bf16 hi + lo pair
        _assert_decode_close(got, ref, vd)
    else:
        assert normwise_rel_err(got, ref) <= 1e-5


DECODE_EDGE_CASES = {
    # name: (context lengths, q heads, kv heads)
    "empty_sequences": ([0, 5, 0, 300, 0], 16, 8),        # no keys: zero output
    "many_sequences": ([17 + (7 * i) % 90 for i in range(200)], 16, 8),   # > 128 sequences per scan chunk
    "one_long_many_short": ([4096, 1, 2, 64], 16, 8),      # one pair spans many CTAs
    "group_1": ([130, 2049, 1], 8, 8),
    "group_4": ([130, 2049, 65], 32, 8),
    "group_8": ([700, 2049], 64, 8),
    "single_key": ([1], 16, 8),
}


@pytest.mark.parametrize("case", sorted(DECODE_EDGE_CASES))
def test_attention_decode_partition_edges(L, case):
    """The bf16 decode kernel splits the (sequence, kv head, 64-key tile)
    sequence into one contiguous range per CTA: empty sequences, more than
    128 sequences, a pair spread over many CTAs and every GQA group size."""
    ctx, nh, nkv = DECODE_EDGE_CASES[case]
    hd = 128
    B = len(ctx)
    cap = [c + 3 for c in ctx]
    base = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int32)
    S = int(sum(cap))
    kc = si.normal(0, f"de.{case}.k", (S, nkv, hd), 1.0, "bf16")
    vc = si.normal(0, f"de.{case}.v", (S, nkv, hd), 1.0, "bf16")
    q = si.normal(0, f"de.{case}.q", (B, nh, hd), 1.0, "bf16")
    out = torch.full((B, nh * hd), 7.0, dtype=torch.bfloat16, device="cuda")
    mc = max(ctx)
    ws = torch.zeros(L.attention_decode_workspace_size(B, mc, nh, hd), dtype=torch.uint8, device="cuda")
    for _ in range(2):   # the completion counters must be left at zero for the next call
        L.attention_decode(dev(q), dev(kc), dev(vc), dev(torch.tensor(ctx, dtype=torch.int32)),
                           dev(torch.tensor(base)), mc, nh, nkv, hd, hd ** -0.5, out, ws)
        sync_ok(L)
        assert int(ws[:64 * 1024].view(torch.int32).abs().sum()) == 0
    got = to_np(out).reshape(B, nh, hd)
    kd, vd = kc.double().numpy(), vc.double().numpy()
    live = [b for b in range(B) if ctx[b] > 0]
    for b in range(B):
        if ctx[b] == 0:
            assert np.all(got[b] == 0.0), b
    ref = O.attention_decode(q.double().numpy()[live], [kd[base[b]:base[b] + ctx[b]] for b in live],
                             [vd[base[b]:base[b] + ctx[b]] for b in live], hd ** -0.5, "bf16")
    _assert_decode_close(got[live], ref, vd, case)


def test_attention_decode_max_context_zero_and_overflow(L):
    """max_context 0 (every sequence empty) gives zero outputs; a context length
    above the call's max_context is reported by qw_device_error instead of
    silently dropping keys."""
    from qwen3_transformer_forward_gb300._lib import QW_ERR_INVALID_ARG, QwError
    nh, nkv, hd, B = 16, 8, 128, 3
    kc = dev(si.normal(0, "dz.k", (256, nkv, hd), 1.0, "bf16"))
    vc = dev(si.normal(0, "dz.v", (256, nkv, hd), 1.0, "bf16"))
    q = dev(si.normal(0, "dz.q", (B, nh, hd), 1.0, "bf16"))
    base = dev(torch.tensor([0, 60, 120], dtype=torch.int32))
    out = torch.full((B, nh * hd), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(L.attention_decode_workspace_size(B, 0, nh, hd), dtype=torch.uint8, device="cuda")
    L.attention_decode(q, kc, vc, dev(torch.zeros(B, dtype=torch.int32)), base, 0, nh, nkv, hd, hd ** -0.5, out, ws)
    sync_ok(L)
    assert torch.all(out == 0)
    # lengths 100 and 130 with max_context 8 (planned as one 64-key tile per pair):
    # the overflow is recorded and reported once
    cl = dev(torch.tensor([100, 3, 130], dtype=torch.int32))
    ws = torch.zeros(L.attention_decode_workspace_size(B, 8, nh, hd), dtype=torch.uint8, device="cuda")
    L.attention_decode(q, kc, vc, cl, base, 8, nh, nkv, hd, hd ** -0.5, out, ws)
    with pytest.raises(QwError) as e:
        L.device_error()
    assert e.value.code == QW_ERR_INVALID_ARG
    sync_ok(L)   # the word was cleared
    # within max_context the same call is clean
    L.attention_decode(q, kc, vc, cl, base, 130, nh, nkv, hd, hd ** -0.5, out,
                       torch.zeros(L.attention_decode_workspace_size(B, 130, nh, hd), dtype=torch.uint8, device="cuda"))
    sync_ok(L)


ROPE_DECODE_CASES = {
    # name: (context lengths, q heads, kv heads, tp)
    "mixed_tp2": ([1, 63, 64, 65, 700], 16, 8, 2),
    "bench_shape": ([2049] * 8, 16, 8, 2),
    "group1_tp1": ([130, 2049, 1], 8, 8, 1),
    "group4": ([700, 2049], 32, 8, 2),
    "not_stored": ([0, 5, 300], 16, 8, 2),    # sequence 0: slot -1, no keys
}


@pytest.mark.parametrize("case", sorted(ROPE_DECODE_CASES))
@pytest.mark.parametrize("history_ready", [False, True])
def test_attention_decode_rope(L, case, history_ready):
    """QK-norm + RoPE + KV store folded into decode attention, against the
    oracle: the stored k (two roundings) and the bit-copied v, and the
    attention output over the cache with this step's rows in place."""
    ctx, nh, nkv, tp = ROPE_DECODE_CASES[case]
    hd, B = 128, len(ctx)
    m = si.ModelShape(vocab=64, hidden=64, n_heads=nh, n_kv_heads=nkv, head_dim=hd, intermediate=64, n_layers=1,
                      tp=tp, dtype="bf16", max_position=4096)
    cap = [c + 3 for c in ctx]
    base = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int32)
    S = int(sum(cap))
    width = tp * (nh // tp + 2 * (nkv // tp)) * hd
    qkv = si.normal(0, f"dr.{case}.qkv", (B, width), 1.0, "bf16")
    qg = (si.normal(0, f"dr.{case}.qg", (hd,), 0.2, "f32") + 1.0).to(torch.bfloat16)
    kg = (si.normal(0, f"dr.{case}.kg", (hd,), 0.2, "f32") + 1.0).to(torch.bfloat16)
    kc = si.normal(0, f"dr.{case}.k", (S, nkv, hd), 1.0, "bf16")
    vc = si.normal(0, f"dr.{case}.v", (S, nkv, hd), 1.0, "bf16")
    pos = torch.tensor([max(c - 1, 0) for c in ctx], dtype=torch.int64)
    slots = torch.tensor([int(base[b]) + ctx[b] - 1 if ctx[b] > 0 else -1 for b in range(B)], dtype=torch.int64)
    cs = L.rope_cos_sin_table(m.max_position, hd, m.rope_theta)
    kc_d, vc_d = dev(kc.clone()), dev(vc.clone())
    out = torch.full((B, nh * hd), 7.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc = max(ctx)
    ws = torch.zeros(L.attention_decode_workspace_size(B, max(mc, 1), nh, hd), dtype=torch.uint8, device="cuda")
    L.attention_decode_rope(dev(qkv), nh, nkv, hd, tp, dev(pos), dev(cs), dev(qg), dev(kg), m.eps, dev(slots),
                            kc_d, vc_d, err, dev(torch.tensor(ctx, dtype=torch.int32)), dev(torch.tensor(base)),
                            max(mc, 1), hd ** -0.5, out, ws, history_ready=history_ready)
    sync_ok(L)
    assert int(err.item()) == 0
    assert int(ws[:64 * 1024].view(torch.int32).abs().sum()) == 0
    # oracle: split the merged rows per shard, norm, rope, store, attend
    cos_t, sin_t = O.rope_cos_sin(m.max_position, hd, m.rope_theta)
    nh_l, nkv_l = nh // tp, nkv // tp
    x = qkv.double().numpy()
    wr = (nh_l + 2 * nkv_l) * hd
    qs, ks, vs = [], [], []
    for r in range(tp):
        blk = x[:, r * wr:(r + 1) * wr]
        qs.append(blk[:, : nh_l * hd].reshape(B, nh_l, hd))
        ks.append(blk[:, nh_l * hd:(nh_l + nkv_l) * hd].reshape(B, nkv_l, hd))
        vs.append(blk[:, (nh_l + nkv_l) * hd:].reshape(B, nkv_l, hd))
    q = O.apply_rope(O.rms_norm(np.concatenate(qs, 1), qg.double().numpy(), m.eps, "bf16"), pos.numpy(), cos_t,
                     sin_t, "bf16")
    k = O.apply_rope(O.rms_norm(np.concatenate(ks, 1), kg.double().numpy(), m.eps, "bf16"), pos.numpy(), cos_t,
                     sin_t, "bf16")
    v = np.concatenate(vs, 1)
    kc_n, vc_n = to_np(kc_d), to_np(vc_d)
    kd, vd = kc.double().numpy(), vc.double().numpy()
    live = [b for b in range(B) if ctx[b] > 0]
    rows = [int(slots[b]) for b in live]
    assert np.array_equal(vc_n[rows], v[live])                          # v: bit copy into the last row
    assert_within_ulps(kc_n[rows], k[live], 2.0, 0.97, "stored k")       # k: two roundings, as qkv_norm_rope
    others = np.ones(S, bool)
    others[rows] = False
    assert np.array_equal(kc_n[others], kd[others]) and np.array_equal(vc_n[others], vd[others])
    got = to_np(out).reshape(B, nh, hd)
    for b in range(B):
        if ctx[b] == 0:
            assert np.all(got[b] == 0.0)
    kref = [kc_n[base[b]:base[b] + ctx[b]].astype(np.float64) for b in live]   # the cache as stored
    vref = [vc_n[base[b]:base[b] + ctx[b]].astype(np.float64) for b in live]
    ref = O.attention_decode(q[live], kref, vref, hd ** -0.5, "bf16")
    _assert_decode_close(got[live], ref, vd, case)


def _paged_cache(name, lens, nkv, hd, block_size, spare_blocks=3, poison=False):
    """A cache of shuffled blocks: sequence s's position p at row
    table[s, p // block_size] * block_size + p % block_size.  Returns the
    cache, the table and each sequence's keys/values in position order."""
    blocks = [(L + block_size - 1) // block_size for L in lens]
    n_blocks = sum(blocks) + spare_blocks
    perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(7)).to(torch.int32)
    max_blocks = max(max(blocks), 1)
    table = torch.full((len(lens), max_blocks), -1, dtype=torch.int32)
    nxt = 0
    for s_, nb in enumerate(blocks):
        table[s_, :nb] = perm[nxt:nxt + nb]
        nxt += nb
    fill = float("nan") if poison else 0.0
    kc = torch.full((n_blocks * block_size, nkv, hd), fill, dtype=torch.bfloat16)
    vc = torch.full((n_blocks * block_size, nkv, hd), fill, dtype=torch.bfloat16)
    ks, vs = [], []
    for s_, L_ in enumerate(lens):
        k = si.normal(0, f"{name}.k{s_}", (L_, nkv, hd), 1.0, "bf16")
        v = si.normal(0, f"{name}.v{s_}", (L_, nkv, hd), 1.0, "bf16")
        pos = torch.arange(L_)
        rows = table[s_, pos // block_size].long() * block_size + pos % block_size
        kc[rows] = k
        vc[rows] = v
        ks.append(k.double().numpy())
        vs.append(v.double().numpy())
    return kc, vc, table, ks, vs


@pytest.mark.parametrize("lens,nh,nkv,block_size,history_ready",
                         [([1, 300, 2049, 256, 257], 16, 8, 256, False), ([700, 64, 1000], 32, 8, 64, True),
                          ([2049] * 8, 16, 8, 256, True)])
def test_attention_decode_paged(L, lens, nh, nkv, block_size, history_ready):
    """Decode attention through a block table over shuffled cache blocks."""
    hd, B = 128, len(lens)
    kc, vc, table, ks, vs = _paged_cache(f"pd{len(lens)}", lens, nkv, hd, block_size, poison=True)
    q = si.normal(0, f"pd{len(lens)}.q", (B, nh, hd), 1.0, "bf16")
    out = torch.full((B, nh * hd), 7.0, dtype=torch.bfloat16, device="cuda")
    mc = table.shape[1] * block_size
    ws = torch.zeros(L.attention_decode_workspace_size(B, mc, nh, hd), dtype=torch.uint8, device="cuda")
    L.attention_decode_paged(dev(q), dev(kc), dev(vc), dev(torch.tensor(lens, dtype=torch.int32)), dev(table),
                             block_size, mc, nh, nkv, hd, hd ** -0.5, out, ws, history_ready=history_ready)
    sync_ok(L)
    ref = O.attention_decode(q.double().numpy(), ks, vs, hd ** -0.5, "bf16")
    got = to_np(out).reshape(B, nh, hd)
    _assert_decode_close(got, ref, np.concatenate(vs), "paged")


@pytest.mark.parametrize("Lk,Lq,nh,nkv", [([600, 130, 256], [90, 130, 1], 16, 8), ([1024, 300], [1024, 44], 16, 4)])
def test_attention_prefill_paged_prefix(L, Lk, Lq, nh, nkv):
    """Prefix-cache prefill: Lq new queries per sequence over Lk keys (the
    cached prefix plus the new tokens), all read through a block table."""
    hd, bs = 128, 256
    kc, vc, table, ks, vs = _paged_cache(f"pp{len(Lk)}", Lk, nkv, hd, bs, poison=True)
    q = si.normal(0, f"pp{len(Lk)}.q", (sum(Lq), nh, hd), 1.0, "bf16")
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(Lq)]), dtype=torch.int32)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(Lk)]), dtype=torch.int32)
    out = torch.empty(sum(Lq), nh * hd, dtype=torch.bfloat16, device="cuda")
    L.attention_prefill_paged(dev(q), dev(kc), dev(vc), dev(cu_q), dev(cu_k), dev(table), bs, max(Lq), nh, nkv, hd,
                              hd ** -0.5, out)
    sync_ok(L)
    qd = q.double().numpy()
    refs = []
    for s_ in range(len(Lk)):
        a, b_ = int(cu_q[s_]), int(cu_q[s_ + 1])
        qfull = np.zeros((Lk[s_], nh, hd))
        qfull[Lk[s_] - Lq[s_]:] = qd[a:b_]
        o = O.attention_prefill(qfull, ks[s_], vs[s_], [0, Lk[s_]], hd ** -0.5, "bf16")
        refs.append(o[Lk[s_] - Lq[s_]:])
    ref = np.concatenate(refs)
    got = to_np(out).reshape(-1, nh, hd)
    err = np.abs(got - ref)
    assert np.all(err <= _attn_tol(ref, np.concatenate(vs))), float(np.nanmax(err))


# ----------------------------------------------------------------------------
# lm_head and argmax
# ----------------------------------------------------------------------------

def test_argmax_lowest_index_on_ties(L):
    """A row is split over several CTAs (contiguous ranges of 512 columns
    here): ties inside one range and across ranges both go to the lowest index."""
    x = si.normal(0, "am.x", (6, 4096), 1.0, "bf16")
    x[0, 100] = 9.0
    x[0, 50] = 9.0          # tie inside one range: 50 wins
    x[1, 4095] = 9.0        # the last column of the last range
    x[2, :] = -1.0          # all equal: 0 wins
    x[3, 3000] = 9.0
    x[3, 600] = 9.0         # tie across ranges: 600 wins
    x[4, 511] = 9.0
    x[4, 512] = 9.0         # tie at a range boundary: 511 wins
    x[5, :] = float("-inf")
    x[5, 4000] = -3.0
    out = torch.empty(6, dtype=torch.int64, device="cuda")
    L.argmax(dev(x), out)
    sync_ok(L)
    assert list(out.cpu().numpy()) == list(O.greedy(x.double().numpy()))
    assert out[0].item() == 50 and out[2].item() == 0 and out[3].item() == 600 and out[4].item() == 511


def test_argmax_full_vocabulary_rows(L):
    """Rows of the lm_head's width (151936, ragged over the CTAs of a row)."""
    x = si.normal(0, "am.full", (9, 151936), 1.0, "bf16")
    x[1, 151935] = 9.0
    x[2, 0] = 9.0
    x[3, 75968] = 9.0
    x[3, 75967] = 9.0
    out = torch.empty(9, dtype=torch.int64, device="cuda")
    L.argmax(dev(x), out)
    sync_ok(L)
    assert list(out.cpu().numpy()) == list(O.greedy(x.double().numpy()))


@pytest.mark.parametrize("tp", [1, 2, 4])
@pytest.mark.parametrize("n_out", [3, 300])
def test_lm_head_with_last_token_select(L, tp, n_out):
    V, H, T = 4096, 1024, 400
    table = si.normal(0, "lm.W", (V, H), 0.02, "bf16")
    hidden = si.normal(0, "lm.h", (T, H), 1.0, "bf16")
    last = si.uniform_int(0, "lm.idx", (n_out,), 0, T).to(torch.int32)
    logits = torch.empty(n_out, V, dtype=torch.bfloat16, device="cuda")
    nt = torch.empty(n_out, dtype=torch.int64, device="cuda")
    ws = torch.zeros(L.lm_head_workspace_size(n_out, V, H, tp, torch.bfloat16), dtype=torch.uint8, device="cuda")
    L.lm_head(dev(hidden), dev(last), n_out, dev(table), tp, logits, nt, ws)
    sync_ok(L)
    m = si.QWEN3_0_6B.replace(vocab=V)
    cu = None
    ref = O.compute_logits(m, table.double().numpy(), hidden.double().numpy()[last.numpy()], tp, cu)
    got = to_np(logits)
    acc = 2.0 ** -18 * (np.abs(hidden.double().numpy()[last.numpy()]) @ np.abs(table.double().numpy()).T)
    assert_within_ulps(got, ref, 1.0, 0.9, "logits", atol=acc)
    assert np.array_equal(nt.cpu().numpy(), O.greedy(got))     # argmax of the kernel's own logits: exact


@pytest.mark.parametrize("T,nh,nkv,tp", [(1, 16, 8, 2), (300, 16, 8, 2), (1000, 16, 8, 1), (257, 8, 8, 2),
                                         (129, 32, 8, 2),
                                         (2500, 16, 8, 2),    # 256-row tiles, the last one's second half partial
                                         (4200, 32, 8, 2)])   # 256-row tiles, the last one's second half past T
def test_qkv_gemm_epilogue_equals_two_step_path(L, T, nh, nkv, tp):
    """qw_qkv_gemm_norm_rope_store_kv against qw_gemm + qw_qkv_norm_rope_store_kv:
    q, both caches (NaN-poisoned rows left alone) and the error count identical
    bit for bit, including invalid positions, slot -1 and out-of-range slots.
    (The reference GEMM runs on at least 128 rows so that it takes the same
    128 x 256 tile path, whose rows do not depend on one another.)"""
    H, hd = 1024, 128
    N = (nh + 2 * nkv) * hd
    A = si.normal(0, f"qe.{T}.{nh}.a", (T, H), 1.0, "bf16")
    W = dev(si.normal(0, f"qe.{T}.{nh}.w", (N, H), 0.05, "bf16"))
    qg = dev((si.normal(0, f"qe.{T}.qg", (hd,), 0.2, "f32") + 1.0).to(torch.bfloat16))
    kg = dev((si.normal(0, f"qe.{T}.kg", (hd,), 0.2, "f32") + 1.0).to(torch.bfloat16))
    max_pos = 4096
    pos = si.uniform_int(0, f"qe.{T}.pos", (T,), 0, max_pos)
    slots = torch.randperm(T + 10, generator=torch.Generator().manual_seed(T))[:T].to(torch.int64)
    if T > 4:
        pos[1], pos[3] = -1, max_pos + 7          # invalid positions: q row zero, nothing stored
        slots[2], slots[4] = -1, T + 10 + 3       # not stored; out of range (counted)
    cs = L.rope_cos_sin_table(max_pos, hd, 1e6).cuda()
    num_slots = T + 10
    caches = [torch.full((num_slots, nkv, hd), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    q1 = torch.full((T, nh * hd), 5.0, dtype=torch.bfloat16, device="cuda")
    q2 = q1.clone()
    e1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    e2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    # reference: the two calls
    Tp = max(T, 128)
    Ap = torch.zeros(Tp, H, dtype=torch.bfloat16)
    Ap[:T] = A
    qkv = torch.empty(Tp, N, dtype=torch.bfloat16, device="cuda")
    L.gemm(dev(Ap), W, qkv, N, tp, L.QW_GEMM_COLUMN, L.QW_EPI_NONE)
    L.qkv_norm_rope_store_kv(qkv[:T], nh, nkv, hd, tp, dev(pos), cs, qg, kg, 1e-6, dev(slots), caches[0], caches[1],
                             q1, e1)
    # fused
    L.qkv_gemm_norm_rope_store_kv(dev(A), W, nh, nkv, hd, tp, dev(pos), cs, qg, kg, 1e-6, dev(slots), caches[2],
                                  caches[3], q2, e2)
    sync_ok(L)
    assert torch.equal(q1.view(torch.int16), q2.view(torch.int16))
    assert torch.equal(caches[0].view(torch.int16), caches[2].view(torch.int16))
    assert torch.equal(caches[1].view(torch.int16), caches[3].view(torch.int16))
    assert int(e1.item()) == int(e2.item()) == (3 if T > 4 else 0)   # two positions, one slot


@pytest.mark.parametrize("M,N,K,tp", [(1, 1024, 2048, 2), (300, 1024, 2048, 2), (130, 1024, 3072, 2),
                                      (200, 512, 1024, 1), (257, 2048, 1024, 4),
                                      (9800, 1024, 2048, 2)])   # 256-row tiles, the last one partial
def test_gemm_add_rmsnorm(L, M, N, K, tp):
    """Row-parallel GEMM + residual add + RMSNorm in one launch, against the two
    calls it replaces (qw_gemm ROW_REDUCE on at least 128 rows, the same tile
    path, then qw_add_rmsnorm) and against the oracle.  The new residual is the
    same bits; y rounds a sum of squares taken in another order, so it may sit
    one bf16 step away where it lies next to a rounding midpoint."""
    A = si.normal(0, f"gar.{M}.{N}.a", (M, K), 1.0, "bf16")
    Wf = si.normal(0, f"gar.{M}.{N}.w", (N, K), 0.05, "bf16")           # checkpoint [N, K]
    W = torch.stack([Wf[:, r * (K // tp):(r + 1) * (K // tp)] for r in range(tp)]).contiguous()
    R = si.normal(0, f"gar.{M}.{N}.r", (M, N), 1.0, "bf16")
    g = (si.normal(0, f"gar.{M}.{N}.g", (N,), 0.1, "f32") + 1.0).to(torch.bfloat16)
    eps = 1e-6
    res = dev(R.clone())
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    L.gemm_add_rmsnorm(dev(A), dev(W), res, dev(g), eps, y, tp)
    # the two calls, on a copy padded to 128 rows
    Mp = max(M, 128)
    Ap = torch.zeros(Mp, K, dtype=torch.bfloat16)
    Ap[:M] = A
    o = torch.empty(Mp, N, dtype=torch.bfloat16, device="cuda")
    L.gemm(dev(Ap), dev(W), o, N, tp, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_NONE)
    res2 = dev(R.clone())
    y2 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    L.add_rmsnorm(o[:M], res2, res2, dev(g), eps, y2)
    sync_ok(L)
    assert torch.equal(res.view(torch.int16), res2.view(torch.int16))
    assert_within_ulps(to_np(y), to_np(y2), 1.0, 0.99, "y vs two calls")
    # the oracle: o = row-parallel linear (one rounding), then add_rms_forward
    xs = [A.double().numpy()[:, r * (K // tp):(r + 1) * (K // tp)] for r in range(tp)]
    o_ref = O.row_parallel_linear(xs, Wf.double().numpy(), tp, "bf16")
    y_ref, s_ref = O.add_rms_norm(o_ref, R.double().numpy(), g.double().numpy(), eps, "bf16")
    acc = 2.0 ** -18 * (np.abs(A.double().numpy()) @ np.abs(Wf.double().numpy()).T)
    assert_within_ulps(to_np(res), s_ref, 1.0, 0.95, "residual", atol=acc + bf16_ulp(o_ref))
    # y = s * inv * gamma: a residual one step of o away (o and r can nearly cancel) moves
    # y by that step times the row's 1/rms and gamma
    inv = 1.0 / np.sqrt(np.mean(s_ref * s_ref, axis=1, keepdims=True) + eps)
    slack = (acc + bf16_ulp(o_ref)) * inv * np.abs(g.double().numpy())[None, :]
    assert_within_ulps(to_np(y), y_ref, 2.0, 0.95, "y", atol=slack + 2.0 ** -9)
