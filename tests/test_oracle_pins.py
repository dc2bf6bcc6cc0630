"""Pins of the CPU oracle to things other than itself.

Each test checks an oracle function against what the pages print (golden
fixtures under tests/golden/, each with its citation), a closed form, a
library routine for a special case, brute force, or an invariant.  The cases
are chosen so that a plausible slip (a dropped term, a wrong sign or index, a
swapped operand or half) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import expit

import oracle as O
import seeded_inputs as si

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------------------
# rounding
# ----------------------------------------------------------------------------

def test_bf16_round_matches_torch_cast_on_fp32_values():
    # torch's fp32 -> bf16 conversion is round-to-nearest-even; on values that
    # are exactly fp32 the oracle's float64 -> bf16 rounding must agree bit for bit.
    e = RNG.integers(-130, 120, size=200000)
    m = RNG.uniform(1.0, 2.0, size=e.size) * RNG.choice([-1.0, 1.0], size=e.size)
    x32 = np.ldexp(m, e).astype(np.float32)
    ours = O.bf16_round(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(ours, ref)


def test_bf16_round_brute_force_on_float64_inputs():
    # float64 inputs carry more bits than fp32, so the torch-cast pin above does
    # not reach them: compare with the two bf16 neighbours found by brute force
    # (8 significant bits via math.frexp, or the 2^-133 grid below 2^-126) and
    # pick the nearer, the even one on a tie
    rng = np.random.default_rng(99)
    e = rng.integers(-138, 128, size=3000)
    x = np.ldexp(rng.uniform(1.0, 2.0, size=e.size), e) * rng.choice([-1.0, 1.0], size=e.size)
    ties = np.ldexp(1.0 + (2 * rng.integers(0, 128, size=300) + 1) * 2.0 ** -8, rng.integers(-100, 100, size=300))
    x = np.concatenate([x, ties, -ties])
    got = O.bf16_round(x)
    for xi, gi in zip(x, got):
        a = abs(float(xi))
        if a >= 2.0 ** -126:
            _, ex = math.frexp(a)
            step = 2.0 ** (ex - 8)
        else:
            step = 2.0 ** -133
        lo = math.floor(a / step) * step
        hi = lo + step
        if a - lo < hi - a or (a - lo == hi - a and (lo / step) % 2 == 0):
            want = lo
        else:
            want = hi
        if want > (2.0 - 2.0 ** -7) * 2.0 ** 127:
            want = math.inf
        assert gi == math.copysign(want, xi), (xi, gi, want)


def test_bf16_round_ties_and_limits():
    u = 2.0 ** -7          # bf16 spacing in [1, 2)
    assert O.bf16_round(1.0 + u / 2)[()] == 1.0                 # tie -> even mantissa
    assert O.bf16_round(1.0 + 3 * u / 2)[()] == 1.0 + 2 * u     # tie -> even mantissa
    assert O.bf16_round(1.0 + u / 2 + 1e-12)[()] == 1.0 + u     # just above the tie
    assert O.bf16_round(-(1.0 + u / 2 + 1e-12))[()] == -(1.0 + u)
    assert O.bf16_round(3.0e39)[()] == np.inf
    assert O.bf16_round(2.0 ** -133)[()] == 2.0 ** -133          # smallest subnormal
    assert O.bf16_round(0.0)[()] == 0.0


# ----------------------------------------------------------------------------
# vocab-parallel embedding and lm_head
# ----------------------------------------------------------------------------

def test_toy_embedding_two_ranks(golden):
    g = golden("vh_toy_embedding.json")
    table = np.array(g["table"], dtype=np.float64)
    assert O.vocab_range(4, 2, 0) == tuple(g["rank0_range"])
    p0 = O.vocab_embedding_rank(g["tokens"], table, g["tp"], 0)
    p1 = O.vocab_embedding_rank(g["tokens"], table, g["tp"], 1)
    assert np.array_equal(p0, g["rank0_partial"])
    assert np.array_equal(p1, g["rank1_partial"])
    s = O.vocab_parallel_embedding(g["tokens"], table, g["tp"])
    assert np.array_equal(s, g["sum"])
    assert np.array_equal(s, O.embedding_unsharded(g["tokens"], table))


def test_worked_12_word_example(golden):
    g = golden("vpe_worked_example.json")
    V, D = g["vocab"], g["dim"]
    table = (np.arange(V)[:, None] * 10.0 + np.arange(D)[None, :])
    ids = np.array(g["ids"])
    assert O.vocab_range(V, 2, 0) == tuple(g["rank0_range"])
    assert O.vocab_range(V, 2, 1) == tuple(g["rank1_range"])
    tr = {}
    z0 = O.vocab_embedding_rank(ids, table, 2, 0, trace=tr)
    assert np.array_equal(tr["mask"], g["rank0_mask"])
    assert np.array_equal(tr["local"], g["rank0_local"])
    assert np.array_equal(tr["lookup"], g["rank0_lookup"])
    assert np.array_equal(z0, g["rank0_zeroed"])
    z1 = O.vocab_embedding_rank(ids, table, 2, 1)
    assert np.array_equal(z1, g["rank1_zeroed"])
    assert np.array_equal(O.vocab_parallel_embedding(ids, table, 2), g["sum"])
    ref = F.embedding(torch.from_numpy(ids), torch.from_numpy(table)).numpy()
    assert np.array_equal(ref, g["nn_embedding"])


@pytest.mark.parametrize("tp", [1, 2, 4])
def test_embedding_sharded_equals_unsharded_at_boundaries(tp):
    V, H = 64, 8
    table = RNG.standard_normal((V, H))
    ids = np.array([0, V // 4 - 1, V // 4, V // 2 - 1, V // 2, 3 * V // 4 - 1, 3 * V // 4, V - 1, 5, 40])
    s = O.vocab_parallel_embedding(ids, table, tp)
    ref = F.embedding(torch.from_numpy(ids), torch.from_numpy(table)).numpy()
    assert np.array_equal(s, ref)
    # exactly one rank owns each id
    owners = sum((O.vocab_embedding_rank(ids, table, tp, r) != 0).any(axis=1).astype(int) for r in range(tp))
    assert np.all(owners == 1)


def test_lm_head_toy_shapes_and_gather(golden):
    g = golden("vh_lm_head_toy.json")
    W = np.array(g["W"], dtype=np.float64)
    x = RNG.standard_normal((g["x_rows"], 2))
    s0 = O.parallel_lm_head_rank(x, W, 2, 0, "f64")
    s1 = O.parallel_lm_head_rank(x, W, 2, 1, "f64")
    assert s0.shape == tuple(g["rank0_shape"]) and s1.shape == tuple(g["rank1_shape"])
    full = F.linear(torch.from_numpy(x), torch.from_numpy(W)).numpy()
    assert np.allclose(s0, full[:, g["rank0_vocab"]], rtol=0, atol=1e-12)
    assert np.allclose(s1, full[:, g["rank1_vocab"]], rtol=0, atol=1e-12)
    m = si.TINY.replace(dtype="f64")
    assert np.allclose(O.compute_logits(m, W, x, 2), full, rtol=0, atol=1e-12)


def test_compute_logits_keeps_last_token_of_each_sequence():
    m = si.TINY.replace(dtype="f64")
    W = RNG.standard_normal((12, 4))
    h = RNG.standard_normal((9, 4))
    cu = np.array([0, 3, 4, 9])
    lg = O.compute_logits(m, W, h, 3, cu_seqlens=cu)
    assert lg.shape == (3, 12)
    assert np.allclose(lg, h[[2, 3, 8]] @ W.T, atol=1e-12)


def test_head_split_and_cache_shapes(golden):
    g = golden("vh_head_split.json")
    assert O.heads_per_rank(g["total_heads"], g["total_kv_heads"], g["tp"]) == tuple(g["heads_per_rank"])
    args = (g["layers"], g["blocks"], g["block_size"], g["total_kv_heads"], g["head_dim"])
    assert O.kv_cache_shape(*args, 1) == tuple(g["kv_cache_shape_tp1"])
    assert O.kv_cache_shape(*args, 2) == tuple(g["kv_cache_shape_tp2"])
    s, e = O.vocab_range(g["vocab"], 2, 1)
    assert e - s == g["vocab_per_rank_tp2"]
    wg = np.zeros((g["intermediate"], 1))
    assert O.gate_up_shard_weight(wg, wg, 2, 0).shape[0] == 2 * g["intermediate_per_rank_tp2"]
    with pytest.raises(AssertionError):
        O.heads_per_rank(16, 8, 3)


# ----------------------------------------------------------------------------
# linear family
# ----------------------------------------------------------------------------

def test_column_and_row_split_identities(golden):
    g = golden("tp_split_identity.json")
    X = np.array(g["X"], dtype=np.float64)
    W = np.array(g["W"], dtype=np.float64)        # the page's Y = X W orientation
    w = W.T                                         # F.linear weight: [out, in]
    assert np.array_equal(O.linear(X, w, "f64"), g["Y"])
    halves = [O.column_parallel_linear(X, w, 2, r, "f64") for r in range(2)]
    assert np.array_equal(halves[0], g["column_halves"][0])
    assert np.array_equal(halves[1], g["column_halves"][1])
    assert np.array_equal(np.concatenate(halves, -1), g["Y"])
    x_sh = [X[:, :2], X[:, 2:]]
    assert np.array_equal(O.row_parallel_linear(x_sh, w, 2, "f64"), g["Y"])
    only0 = O.row_parallel_linear([x_sh[0], np.zeros_like(x_sh[1])], w, 2, "f64")
    only1 = O.row_parallel_linear([np.zeros_like(x_sh[0]), x_sh[1]], w, 2, "f64")
    assert np.array_equal(only0, g["row_partials"][0])
    assert np.array_equal(only1, g["row_partials"][1])


@pytest.mark.parametrize("tp", [1, 2, 4])
def test_split_linear_equals_torch_linear(tp):
    x = RNG.standard_normal((5, 16))
    w = RNG.standard_normal((12, 16))
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(w)).numpy()
    col = np.concatenate([O.column_parallel_linear(x, w, tp, r, "f64") for r in range(tp)], -1)
    assert np.allclose(col, ref, atol=1e-12, rtol=0)
    k_l = 16 // tp
    row = O.row_parallel_linear([x[:, r * k_l:(r + 1) * k_l] for r in range(tp)], w, tp, "f64")
    assert np.allclose(row, ref, atol=1e-12, rtol=0)


def test_qkv_and_gate_up_shard_rows():
    nh, nkv, d, H = 4, 2, 3, 5
    wq = np.arange(nh * d * H).reshape(nh * d, H) * 1.0
    wk = -np.arange(nkv * d * H).reshape(nkv * d, H) - 1.0
    wv = 1000 + np.arange(nkv * d * H).reshape(nkv * d, H) * 1.0
    s1 = O.qkv_shard_weight(wq, wk, wv, nh, nkv, d, 2, 1)
    assert np.array_equal(s1[: 2 * d], wq[2 * d: 4 * d])
    assert np.array_equal(s1[2 * d: 3 * d], wk[d: 2 * d])
    assert np.array_equal(s1[3 * d:], wv[d: 2 * d])
    wg = np.arange(8.0)[:, None]
    wu = 100 + np.arange(8.0)[:, None]
    assert np.array_equal(O.gate_up_shard_weight(wg, wu, 2, 1)[:, 0], [4, 5, 6, 7, 104, 105, 106, 107])


# ----------------------------------------------------------------------------
# RMSNorm
# ----------------------------------------------------------------------------

def test_rmsnorm_closed_forms():
    # constant vector c: y = c / sqrt(c^2 + eps) * gamma
    for c in (1e-3, 0.5, -7.0):
        x = np.full((1, 6), c)
        gamma = np.array([1.0, 2.0, -0.5, 3.0, 1.0, 0.25])
        y = O.rms_norm(x, gamma, 1e-6, "f64")
        assert np.allclose(y, c / math.sqrt(c * c + 1e-6) * gamma, rtol=1e-14, atol=0)
    # [3, 4]: mean of squares 12.5
    y = O.rms_norm(np.array([[3.0, 4.0]]), np.array([2.0, 0.5]), 0.0, "f64")
    assert np.allclose(y, [[3 / math.sqrt(12.5) * 2, 4 / math.sqrt(12.5) * 0.5]], rtol=1e-15)


def test_rmsnorm_matches_torch_rms_norm_and_invariants():
    x = RNG.standard_normal((7, 64)) * 3
    gamma = 1 + 0.1 * RNG.standard_normal(64)
    ref = F.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(gamma), eps=1e-6).numpy()
    y = O.rms_norm(x, gamma, 1e-6, "f64")
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-14)
    # scale invariance and unit mean square when gamma = 1 and eps << rms^2
    assert np.allclose(O.rms_norm(5 * x, gamma, 1e-12, "f64"), O.rms_norm(x, gamma, 1e-12, "f64"), rtol=1e-12)
    y1 = O.rms_norm(x, np.ones(64), 1e-12, "f64")
    assert np.allclose(np.mean(y1 * y1, -1), 1.0, rtol=1e-12)


def test_add_rmsnorm_returns_rounded_sum_as_residual():
    x = np.array([[1.0, 2.0 ** -9, 3.0, 4.0]])
    r = np.array([[1.0, 1.0, -3.0, 0.0]])
    y, res = O.add_rms_norm(x, r, np.ones(4), 1e-6, "bf16")
    assert np.array_equal(res, [[2.0, 1.0, 0.0, 4.0]])        # 1 + 2^-9 rounds to 1 in bf16
    assert np.array_equal(y, O.rms_norm(res, np.ones(4), 1e-6, "bf16"))


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------

def test_rope_table_closed_form():
    cos_t, sin_t = O.rope_cos_sin(4, 4, 1e6)
    # d = 4: inv_freq = [theta^0, theta^(-2/4)] = [1, 1e-3]
    assert np.array_equal(cos_t[0], [1.0, 1.0]) and np.array_equal(sin_t[0], [0.0, 0.0])
    assert np.allclose(cos_t[3], [math.cos(3.0), math.cos(3e-3)], atol=1e-7)
    assert np.allclose(sin_t[3], [math.sin(3.0), math.sin(3e-3)], atol=1e-7)


def test_rope_is_complex_rotation_of_half_pairs():
    d = 16
    cos_t, sin_t = O.rope_cos_sin(64, d, 1e6)
    x = RNG.standard_normal((5, 3, d))
    pos = np.array([0, 1, 7, 33, 63])
    y = O.apply_rope(x, pos, cos_t, sin_t, "f64")
    z = (x[..., : d // 2] + 1j * x[..., d // 2:]) * (cos_t[pos] + 1j * sin_t[pos])[:, None, :]
    assert np.allclose(y[..., : d // 2], z.real, atol=1e-14)
    assert np.allclose(y[..., d // 2:], z.imag, atol=1e-14)
    assert np.array_equal(y[0], x[0])                                     # position 0: identity
    n_in = x[..., : d // 2] ** 2 + x[..., d // 2:] ** 2
    n_out = y[..., : d // 2] ** 2 + y[..., d // 2:] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-6)                           # |cos|^2+|sin|^2 = 1 in fp32


def test_rope_pairs_and_relative_position():
    d = 8
    cos_t, sin_t = O.rope_cos_sin(300, d, 1e4)
    x = np.zeros((1, 1, d))
    x[0, 0, 2] = 1.0
    y = O.apply_rope(x, np.array([5]), cos_t, sin_t, "f64")
    assert set(np.nonzero(y[0, 0])[0]) == {2, 2 + d // 2}
    q = RNG.standard_normal((1, 1, d))
    k = RNG.standard_normal((1, 1, d))

    def dot(m, n):
        return float(np.sum(O.apply_rope(q, [m], cos_t, sin_t, "f64") * O.apply_rope(k, [n], cos_t, sin_t, "f64")))
    assert abs(dot(10, 3) - dot(110, 103)) < 1e-4
    assert abs(dot(10, 3) - dot(3, 10)) > 1e-3                          # depends on the sign of m - n


# ----------------------------------------------------------------------------
# SiluAndMul
# ----------------------------------------------------------------------------

def test_silu_and_mul():
    g = RNG.standard_normal((4, 6)) * 4
    u = RNG.standard_normal((4, 6))
    y = O.silu_and_mul(np.concatenate([g, u], -1), "f64")
    assert np.allclose(y, g * expit(g) * u, rtol=1e-14, atol=1e-15)
    assert np.array_equal(O.silu_and_mul(np.array([[0.0, 5.0]]), "f64"), [[0.0]])
    assert abs(O.silu_and_mul(np.array([[40.0, 1.0]]), "f64")[0, 0] - 40.0) < 1e-12
    assert abs(O.silu_and_mul(np.array([[1.0, 40.0]]), "f64")[0, 0] - 40 * expit(1.0)) < 1e-12


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def _sdpa_ref(q, k, v, cu, scale):
    group = q.shape[1] // k.shape[1]
    out = np.zeros_like(q)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        qt = torch.from_numpy(q[a:b]).transpose(0, 1)
        kt = torch.from_numpy(k[a:b]).transpose(0, 1).repeat_interleave(group, 0)
        vt = torch.from_numpy(v[a:b]).transpose(0, 1).repeat_interleave(group, 0)
        o = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
        out[a:b] = o.transpose(0, 1).numpy()
    return out


def test_prefill_attention_matches_sdpa():
    nh, nkv, d = 6, 2, 8
    cu = [0, 5, 6, 13]
    q = RNG.standard_normal((13, nh, d))
    k = RNG.standard_normal((13, nkv, d))
    v = RNG.standard_normal((13, nkv, d))
    o = O.attention_prefill(q, k, v, cu, d ** -0.5, "f64")
    assert np.allclose(o, _sdpa_ref(q, k, v, cu, d ** -0.5), atol=1e-12)


def test_attention_special_cases():
    d = 4
    v = RNG.standard_normal((6, 1, d))
    k = RNG.standard_normal((6, 1, d))
    # one key: output equals its value
    o = O.attention_prefill(RNG.standard_normal((1, 1, d)), k[:1], v[:1], [0, 1], 0.5, "f64")
    assert np.allclose(o[0, 0], v[0, 0], atol=1e-15)
    # zero query: running mean of the visible values
    o = O.attention_prefill(np.zeros((6, 1, d)), k, v, [0, 6], 0.5, "f64")
    run_mean = np.cumsum(v[:, 0], 0) / np.arange(1, 7)[:, None]
    assert np.allclose(o[:, 0], run_mean, atol=1e-14)
    # identical keys: uniform weights, whatever the query
    o = O.attention_prefill(RNG.standard_normal((6, 1, d)), np.repeat(k[:1], 6, 0), v, [0, 6], 0.5, "f64")
    assert np.allclose(o[:, 0], run_mean, atol=1e-14)


def test_attention_causal_and_sequence_isolation():
    nh, nkv, d = 4, 2, 8
    cu = [0, 7, 12]
    q = RNG.standard_normal((12, nh, d))
    k = RNG.standard_normal((12, nkv, d))
    v = RNG.standard_normal((12, nkv, d))
    o = O.attention_prefill(q, k, v, cu, 0.3, "f64")
    k2, v2 = k.copy(), v.copy()
    k2[4] += 1.0
    v2[4] -= 2.0
    o2 = O.attention_prefill(q, k2, v2, cu, 0.3, "f64")
    assert np.array_equal(o[:4], o2[:4])            # earlier tokens of the same sequence
    assert np.array_equal(o[7:], o2[7:])            # the other sequence
    assert not np.allclose(o[4:7], o2[4:7])


def test_decode_attention_equals_prefill_row():
    nh, nkv, d, L = 4, 2, 8, 9
    q = RNG.standard_normal((L, nh, d))
    k = RNG.standard_normal((L, nkv, d))
    v = RNG.standard_normal((L, nkv, d))
    o = O.attention_prefill(q, k, v, [0, L], 0.35, "f64")
    for i in (0, 3, L - 1):
        od = O.attention_decode(q[i:i + 1], [k[: i + 1]], [v[: i + 1]], 0.35, "f64")
        assert np.allclose(od[0], o[i], atol=1e-13)


def test_greedy_lowest_index_on_ties():
    assert list(O.greedy(np.array([[1.0, 3.0, 3.0, 2.0], [0.0, -1.0, 0.0, 0.0]]))) == [1, 0]


# ----------------------------------------------------------------------------
# layer / model structure
# ----------------------------------------------------------------------------

SMALL = si.ModelShape(vocab=64, hidden=32, n_heads=8, n_kv_heads=4, head_dim=8, intermediate=64,
                      n_layers=2, tp=1, dtype="f32", max_position=64, weight_sigma=0.2, gamma_sigma=0.2)


def _weights(m):
    return O.load_weights(m)


def _run(m, w, tp, seq_lens, dtype):
    mm = m.replace(dtype=dtype)
    b = si.prefill_batch(m, seq_lens)
    cache = O.KVCache(m.n_layers, b.num_slots, m.n_kv_heads, m.head_dim, tp)
    ctx = O.AttnContext(True, b.slot_mapping.numpy(), cu_seqlens=b.cu_seqlens.numpy())
    h = O.model_forward(mm, w, b.ids.numpy(), b.positions.numpy(), ctx, cache)
    return h, cache, b


@pytest.mark.parametrize("tp", [2, 4])
def test_model_sharded_equals_unsharded(tp):
    w = _weights(SMALL)
    h1, c1, b = _run(SMALL, w, 1, [5, 3], "f64")
    ht, ct, _ = _run(SMALL, w, tp, [5, 3], "f64")
    assert np.allclose(h1, ht, rtol=0, atol=1e-12)
    nkv_l = SMALL.n_kv_heads // tp
    for l in range(SMALL.n_layers):
        k_cat = np.concatenate([ct.k[r][l] for r in range(tp)], axis=1)
        assert np.allclose(k_cat, c1.k[0][l], atol=1e-6)
        assert k_cat.shape[1] == nkv_l * tp
    m = SMALL.replace(dtype="f64")
    lg1 = O.compute_logits(m, w.embed, h1, 1, b.cu_seqlens.numpy())
    lgt = O.compute_logits(m, w.embed, ht, tp, b.cu_seqlens.numpy())
    assert np.allclose(lg1, lgt, atol=1e-12)


def test_layer_residual_path():
    # with o_proj = 0 and down_proj = 0 both sub-blocks add nothing: the layer
    # returns h = 0 and residual = its input
    w = _weights(SMALL)
    lw = w.layers[0]
    lw.wo[:] = 0
    lw.wd[:] = 0
    m = SMALL.replace(dtype="f64")
    b = si.prefill_batch(m, [4])
    cache = O.KVCache(1, b.num_slots, m.n_kv_heads, m.head_dim, 1)
    ctx = O.AttnContext(True, b.slot_mapping.numpy(), cu_seqlens=b.cu_seqlens.numpy())
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    x = RNG.standard_normal((4, m.hidden))
    r0 = RNG.standard_normal((4, m.hidden))
    h, res = O.decoder_layer(m, lw, 0, b.positions.numpy(), x, None, ctx, cache, *cos_sin)
    assert np.array_equal(h, np.zeros_like(h)) and np.array_equal(res, x)
    h, res = O.decoder_layer(m, lw, 0, b.positions.numpy(), x, r0, ctx, cache, *cos_sin)
    assert np.allclose(res, x + r0, atol=1e-15)


def test_batch_independence_and_prefill_decode_consistency():
    w = _weights(SMALL)
    m = SMALL.replace(dtype="f64")
    h_both, _, b = _run(SMALL, w, 2, [6, 4], "f64")
    ids = b.ids.numpy()
    # sequence 1 alone gives the same hidden states
    b1 = si.prefill_batch(SMALL, [4])
    cache = O.KVCache(2, 4, m.n_kv_heads, m.head_dim, 2)
    ctx = O.AttnContext(True, np.arange(4), cu_seqlens=np.array([0, 4]))
    h1 = O.model_forward(m, w, ids[6:], np.arange(4), ctx, cache)
    assert np.allclose(h1, h_both[6:], atol=1e-12)
    # prefill of the first 5 tokens of sequence 0, then decode token 5 from the cache
    cache = O.KVCache(2, 6, m.n_kv_heads, m.head_dim, 2)
    ctx = O.AttnContext(True, np.arange(5), cu_seqlens=np.array([0, 5]))
    O.model_forward(m, w, ids[:5], np.arange(5), ctx, cache)
    dctx = O.AttnContext(False, np.array([5]), seq_base=np.array([0]), context_lens=np.array([6]))
    hd = O.model_forward(m, w, ids[5:6], np.array([5]), dctx, cache)
    assert np.allclose(hd[0], h_both[5], atol=1e-12)
    lg_d = O.compute_logits(m, w.embed, hd, 2)
    lg_p = O.compute_logits(m, w.embed, h_both, 2, cu_seqlens=np.array([0, 6, 10]))
    assert np.allclose(lg_d[0], lg_p[0], atol=1e-12)


def test_kv_store_skips_minus_one_and_keeps_other_slots():
    c = O.KVCache(1, 6, 2, 4, 1)
    c.k[0][0][:] = 7.0
    c.v[0][0][:] = 9.0
    k = RNG.standard_normal((3, 2, 4)).astype(np.float32)
    v = RNG.standard_normal((3, 2, 4)).astype(np.float32)
    c.store(0, 0, k, v, np.array([4, -1, 1]))
    assert np.array_equal(c.k[0][0][4], k[0]) and np.array_equal(c.v[0][0][1], v[2])
    for s in (0, 2, 3, 5):
        assert np.all(c.k[0][0][s] == 7.0) and np.all(c.v[0][0][s] == 9.0)


def test_row_parallel_adds_partials_before_rounding():
    # partials 1 + 2^-8 and 2^-8: the exact sum 1 + 2^-7 is a bf16 value, while
    # rounding each partial first would give bf16(1 + 2^-8) + 2^-8 -> 1.0
    x = np.array([[1.0, 1.0]])
    w = np.array([[1.0 + 2.0 ** -8, 2.0 ** -8]])
    y = O.row_parallel_linear([x[:, :1], x[:, 1:]], w, 2, "bf16")
    assert y[0, 0] == 1.0 + 2.0 ** -7


def test_attention_block_uses_default_softmax_scale():
    # SDPA's default scale is 1/sqrt(head_dim): the layer's attention output must
    # equal it on the layer's own (traced) q, k, v
    w = _weights(SMALL)
    m = SMALL.replace(dtype="f64")
    b = si.prefill_batch(m, [7])
    cache = O.KVCache(1, b.num_slots, m.n_kv_heads, m.head_dim, 2)
    ctx = O.AttnContext(True, b.slot_mapping.numpy(), cu_seqlens=b.cu_seqlens.numpy())
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    tr = {}
    O.attention_block(m, w.layers[0], 0, b.positions.numpy(), RNG.standard_normal((7, m.hidden)), ctx,
                      cache, *cos_sin, trace=tr)
    for r in range(2):
        q, k, v = tr["q"][r], tr["k"][r], tr["v"][r]
        group = q.shape[1] // k.shape[1]
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(q).transpose(0, 1), torch.from_numpy(k).transpose(0, 1).repeat_interleave(group, 0),
            torch.from_numpy(v).transpose(0, 1).repeat_interleave(group, 0), is_causal=True).transpose(0, 1)
        assert np.allclose(tr["o"][r], ref.numpy(), atol=1e-12)


# ----------------------------------------------------------------------------
# sampler (temperature / top-p, Gumbel-max draw)
# ----------------------------------------------------------------------------

def test_sample_zero_temperature_is_greedy_and_shift_invariant():
    lg = np.array([[0.5, 2.0, 2.0, -1.0], [1.0, 1.0, 1.0, 1.0]])
    u = si.uniform01(0, "pin.sample.u", lg.shape).double().numpy()
    assert list(O.sample(lg, [0.0, 0.0], [0.9, 0.1], u)) == [1, 0]      # lowest index on ties
    t = O.sample(lg, [0.8, 1.3], [1.0, 0.6], u)
    assert np.array_equal(O.sample(lg + 7.25, [0.8, 1.3], [1.0, 0.6], u), t)


def test_sample_nucleus_of_a_worked_row():
    # logits [3, 1, 1, 0] at T = 1: p = [e^3, e, e, 1] / (e^3 + 2e + 1) = [0.7573, 0.1025, 0.1025, 0.0377];
    # P = 0.8 needs the first two distinct values, so the nucleus is {0, 1, 2} (the tie at 1 kept whole);
    # P = 0.97 needs all four.  u_3 near 1 gives token 3 a Gumbel value of about 13.8.
    lg = np.array([[3.0, 1.0, 1.0, 0.0]])
    u = np.array([[0.5, 0.5, 0.5, 1.0 - 1e-6]])
    assert O.sample(lg, [1.0], [0.8], u)[0] == 0
    assert O.sample(lg, [1.0], [0.97], u)[0] == 3
    u2 = np.array([[0.5, 0.5, 1.0 - 1e-6, 0.5]])
    assert O.sample(lg, [1.0], [0.8], u2)[0] == 2        # inside the nucleus, the large draw wins
    assert O.sample(lg, [1.0], [0.7], u2)[0] == 0        # P below m_1 = 0.757: only token 0
    assert O.sample(lg, [1.0], [1e-9], u2)[0] == 0


@pytest.mark.parametrize("T,P", [(0.7, 1.0), (1.5, 0.8)])
def test_sample_frequencies_follow_the_restricted_softmax(T, P):
    # many rows of the same logits, each with its own uniforms: the token
    # frequencies converge to softmax(l / T) over the nucleus, renormalised
    lg = np.array([1.2, -0.3, 0.4, 2.0, 0.0, -1.1])
    N = 120000
    u = si.uniform01(0, f"pin.sample.freq.{T}", (N, lg.size)).double().numpy()
    tok = O.sample(np.tile(lg, (N, 1)), np.full(N, T), np.full(N, P), u)
    p = np.exp(lg / T)
    p /= p.sum()
    order = np.argsort(-lg)
    keep = np.zeros(lg.size, bool)
    cum = np.cumsum(p[order])
    keep[order[:int(np.argmax(cum >= P * cum[-1])) + 1]] = True
    q = np.where(keep, p, 0.0)
    q /= q.sum()
    freq = np.bincount(tok, minlength=lg.size) / N
    assert np.all(freq[~keep] == 0)
    assert np.max(np.abs(freq - q)) < 5 * np.sqrt(0.25 / N), (freq, q)
