"""Pins of the oracle's layer and model ASSEMBLY to an independent composition.

The per-function pins (tests/test_oracle_pins.py) check each oracle step on
its own.  This file checks how the steps are put together: the order of the
sub-blocks, which gamma feeds which norm, where the residual is taken, that
QK-RMSNorm comes before RoPE, and that the model ends with the final
add+RMSNorm.  The composition below is written from the pages' forward order
with PyTorch library routines only (F.embedding, F.rms_norm, F.linear,
F.scaled_dot_product_attention with a causal mask and GQA, F.silu, complex
multiplication for the rotation) in float64, sharing no code with the
oracle:

  [SK] §1 Qwen3DecoderLayer.forward: input_layernorm (first layer: norm of the
       input, residual = input; later: add then norm) -> self_attn ->
       post_attention_layernorm (add then norm) -> mlp; returns (h, residual)
  [SK] §8 ① Qwen3Attention.forward: qkv_proj -> split q, k, v -> q_norm on q,
       k_norm on k (per head, over head_dim) -> rotary_emb(positions, q, k)
       -> attention -> o_proj
  [SK] §3 RoPE on the two halves of each head, theta 1e6, no scaling
  [SK] §4 SiluAndMul: silu(gate) * up after the merged gate_up projection
  [SK] §8 Qwen3Model: embed_tokens -> layers -> final norm (add then norm);
       the lm_head (tied to embed_tokens) projects the last token of each
       sequence ([SK] §6)

Every gamma is drawn distinct from 1 (gamma_sigma > 0), so that a swapped or
dropped gamma changes the result.  Mistakes this file is built to catch:
q_norm / k_norm gammas swapped, input / post-attention gammas swapped, RoPE
applied before QK-RMSNorm, the final norm's gamma dropped, a residual taken
at the wrong point.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
import seeded_inputs as si

# small but with every structural feature: GQA groups of 2, two layers,
# head_dim 8 (4 rotation pairs), tp 2 on the oracle side
SHAPE = si.ModelShape(vocab=96, hidden=32, n_heads=4, n_kv_heads=2, head_dim=8, intermediate=48,
                      n_layers=2, tp=2, dtype="f64", max_position=64, weight_sigma=0.2, gamma_sigma=0.25)


def _ck(m):
    """The checkpoint tensors (unsharded) as float64 torch tensors."""
    names = ["embed_tokens", "norm"]
    for l in range(m.n_layers):
        names += si.weight_names(l) + [f"layer{l}.{x}" for x in
                                       ("input_layernorm", "post_attention_layernorm", "q_norm", "k_norm")]
    return {n: si.checkpoint_tensor(m.replace(dtype="f32"), n).double() for n in names}


def _rotate(x, positions, theta):
    """RoPE on [T, heads, d] with the halves pairing, as a complex rotation by position * f_i.

    The frequencies are those of the pages' fp32 table: f_i = 1 / theta^(2i/d)
    and the angle p * f_i each rounded to fp32, as the pages' float32 outer
    product makes them."""
    d = x.shape[-1]
    i2 = torch.arange(0, d, 2, dtype=torch.float64)
    inv = (1.0 / torch.pow(torch.tensor(theta, dtype=torch.float64), i2 / d)).float()
    ang = (positions.double()[:, None] * inv.double()[None, :]).float().double()
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]
    z = torch.complex(x[..., : d // 2], x[..., d // 2:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def _reference_forward(m, ck, ids, positions, cu_seqlens):
    """The whole model in float64 torch, unsharded: returns (final hidden, last-token logits)."""
    nh, nkv, d, H = m.n_heads, m.n_kv_heads, m.head_dim, m.hidden
    T = ids.shape[0]
    x = F.embedding(ids, ck["embed_tokens"])
    residual = None
    for l in range(m.n_layers):
        p = f"layer{l}."
        # input_layernorm, fused with the residual add after the first layer
        if residual is None:
            residual = x
        else:
            residual = x + residual
        h = F.rms_norm(residual, (H,), weight=ck[p + "input_layernorm"], eps=m.eps)
        # self attention
        q = F.linear(h, ck[p + "q_proj"]).view(T, nh, d)
        k = F.linear(h, ck[p + "k_proj"]).view(T, nkv, d)
        v = F.linear(h, ck[p + "v_proj"]).view(T, nkv, d)
        q = F.rms_norm(q, (d,), weight=ck[p + "q_norm"], eps=m.eps)
        k = F.rms_norm(k, (d,), weight=ck[p + "k_norm"], eps=m.eps)
        q = _rotate(q, positions, m.rope_theta)
        k = _rotate(k, positions, m.rope_theta)
        o = torch.empty(T, nh, d, dtype=torch.float64)
        for s in range(len(cu_seqlens) - 1):
            a, b = int(cu_seqlens[s]), int(cu_seqlens[s + 1])
            o[a:b] = F.scaled_dot_product_attention(q[a:b].transpose(0, 1), k[a:b].transpose(0, 1),
                                                    v[a:b].transpose(0, 1), is_causal=True,
                                                    enable_gqa=True).transpose(0, 1)
        x = F.linear(o.reshape(T, nh * d), ck[p + "o_proj"])
        # post_attention_layernorm, then the MLP
        residual = x + residual
        h = F.rms_norm(residual, (H,), weight=ck[p + "post_attention_layernorm"], eps=m.eps)
        a = F.silu(F.linear(h, ck[p + "gate_proj"])) * F.linear(h, ck[p + "up_proj"])
        x = F.linear(a, ck[p + "down_proj"])
    hidden = F.rms_norm(x + residual, (H,), weight=ck["norm"], eps=m.eps)
    last = torch.as_tensor(cu_seqlens[1:], dtype=torch.int64) - 1
    return hidden, F.linear(hidden[last], ck["embed_tokens"])


def _oracle_prefill(m, w, b):
    cache = O.KVCache(m.n_layers, b.num_slots, m.n_kv_heads, m.head_dim, m.tp)
    ctx = O.AttnContext(True, b.slot_mapping.numpy(), cu_seqlens=b.cu_seqlens.numpy())
    h = O.model_forward(m, w, b.ids.numpy(), b.positions.numpy(), ctx, cache)
    return h, O.compute_logits(m, w.embed, h, m.tp, b.cu_seqlens.numpy()), cache


@pytest.mark.parametrize("tp", [1, 2])
def test_model_prefill_equals_independent_composition(tp):
    m = SHAPE.replace(tp=tp)
    ck = _ck(m)
    w = O.load_weights(m.replace(dtype="f32"))
    b = si.prefill_batch(m, [7, 1, 12])
    h_ref, lg_ref = _reference_forward(m, ck, b.ids, b.positions, b.cu_seqlens.tolist())
    h, lg, _ = _oracle_prefill(m, w, b)
    # the only difference allowed: the last bits of the fp32 RoPE table's cos/sin
    assert np.allclose(h, h_ref.numpy(), rtol=0, atol=1e-6), np.abs(h - h_ref.numpy()).max()
    assert np.allclose(lg, lg_ref.numpy(), rtol=0, atol=1e-6), np.abs(lg - lg_ref.numpy()).max()


def test_decoder_layer_equals_independent_composition():
    """One layer from given hidden states, both outputs (h, residual) of [SK] §1."""
    m = SHAPE.replace(n_layers=1, tp=2)
    ck = _ck(m)
    w = O.load_weights(m.replace(dtype="f32"))
    b = si.prefill_batch(m, [9, 4])
    T = b.ids.shape[0]
    rng = np.random.default_rng(7)
    x = rng.standard_normal((T, m.hidden))
    r = rng.standard_normal((T, m.hidden))
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    ctx = O.AttnContext(True, b.slot_mapping.numpy(), cu_seqlens=b.cu_seqlens.numpy())
    cache = O.KVCache(1, b.num_slots, m.n_kv_heads, m.head_dim, m.tp)
    h, res = O.decoder_layer(m, w.layers[0], 0, b.positions.numpy(), x, r, ctx, cache, *cos_sin)

    # independent: one layer with an incoming residual
    nh, nkv, d, H = m.n_heads, m.n_kv_heads, m.head_dim, m.hidden
    xt, rt = torch.from_numpy(x), torch.from_numpy(r)
    s = xt + rt
    hh = F.rms_norm(s, (H,), weight=ck["layer0.input_layernorm"], eps=m.eps)
    q = F.rms_norm(F.linear(hh, ck["layer0.q_proj"]).view(T, nh, d), (d,), weight=ck["layer0.q_norm"], eps=m.eps)
    k = F.rms_norm(F.linear(hh, ck["layer0.k_proj"]).view(T, nkv, d), (d,), weight=ck["layer0.k_norm"], eps=m.eps)
    v = F.linear(hh, ck["layer0.v_proj"]).view(T, nkv, d)
    q, k = _rotate(q, b.positions, m.rope_theta), _rotate(k, b.positions, m.rope_theta)
    cu = b.cu_seqlens.tolist()
    o = torch.cat([F.scaled_dot_product_attention(q[a:e].transpose(0, 1), k[a:e].transpose(0, 1),
                                                  v[a:e].transpose(0, 1), is_causal=True,
                                                  enable_gqa=True).transpose(0, 1)
                   for a, e in zip(cu[:-1], cu[1:])])
    s2 = F.linear(o.reshape(T, nh * d), ck["layer0.o_proj"]) + s
    h2 = F.rms_norm(s2, (H,), weight=ck["layer0.post_attention_layernorm"], eps=m.eps)
    out = F.linear(F.silu(F.linear(h2, ck["layer0.gate_proj"])) * F.linear(h2, ck["layer0.up_proj"]),
                   ck["layer0.down_proj"])
    assert np.allclose(res, s2.numpy(), rtol=0, atol=1e-6)
    assert np.allclose(h, out.numpy(), rtol=0, atol=1e-6)
    # the cache holds the normed, rotated k and the raw v ([SK] §7.1, §8 ①)
    k_cat = np.concatenate([cache.k[rk][0] for rk in range(m.tp)], axis=1)
    v_cat = np.concatenate([cache.v[rk][0] for rk in range(m.tp)], axis=1)
    slots = b.slot_mapping.numpy()
    assert np.allclose(k_cat[slots], k.numpy(), rtol=0, atol=1e-6)
    assert np.allclose(v_cat[slots], v.numpy(), rtol=0, atol=1e-12)


def test_decode_step_equals_independent_composition():
    """Prefill of L-1 tokens, then the decode of token L-1 from the cache, against
    the independent prefill of all L tokens (its last row and logits)."""
    m = SHAPE.replace(tp=2)
    ck = _ck(m)
    w = O.load_weights(m.replace(dtype="f32"))
    L = 11
    full = si.prefill_batch(m, [L])
    ids = full.ids
    h_ref, lg_ref = _reference_forward(m, ck, ids, full.positions, [0, L])
    cache = O.KVCache(m.n_layers, L, m.n_kv_heads, m.head_dim, m.tp)
    ctx = O.AttnContext(True, np.arange(L - 1), cu_seqlens=np.array([0, L - 1]))
    O.model_forward(m, w, ids.numpy()[:L - 1], np.arange(L - 1), ctx, cache)
    dctx = O.AttnContext(False, np.array([L - 1]), seq_base=np.array([0]), context_lens=np.array([L]))
    hd = O.model_forward(m, w, ids.numpy()[L - 1:], np.array([L - 1]), dctx, cache)
    lg = O.compute_logits(m, w.embed, hd, m.tp)
    assert np.allclose(hd[0], h_ref.numpy()[L - 1], rtol=0, atol=1e-6)
    assert np.allclose(lg[0], lg_ref.numpy()[0], rtol=0, atol=1e-6)


def test_gammas_are_distinct_so_swaps_are_visible():
    """The fixture's premise: every norm's gamma differs from the others and from 1."""
    ck = _ck(SHAPE)
    g = [ck["norm"], ck["layer0.input_layernorm"], ck["layer0.post_attention_layernorm"],
         ck["layer1.input_layernorm"]]
    for i in range(len(g)):
        assert (g[i] - 1.0).abs().max() > 0.1
        for j in range(i):
            assert (g[i] - g[j]).abs().max() > 0.1
    assert (ck["layer0.q_norm"] - ck["layer0.k_norm"]).abs().max() > 0.1
    assert (ck["layer0.q_norm"] - 1.0).abs().max() > 0.1


def test_layerwise_helpers_equal_model_forward():
    """The layer-at-a-time oracle drivers used by the full-size parity tests
    (one layer's cache alive at a time) give exactly O.model_forward's results."""
    from tests.model_parity import oracle_decode_layerwise, oracle_prefill_layerwise
    m = SHAPE.replace(tp=2, dtype="bf16")
    w = O.load_weights(m)
    lens = [9, 4, 13]
    b = si.prefill_batch(m, lens)
    cache = O.KVCache(m.n_layers, b.num_slots, m.n_kv_heads, m.head_dim, m.tp)
    ctx = O.AttnContext(True, b.slot_mapping.numpy(), cu_seqlens=b.cu_seqlens.numpy())
    h = O.model_forward(m, w, b.ids.numpy(), b.positions.numpy(), ctx, cache)
    rows = np.array([0, 8, 12, 25])
    hl, lg = oracle_prefill_layerwise(m, w, b.ids.numpy(), lens, rows)
    assert np.array_equal(hl, h[rows])
    assert np.array_equal(lg, O.compute_logits(m, w.embed, h[rows], m.tp))
    # one decode step over the prefill's cache, its rows handed over layer by layer
    base = b.seq_base.numpy().astype(np.int64)
    ext = si.prefill_batch(m, lens, extra_capacity=1)
    cache2 = O.KVCache(m.n_layers, ext.num_slots, m.n_kv_heads, m.head_dim, m.tp)
    ctx2 = O.AttnContext(True, ext.slot_mapping.numpy(), cu_seqlens=ext.cu_seqlens.numpy())
    O.model_forward(m, w, ext.ids.numpy(), ext.positions.numpy(), ctx2, cache2)
    snapshot = [[np.concatenate([cache2.k[r][l] for r in range(m.tp)], axis=1) for l in range(m.n_layers)],
                [np.concatenate([cache2.v[r][l] for r in range(m.tp)], axis=1) for l in range(m.n_layers)]]
    base = ext.seq_base.numpy().astype(np.int64)
    pos = np.array(lens, dtype=np.int64)
    slots = base + pos
    ids = np.array([5, 77, 31])
    dctx = O.AttnContext(False, slots, seq_base=base, context_lens=pos + 1)
    hd = O.model_forward(m, w, ids, pos, dctx, cache2)
    hl, lg = oracle_decode_layerwise(m, w, ids, pos, pos + 1, slots, base, ext.num_slots,
                                     lambda l: (snapshot[0][l].copy(), snapshot[1][l].copy()))
    assert np.array_equal(hl, hd)
    assert np.array_equal(lg, O.compute_logits(m, w.embed, hd, m.tp))
