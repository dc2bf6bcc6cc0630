"""Plain, slow CPU oracle of the nano-vllm-style Qwen3 forward pass.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path.  It
shares no code with the CUDA library; the only common module is the seeded
input generator (``seeded_inputs``), which holds none of the model's
arithmetic.

Arithmetic is float64 (numpy).  Tensors that the pages' model keeps in the
model dtype are rounded to that dtype (bf16 or fp32) at the same module
boundaries the pages' code has: the output of each Linear, of each RMSNorm,
of RoPE, of the residual add, of SiluAndMul, of attention and of the
lm_head.  bf16 rounding is round-to-nearest-even, implemented below from the
IEEE-754 definition.

Sources (web pages on nano-vllm's Qwen3 model code; cited by page and section):

  [VH]  devpress page "vocab 切 / head 切": §3 VocabParallelEmbedding,
        §4 ParallelLMHead, §5 attention and KV cache head split, §6 check
  [TP]  devpress page on tensor-parallel maths: §3 column vs row split
        (Y = [X W0 | X W1], Y = X0 W0 + X1 W1), §4 the two column->row
        pairs and the head split, §5 embedding and LM head, §6 why RMSNorm
        is replicated
  [VPE] "从零实现 vLLM (1.1): 并行词嵌入 VocabParallelEmbedding": the worked
        12-word example and the nano-vllm source of the class
  [SK]  "3.3 模型骨架与核心算子" (AIInfraGuide): §1 Qwen3DecoderLayer,
        §2 RMSNorm, §3 RoPE, §4 SiluAndMul, §5 parallel Linear family,
        §6 vocab-parallel Embedding and LMHead, §7 attention (KV store,
        prefill and decode paths), §8 Qwen3 assembly

Readings where the pages are silent (each listed with its reason in the
design notes of the repository):
  * the model ends with a final add+RMSNorm (the layer returns h and the
    residual unsummed, [SK] §1);
  * RMSNorm eps = 1e-6 everywhere, including q_norm/k_norm;
  * residual add is rounded to the model dtype, and that rounded sum is both
    the new residual and the norm input ([SK] §2 add_rms_forward);
  * RoPE: rotary_dim = head_dim, halves pairing (i, i + d/2); inv_freq is the
    exact 1/theta^(2i/d) rounded to fp32, angle = fp32(t * inv_freq) as the
    page's fp32 outer product, cos/sin exact then rounded to fp32;
  * GQA: kv head = q head // (n_heads / n_kv_heads);
  * row-parallel partial sums are added before one rounding (the emulated
    all_reduce of [TP] §3 is exact);
  * SiluAndMul rounds once;
  * argmax ties go to the lowest index.

Every function here is pinned by ``tests/test_oracle_pins.py`` (worked
values the pages print, closed forms, library routines for special cases,
brute force and invariants).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

__all__ = [
    "round_to", "bf16_round", "f32_round",
    "vocab_range", "vocab_embedding_rank", "vocab_parallel_embedding", "embedding_unsharded",
    "rms_norm", "add_rms_norm",
    "linear", "column_parallel_linear", "row_parallel_linear",
    "qkv_shard_weight", "gate_up_shard_weight", "heads_per_rank", "kv_cache_shape",
    "rope_cos_sin", "apply_rope",
    "silu_and_mul", "attention_prefill", "attention_decode",
    "KVCache", "LayerWeights", "ModelWeights", "load_weights", "load_layer", "AttnContext",
    "attention_block", "mlp_block",
    "decoder_layer", "model_forward", "compute_logits", "greedy",
    "parallel_lm_head_rank", "lm_head_unsharded", "sample",
]


# ----------------------------------------------------------------------------
# rounding to the model dtype
# ----------------------------------------------------------------------------

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even (IEEE-754 RNE).

    bf16 keeps 8 significant bits; for |x| in [2^(e-1), 2^e) one unit in the
    last place is 2^(e-8).  Below the smallest normal (2^-126) the spacing is
    fixed at 2^-133.  Results at or beyond the overflow threshold become +-inf.

    For |x| >= 2^-126 the float64 encoding already holds x exactly, so the
    rounding is done on its bits: keep the sign, the exponent and the top 7
    of the 52 stored fraction bits, and round the 45 dropped bits to nearest,
    ties to the even kept bit (adding 2^44 - 1 plus the kept LSB, then
    clearing the dropped bits; a carry out of the fraction correctly bumps
    the exponent).  Below 2^-126 the fixed spacing is applied by scaling.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    bits = out.reshape(-1).view(np.uint64)
    expo = (bits >> np.uint64(52)) & np.uint64(0x7FF)
    normal = (expo >= np.uint64(1023 - 126)) & (expo < np.uint64(0x7FF))
    kept = bits[normal]
    lsb = (kept >> np.uint64(45)) & np.uint64(1)
    bits[normal] = (kept + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    flat = x.reshape(-1)
    small = (expo < np.uint64(1023 - 126)) & (flat != 0)
    if small.any():
        spacing = 2.0 ** -133
        bits[small] = (np.rint(flat[small] / spacing) * spacing).view(np.uint64)
    big = (np.abs(out) > _BF16_MAX) & np.isfinite(x)
    out[big] = np.copysign(np.inf, out[big])
    return out


def f32_round(x) -> np.ndarray:
    """Round float64 values to the nearest fp32 value (numpy's IEEE cast)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to(x, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_round(x)
    if dtype in ("f32", "fp32"):
        return f32_round(x)
    if dtype in ("f64", None):
        return np.asarray(x, dtype=np.float64)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# vocab-parallel embedding  ([VH] §3, [VPE], [SK] §6)
# ----------------------------------------------------------------------------

def vocab_range(vocab: int, tp: int, rank: int):
    """[start, end) of the vocab ids rank `rank` owns: per = V // tp ([VH] §3 __init__)."""
    per = vocab // tp
    start = per * rank
    return start, start + per


def vocab_embedding_rank(ids, table, tp: int, rank: int, trace: Optional[dict] = None) -> np.ndarray:
    """One rank's partial output: the five steps of [VH] §3 without the final all_reduce.

    1. mask = start <= x < end;  2. x = mask * (x - start);  3. y = W_r[x];
    4. y = mask[:, None] * y.  W_r is the rank's row block, cut from the full
    table with narrow(0, rank * per, per) as in the weight_loader.
    """
    ids = np.asarray(ids, dtype=np.int64)
    table = np.asarray(table, dtype=np.float64)
    start, end = vocab_range(table.shape[0], tp, rank)
    w_r = table[start:end]
    mask = (ids >= start) & (ids < end)
    local = mask * (ids - start)
    y = w_r[local]
    y_zeroed = mask[..., None] * y
    if trace is not None:
        trace.update(mask=mask, local=local, lookup=y, zeroed=y_zeroed)
    return y_zeroed


def vocab_parallel_embedding(ids, table, tp: int) -> np.ndarray:
    """Sum of the ranks' partial outputs: the all_reduce of [VH] §3 step 5 emulated in one process.

    The ranks' partials are added in rank order, as [VPE]'s stack(...).sum(0).
    """
    out = None
    for r in range(tp):
        p = vocab_embedding_rank(ids, table, tp, r)
        out = p if out is None else out + p
    return out


def embedding_unsharded(ids, table) -> np.ndarray:
    """F.embedding on the full table (the single-card side of [VH] §6)."""
    return np.asarray(table, dtype=np.float64)[np.asarray(ids, dtype=np.int64)]


# ----------------------------------------------------------------------------
# RMSNorm  ([SK] §2, [TP] §6)
# ----------------------------------------------------------------------------

def rms_norm(x, gamma, eps: float, dtype: str) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gamma over the last axis, rounded once to `dtype`."""
    x = np.asarray(x, dtype=np.float64)
    var = np.mean(x * x, axis=-1, keepdims=True)
    y = x * (1.0 / np.sqrt(var + eps)) * np.asarray(gamma, dtype=np.float64)
    return round_to(y, dtype)


def add_rms_norm(x, residual, gamma, eps: float, dtype: str):
    """add_rms_forward of [SK] §2: x = x + residual; residual = x; return (norm(x), residual)."""
    s = round_to(np.asarray(x, dtype=np.float64) + np.asarray(residual, dtype=np.float64), dtype)
    return rms_norm(s, gamma, eps, dtype), s


# ----------------------------------------------------------------------------
# Linear family  ([TP] §3-§4, [SK] §5)
# ----------------------------------------------------------------------------

def linear(x, w, dtype: str) -> np.ndarray:
    """F.linear(x, w) = x @ w^T, exact in float64, rounded once to the model dtype."""
    return round_to(np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T, dtype)


def column_parallel_linear(x, w_full, tp: int, rank: int, dtype: str) -> np.ndarray:
    """Rank `rank`'s output columns: W cut along the output dim (tp_dim=0), [TP] §3 Y=[XW0|XW1]."""
    n_l = w_full.shape[0] // tp
    return linear(x, w_full[rank * n_l:(rank + 1) * n_l], dtype)


def row_parallel_linear(x_shards: Sequence[np.ndarray], w_full, tp: int, dtype: str) -> np.ndarray:
    """Y = sum_r X_r W_r^T with W cut along the input dim (tp_dim=1), [TP] §3 Y = X0W0 + X1W1.

    Each rank's partial sum stays unrounded; the emulated all_reduce adds them
    exactly and the result is rounded once.
    """
    k_l = w_full.shape[1] // tp
    acc = None
    for r in range(tp):
        part = np.asarray(x_shards[r], dtype=np.float64) @ np.asarray(
            w_full[:, r * k_l:(r + 1) * k_l], dtype=np.float64).T
        acc = part if acc is None else acc + part
    return round_to(acc, dtype)


def heads_per_rank(n_heads: int, n_kv_heads: int, tp: int):
    """num_heads // tp and num_kv_heads // tp, asserting divisibility ([VH] §5)."""
    assert n_heads % tp == 0 and n_kv_heads % tp == 0
    return n_heads // tp, n_kv_heads // tp


def kv_cache_shape(layers: int, blocks: int, block_size: int, n_kv_heads: int, head_dim: int, tp: int):
    """allocate_kv_cache's per-rank shape (2, layers, blocks, block_size, kv_heads/tp, head_dim) ([VH] §5)."""
    return (2, layers, blocks, block_size, n_kv_heads // tp, head_dim)


def qkv_shard_weight(wq, wk, wv, n_heads, n_kv_heads, head_dim, tp, rank) -> np.ndarray:
    """QKVParallelLinear's rank weight: its q rows, then k rows, then v rows ([SK] §5, [VH] §5)."""
    nh_l, nkv_l = heads_per_rank(n_heads, n_kv_heads, tp)
    q = wq[rank * nh_l * head_dim:(rank + 1) * nh_l * head_dim]
    k = wk[rank * nkv_l * head_dim:(rank + 1) * nkv_l * head_dim]
    v = wv[rank * nkv_l * head_dim:(rank + 1) * nkv_l * head_dim]
    return np.concatenate([q, k, v], axis=0)


def gate_up_shard_weight(wg, wu, tp, rank) -> np.ndarray:
    """MergedColumnParallelLinear's rank weight: its half of gate, then its half of up ([TP] §4.2)."""
    i_l = wg.shape[0] // tp
    return np.concatenate([wg[rank * i_l:(rank + 1) * i_l], wu[rank * i_l:(rank + 1) * i_l]], axis=0)


# ----------------------------------------------------------------------------
# RoPE  ([SK] §3)
# ----------------------------------------------------------------------------

def rope_cos_sin(max_position: int, rotary_dim: int, theta: float):
    """cos/sin tables [max_position, rotary_dim/2] in fp32 (returned as float64 arrays).

    inv_freq_i = 1 / theta^(2i/d) (exact, rounded to fp32); freqs = t * inv_freq
    as an fp32 outer product; cos and sin of those fp32 angles rounded to fp32.
    """
    i2 = np.arange(0, rotary_dim, 2, dtype=np.float64)
    inv_freq = f32_round(1.0 / np.power(float(theta), i2 / rotary_dim))
    t = np.arange(max_position, dtype=np.float64)
    freqs = f32_round(t[:, None] * inv_freq[None, :])
    return f32_round(np.cos(freqs)), f32_round(np.sin(freqs))


def apply_rope(x, positions, cos_t, sin_t, dtype: str) -> np.ndarray:
    """Rotate each (x1, x2) half pair: y1 = x1 cos - x2 sin, y2 = x2 cos + x1 sin ([SK] §3).

    x: [T, heads, d]; positions: [T].  Applied to q and k only.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    cos = cos_t[np.asarray(positions, dtype=np.int64)][:, None, :]
    sin = sin_t[np.asarray(positions, dtype=np.int64)][:, None, :]
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    y1 = x1 * cos - x2 * sin
    y2 = x2 * cos + x1 * sin
    return round_to(np.concatenate([y1, y2], axis=-1), dtype)


# ----------------------------------------------------------------------------
# SiluAndMul  ([SK] §4, [TP] §4.2)
# ----------------------------------------------------------------------------

def silu_and_mul(x, dtype: str) -> np.ndarray:
    """gate, up = x.chunk(2, -1); silu(gate) * up with silu(g) = g / (1 + e^-g); one rounding."""
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    gate, up = x[..., :h], x[..., h:]
    return round_to(gate / (1.0 + np.exp(-gate)) * up, dtype)


# ----------------------------------------------------------------------------
# attention  ([SK] §7, [VH] §5)
# ----------------------------------------------------------------------------

def _softmax_rows(s):
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention_prefill(q, k, v, cu_seqlens, scale: float, dtype: str) -> np.ndarray:
    """flash_attn_varlen_func(q, k, v, cu_seqlens, causal=True) as the plain definition.

    q: [T, nh, d]; k, v: [T, nkv, d] (the batch's fresh keys/values, sequences
    packed by cu_seqlens).  Query i of a sequence sees keys 0..i of the same
    sequence; q head h reads kv head h // (nh / nkv).  Full softmax in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, nh, d = q.shape
    nkv = k.shape[1]
    group = nh // nkv
    out = np.zeros((T, nh, d))
    cu = [int(c) for c in cu_seqlens]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        L = b - a
        if L == 0:
            continue
        causal = np.tril(np.ones((L, L), dtype=bool))
        for h in range(nh):
            g = h // group
            sc = (q[a:b, h] @ k[a:b, g].T) * scale
            sc = np.where(causal, sc, -np.inf)
            out[a:b, h] = _softmax_rows(sc) @ v[a:b, g]
    return round_to(out, dtype)


def attention_decode(q, k_seq: Sequence[np.ndarray], v_seq: Sequence[np.ndarray], scale: float,
                     dtype: str) -> np.ndarray:
    """flash_attn_with_kvcache for one new token per sequence.

    q: [B, nh, d]; k_seq[b], v_seq[b]: [context_len_b, nkv, d], the cached keys
    of sequence b including the token stored by this step.
    """
    q = np.asarray(q, dtype=np.float64)
    B, nh, d = q.shape
    out = np.zeros((B, nh, d))
    for b in range(B):
        kb = np.asarray(k_seq[b], dtype=np.float64)
        vb = np.asarray(v_seq[b], dtype=np.float64)
        group = nh // kb.shape[1]
        for h in range(nh):
            g = h // group
            sc = (kb[:, g] @ q[b, h]) * scale
            p = _softmax_rows(sc[None, :])[0]
            out[b, h] = p @ vb[:, g]
    return round_to(out, dtype)


# ----------------------------------------------------------------------------
# KV cache and weights
# ----------------------------------------------------------------------------

class KVCache:
    """Per-rank, per-layer caches k/v[slot, kv_heads/tp, d] ([VH] §5, [SK] §7.1)."""

    def __init__(self, n_layers: int, num_slots: int, n_kv_heads: int, head_dim: int, tp: int):
        nkv_l = n_kv_heads // tp
        self.tp = tp
        self.k = [[np.zeros((num_slots, nkv_l, head_dim), np.float64) for _ in range(n_layers)]
                  for _ in range(tp)]
        self.v = [[np.zeros((num_slots, nkv_l, head_dim), np.float64) for _ in range(n_layers)]
                  for _ in range(tp)]

    def store(self, rank: int, layer: int, k, v, slot_mapping):
        """store_kvcache: row slot of the cache <- the token's k and v; slot -1 is skipped."""
        for i, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
            if slot == -1:
                continue
            self.k[rank][layer][slot] = k[i]
            self.v[rank][layer][slot] = v[i]


@dataclass
class LayerWeights:
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    wg: np.ndarray
    wu: np.ndarray
    wd: np.ndarray
    input_ln: np.ndarray
    post_ln: np.ndarray
    q_norm: np.ndarray
    k_norm: np.ndarray


@dataclass
class ModelWeights:
    embed: np.ndarray                 # tied with the lm_head ([SK] §8)
    layers: List[LayerWeights]
    final_norm: np.ndarray


def _np(t):
    return t.detach().to("cpu").double().numpy()


def load_layer(m, layer: int, seed: int = 0) -> LayerWeights:
    """The layer's checkpoint tensors from the seeded generator, as float64 arrays."""
    from seeded_inputs import checkpoint_tensor as ct
    p = f"layer{layer}."
    return LayerWeights(*[_np(ct(m, p + n, seed)) for n in (
        "q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj",
        "input_layernorm", "post_attention_layernorm", "q_norm", "k_norm")])


def load_weights(m, seed: int = 0, layers: Optional[int] = None, lazy: bool = False,
                 with_embed: bool = True) -> ModelWeights:
    from seeded_inputs import checkpoint_tensor as ct
    n = m.n_layers if layers is None else layers
    embed = _np(ct(m, "embed_tokens", seed)) if with_embed else None
    lw = [None] * n if lazy else [load_layer(m, l, seed) for l in range(n)]
    return ModelWeights(embed, lw, _np(ct(m, "norm", seed)))


# ----------------------------------------------------------------------------
# decoder layer and model  ([SK] §1, §8; [TP] §4)
# ----------------------------------------------------------------------------

@dataclass
class AttnContext:
    """The fields of get_context() the layers read ([SK] §6-§7)."""
    is_prefill: bool
    slot_mapping: np.ndarray
    cu_seqlens: Optional[np.ndarray] = None       # prefill
    seq_base: Optional[np.ndarray] = None         # decode: first cache slot of each sequence
    context_lens: Optional[np.ndarray] = None     # decode: keys visible, incl. the new token


def attention_block(m, lw: LayerWeights, layer: int, positions, h, ctx: AttnContext, cache: KVCache,
                    cos_t, sin_t, trace: Optional[dict] = None) -> np.ndarray:
    """Qwen3Attention.forward per rank ([SK] §8 ①), heads split across ranks ([VH] §5),
    then o_proj as a row-parallel Linear with the emulated all_reduce ([TP] §4.1)."""
    tp = cache.tp
    dt = m.dtype
    nh_l, nkv_l = heads_per_rank(m.n_heads, m.n_kv_heads, tp)
    d = m.head_dim
    o_shards = []
    for r in range(tp):
        w_qkv = qkv_shard_weight(lw.wq, lw.wk, lw.wv, m.n_heads, m.n_kv_heads, d, tp, r)
        qkv = linear(h, w_qkv, dt)
        T = qkv.shape[0]
        q = qkv[:, : nh_l * d].reshape(T, nh_l, d)
        k = qkv[:, nh_l * d:(nh_l + nkv_l) * d].reshape(T, nkv_l, d)
        v = qkv[:, (nh_l + nkv_l) * d:].reshape(T, nkv_l, d)
        q = rms_norm(q, lw.q_norm, m.eps, dt)
        k = rms_norm(k, lw.k_norm, m.eps, dt)
        q = apply_rope(q, positions, cos_t, sin_t, dt)
        k = apply_rope(k, positions, cos_t, sin_t, dt)
        cache.store(r, layer, k, v, ctx.slot_mapping)
        scale = d ** -0.5
        if ctx.is_prefill:
            o = attention_prefill(q, k, v, ctx.cu_seqlens, scale, dt)
        else:
            ks, vs = [], []
            for b in range(T):
                s0 = int(ctx.seq_base[b])
                L = int(ctx.context_lens[b])
                ks.append(cache.k[r][layer][s0:s0 + L])
                vs.append(cache.v[r][layer][s0:s0 + L])
            o = attention_decode(q, ks, vs, scale, dt)
        if trace is not None:
            trace.setdefault("qkv", []).append(qkv)
            trace.setdefault("q", []).append(q)
            trace.setdefault("k", []).append(k)
            trace.setdefault("v", []).append(v)
            trace.setdefault("o", []).append(o)
        o_shards.append(o.reshape(T, nh_l * d))
    return row_parallel_linear(o_shards, lw.wo, tp, dt)


def mlp_block(m, lw: LayerWeights, h, tp: int, trace: Optional[dict] = None) -> np.ndarray:
    """gate_up (column) -> SiluAndMul -> down (row + all_reduce), [TP] §4.2, [SK] §4-§5."""
    a_shards = []
    for r in range(tp):
        gu = linear(h, gate_up_shard_weight(lw.wg, lw.wu, tp, r), m.dtype)
        a = silu_and_mul(gu, m.dtype)
        if trace is not None:
            trace.setdefault("gate_up", []).append(gu)
            trace.setdefault("act", []).append(a)
        a_shards.append(a)
    return row_parallel_linear(a_shards, lw.wd, tp, m.dtype)


def decoder_layer(m, lw: LayerWeights, layer: int, positions, hidden, residual, ctx: AttnContext,
                  cache: KVCache, cos_t, sin_t, trace: Optional[dict] = None):
    """Qwen3DecoderLayer.forward ([SK] §1): pre-norm, with the residual add fused into RMSNorm."""
    if residual is None:
        h, residual = rms_norm(hidden, lw.input_ln, m.eps, m.dtype), np.asarray(hidden, np.float64)
    else:
        h, residual = add_rms_norm(hidden, residual, lw.input_ln, m.eps, m.dtype)
    if trace is not None:
        trace["attn_in"] = h
    h = attention_block(m, lw, layer, positions, h, ctx, cache, cos_t, sin_t, trace)
    if trace is not None:
        trace["attn_out"] = h
    h, residual = add_rms_norm(h, residual, lw.post_ln, m.eps, m.dtype)
    if trace is not None:
        trace["mlp_in"] = h
    h = mlp_block(m, lw, h, cache.tp, trace)
    return h, residual


def model_forward(m, w: ModelWeights, ids, positions, ctx: AttnContext, cache: KVCache,
                  cos_sin=None, layer_loader=None, hidden_in=None):
    """Qwen3ForCausalLM.forward: embedding -> layers -> final add+RMSNorm; returns hidden.

    `hidden_in`, if given, replaces the embedding output (single-layer workloads
    start from given hidden states).  `layer_loader(l)` supplies layer weights
    lazily when `w.layers[l]` is None.
    """
    tp = cache.tp
    cos_t, sin_t = cos_sin if cos_sin is not None else rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    if hidden_in is None:
        h = vocab_parallel_embedding(ids, w.embed, tp)
    else:
        h = np.asarray(hidden_in, dtype=np.float64)
    residual = None
    for l in range(len(w.layers)):
        lw = w.layers[l] if w.layers[l] is not None else layer_loader(l)
        h, residual = decoder_layer(m, lw, l, positions, h, residual, ctx, cache, cos_t, sin_t)
    h, _ = add_rms_norm(h, residual, w.final_norm, m.eps, m.dtype)
    return h


def parallel_lm_head_rank(x, table, tp: int, rank: int, dtype: str) -> np.ndarray:
    """One rank's logit slice F.linear(x, W_r) over its vocab rows ([VH] §4)."""
    start, end = vocab_range(table.shape[0], tp, rank)
    return linear(x, table[start:end], dtype)


def lm_head_unsharded(x, table, dtype: str) -> np.ndarray:
    return linear(x, table, dtype)


def compute_logits(m, table, hidden, tp: int, cu_seqlens=None) -> np.ndarray:
    """ParallelLMHead.forward ([SK] §6): in prefill keep each sequence's last token
    (cu_seqlens[1:] - 1), then each rank's logit slice, concatenated (the gather)."""
    x = np.asarray(hidden, dtype=np.float64)
    if cu_seqlens is not None:
        last = np.asarray(cu_seqlens, dtype=np.int64)[1:] - 1
        x = x[last]
    return np.concatenate([parallel_lm_head_rank(x, table, tp, r, m.dtype) for r in range(tp)], axis=-1)


def greedy(logits) -> np.ndarray:
    """Greedy sampling: argmax over the vocab, lowest index on ties (np.argmax's first occurrence)."""
    return np.argmax(np.asarray(logits), axis=-1).astype(np.int64)


# ----------------------------------------------------------------------------
# sampling  ([SK] §3 note: the Sampler is one of the small compiled operators)
# ----------------------------------------------------------------------------

def sample(logits, temperature, top_p, uniforms) -> np.ndarray:
    """Temperature / top-p sampling of one token per row (a reading: the pages
    name the Sampler among nano-vllm's compiled small operators but give no
    semantics).

    Row b with temperature T and nucleus mass P:
      * T == 0: greedy, the argmax of the logits (lowest index on ties).
      * otherwise the token is drawn from softmax(logits / T) restricted to the
        nucleus: with c_1 > c_2 > ... the row's distinct logit values and
        m_k the softmax mass of the tokens whose logit is c_k, K is the first k
        with m_1 + ... + m_k >= P (mass relative to the whole row); the nucleus
        is every token with logit >= c_K (tokens tied at the boundary value are
        all kept).  P = 1 keeps the whole row.
      * the draw uses the Gumbel-max identity: with u_v uniform in (0, 1) and
        G_v = -log(-log u_v), argmax over the nucleus of logits_v / T + G_v is
        distributed as the restricted softmax (E. J. Gumbel's extreme-value
        distribution; argmax ties to the lowest index).
    logits [B, V]; temperature, top_p [B]; uniforms [B, V] in (0, 1), the random
    numbers of the draw (an input, so both sides use the same ones).
    """
    logits = np.asarray(logits, dtype=np.float64)
    uniforms = np.asarray(uniforms, dtype=np.float64)
    out = np.zeros(logits.shape[0], dtype=np.int64)
    for b in range(logits.shape[0]):
        lg = logits[b]
        T = float(temperature[b])
        if T == 0.0:
            out[b] = int(np.argmax(lg))
            continue
        z = lg / T
        e = np.exp(z - np.max(z))
        values, which = np.unique(lg, return_inverse=True)          # ascending distinct values
        mass = np.bincount(which, weights=e, minlength=len(values))
        cum = np.cumsum(mass[::-1])                                    # from the largest value down
        K = int(np.argmax(cum >= float(top_p[b]) * cum[-1]))
        nucleus = lg >= values[::-1][K]
        g = -np.log(-np.log(uniforms[b]))
        out[b] = int(np.argmax(np.where(nucleus, z + g, -np.inf)))
    return out
