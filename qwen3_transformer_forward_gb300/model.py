"""Qwen3 forward pass on one GB300: sequences the libqw entry points.

This module does no arithmetic of the model.  It owns device buffers (via
PyTorch), builds the tensor-parallel weight layout at load time, and calls
one C-ABI entry point per step, in the order of Qwen3DecoderLayer.forward
and Qwen3ForCausalLM ([SK] §1, §8; [VH] §3-§5):

  embed (vocab-parallel) -> per layer:
     add+RMSNorm -> QKV GEMM (column) -> QK-norm + RoPE + KV store ->
     attention (prefill: varlen causal; decode: over the cache) ->
     o_proj GEMM (row, shard sum) -> add+RMSNorm ->
     gate_up GEMM (column) with fused SiluAndMul -> down GEMM (row, shard sum)
  -> final add+RMSNorm -> lm_head (last token per sequence in prefill) -> argmax

Sources: [VH] devpress "vocab 切 / head 切"; [TP] devpress tensor-parallel
maths; [SK] AIInfraGuide "3.3 模型骨架与核心算子".
"""
from __future__ import annotations

import contextlib
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

from . import _lib as L


# ----------------------------------------------------------------------------
# load-time layout (the weight_loader of the parallel Linear family)
# ----------------------------------------------------------------------------

@dataclass
class LayerParams:
    qkv: torch.Tensor        # [tp * (nh/tp + 2 nkv/tp) * hd, H]   shard r = [q_r; k_r; v_r]
    o: torch.Tensor          # [tp, H, nh/tp * hd]                 shard r = input columns of its heads
    gate_up: torch.Tensor    # [tp * 2 * I/tp, H]                  shard r = [gate_r; up_r]
    down: torch.Tensor       # [tp, H, I/tp]
    input_ln: torch.Tensor
    post_ln: torch.Tensor
    q_norm: torch.Tensor
    k_norm: torch.Tensor


@dataclass
class ModelParams:
    embed: torch.Tensor      # [V, H]; tied with the lm_head ([SK] §8); shard r = row block r
    layers: List[LayerParams]
    final_norm: torch.Tensor


def shard_layer(shape, ck: Dict[str, torch.Tensor], layer: int, device) -> LayerParams:
    """Places one layer's checkpoint tensors into the per-shard stacked layout.

    QKVParallelLinear / MergedColumnParallelLinear narrow each checkpoint
    tensor along the output dim per shard; RowParallelLinear narrows along the
    input dim ([SK] §5, [TP] §3-§4).  Runs once at load time.
    """
    tp, hd = shape.tp, shape.head_dim
    nh_l, nkv_l, i_l = shape.n_heads // tp, shape.n_kv_heads // tp, shape.intermediate // tp
    p = f"layer{layer}."
    wq, wk, wv = ck[p + "q_proj"], ck[p + "k_proj"], ck[p + "v_proj"]
    wg, wu = ck[p + "gate_proj"], ck[p + "up_proj"]
    qkv = torch.cat([torch.cat([wq.narrow(0, r * nh_l * hd, nh_l * hd), wk.narrow(0, r * nkv_l * hd, nkv_l * hd),
                                wv.narrow(0, r * nkv_l * hd, nkv_l * hd)]) for r in range(tp)])
    gate_up = torch.cat([torch.cat([wg.narrow(0, r * i_l, i_l), wu.narrow(0, r * i_l, i_l)]) for r in range(tp)])
    wo, wd = ck[p + "o_proj"], ck[p + "down_proj"]
    o = torch.stack([wo.narrow(1, r * nh_l * hd, nh_l * hd) for r in range(tp)])
    down = torch.stack([wd.narrow(1, r * i_l, i_l) for r in range(tp)])

    def dev(t):
        return t.contiguous().to(device)
    return LayerParams(dev(qkv), dev(o), dev(gate_up), dev(down), dev(ck[p + "input_layernorm"]),
                       dev(ck[p + "post_attention_layernorm"]), dev(ck[p + "q_norm"]), dev(ck[p + "k_norm"]))


def load_params(shape, seed: int = 0, device="cuda", n_layers: Optional[int] = None, gen_device=None) -> ModelParams:
    """Random-init parameters of the given shape from the seeded generator."""
    import seeded_inputs as si
    gen_device = gen_device or device
    nl = shape.n_layers if n_layers is None else n_layers
    embed = si.checkpoint_tensor(shape, "embed_tokens", seed, gen_device).to(device)
    layers = []
    for l in range(nl):
        ck = {n: si.checkpoint_tensor(shape, n, seed, gen_device)
              for n in si.weight_names(l) + [f"layer{l}.{x}" for x in
                                             ("input_layernorm", "post_attention_layernorm", "q_norm", "k_norm")]}
        layers.append(shard_layer(shape, ck, l, device))
        del ck
    final = si.checkpoint_tensor(shape, "norm", seed, gen_device).to(device)
    return ModelParams(embed, layers, final)


# ----------------------------------------------------------------------------
# batch descriptions (the get_context() fields, [SK] §6-§7)
# ----------------------------------------------------------------------------

@dataclass
class PrefillContext:
    ids: torch.Tensor            # int64 [T]
    positions: torch.Tensor      # int64 [T]
    cu_seqlens: torch.Tensor     # int32 [S+1]
    slot_mapping: torch.Tensor   # int64 [T]
    seq_base: torch.Tensor       # int32 [S]
    last_idx: torch.Tensor       # int32 [S]
    max_seqlen: int

    @property
    def n_tokens(self):
        return self.ids.shape[0]


@dataclass
class DecodeContext:
    ids: torch.Tensor            # int64 [B]
    positions: torch.Tensor      # int64 [B]
    context_lens: torch.Tensor   # int32 [B]
    slot_mapping: torch.Tensor   # int64 [B]
    seq_base: torch.Tensor       # int32 [B]
    max_context: int

    @property
    def n_tokens(self):
        return self.ids.shape[0]


def to_device_prefill(b, device="cuda") -> PrefillContext:
    return PrefillContext(b.ids.to(device), b.positions.to(device), b.cu_seqlens.to(device),
                          b.slot_mapping.to(device), b.seq_base.to(device), b.last_idx.to(device), max(b.seq_lens))


def to_device_decode(b, device="cuda") -> DecodeContext:
    return DecodeContext(b.ids.to(device), b.positions.to(device), b.context_lens.to(device),
                         b.slot_mapping.to(device), b.seq_base.to(device), int(b.context_lens.max()))


# ----------------------------------------------------------------------------
# the forward pass
# ----------------------------------------------------------------------------

class Qwen3Forward:
    """Device buffers + the sequence of libqw calls for prefill and decode."""

    def __init__(self, shape, params: ModelParams, max_tokens: int, num_slots: int, max_seqs: int,
                 max_context: int, device="cuda", kv_caches=None):
        self.m = shape
        self.p = params
        self.device = device
        dt = params.embed.dtype
        self.dtype = dt
        H, I, hd = shape.hidden, shape.intermediate, shape.head_dim
        tp = shape.tp
        self.qkv_width = tp * (shape.n_heads // tp + 2 * (shape.n_kv_heads // tp)) * hd
        T = max_tokens
        z = lambda *s: torch.empty(*s, dtype=dt, device=device)  # noqa: E731
        self.h = z(T, H)
        self.res = z(T, H)
        self.res2 = z(max(max_seqs, 1), H)   # decode: the residual alternates between res and res2
        self.y = z(T, H)
        self.qkv = z(T, self.qkv_width)
        self.q = z(T, shape.n_heads * hd)
        self.attn = z(T, shape.n_heads * hd)
        self.act = z(T, I)
        self.logits = z(max_seqs if max_seqs > 0 else T, shape.vocab)
        self.next_tokens = torch.empty(max(max_seqs, T), dtype=torch.int64, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        nl = len(params.layers)
        if kv_caches is None:
            self.k_cache = [torch.zeros(num_slots, shape.n_kv_heads, hd, dtype=dt, device=device) for _ in range(nl)]
            self.v_cache = [torch.zeros(num_slots, shape.n_kv_heads, hd, dtype=dt, device=device) for _ in range(nl)]
        else:
            self.k_cache, self.v_cache = kv_caches
        self.cos_sin = L.rope_cos_sin_table(shape.max_position, hd, shape.rope_theta).to(device)
        ws = 0
        for (M, N, K, mode, epi) in self._gemm_shapes(T) + self._gemm_shapes(max(max_seqs, 1)):
            ws = max(ws, L.gemm_workspace_size(M, N, K, tp, mode, epi, dt))
        ws = max(ws, L.attention_decode_workspace_size(max(max_seqs, 1), max_context, shape.n_heads, hd))
        ws = max(ws, L.lm_head_workspace_size(max(max_seqs, 1), shape.vocab, H, tp, dt))
        # completion counters at its start must be zero before the first call
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=device)
        self.scale = hd ** -0.5
        self.probe = None      # optional timing hook: probe(name, layer) -> context manager
        self.max_context = max_context
        self.max_seqs = max_seqs
        # decode batches of at most 16 tokens can run every layer in one
        # persistent kernel (qw_decode_layers); off by default: on GB300 it is
        # slower today than the per-operation kernels chained with programmatic
        # dependent launch (2.4 vs 1.4 ms per 28-layer step of 8 tokens)
        self.fused_decode = False
        # decode attention may stream cached history before the previous kernel ends
        # (valid while slot_mapping[b] == seq_base[b] + context_lens[b] - 1, which the
        # folded KV store requires anyway)
        self._history_ready = True
        self._fused = None     # (layer table, workspace), built on first use
        # prefill: QK-norm + RoPE + KV store in the QKV GEMM's epilogue (persistent
        # tensor-core kernel, the same results bit for bit); off by default: once
        # the plain QKV GEMM ran on 256-row tiles, it and the standalone kernel
        # took 19.4 ms per 8 x 2048-token prefill against 19.6 ms fused
        self.fused_qkv = False
        # prefill in five kernels per layer (QK-norm + RoPE + KV store in the QKV GEMM's
        # epilogue, residual add + RMSNorm in the o_proj and down GEMMs' epilogues);
        # off by default: on GB300 the longer epilogues, run after each tile's
        # mainloop with the tensor pipe idle, cost more than the kernels they
        # replace (8 x 2048-token prefill: 21.0 ms fused, 19.1 ms unfused)
        self.fused_prefill = False

    def _around(self, name: str, layer: int):
        if self.probe is None:
            return contextlib.nullcontext()
        return self.probe(name, layer)

    def _gemm_shapes(self, M):
        m = self.m
        return [(M, self.qkv_width, m.hidden, L.QW_GEMM_COLUMN, L.QW_EPI_NONE),
                (M, m.hidden, m.n_heads * m.head_dim, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_NONE),
                (M, 2 * m.intermediate, m.hidden, L.QW_GEMM_COLUMN, L.QW_EPI_SILU_MUL),
                (M, m.hidden, m.intermediate, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_NONE)]

    def qkv_epilogue_ok(self) -> bool:
        """Prefill: QK-norm + RoPE + KV store as the QKV GEMM's epilogue (bf16,
        head_dim 128, two whole heads of one shard per 256-column tile)."""
        m = self.m
        return (self.fused_qkv and self.dtype == torch.bfloat16 and m.head_dim == 128
                and ((m.n_heads + 2 * m.n_kv_heads) // m.tp) % 2 == 0 and m.hidden % 8 == 0)

    def prefill_fusion_ok(self) -> bool:
        """Prefill through the fused epilogues: QK-norm + RoPE + KV store in the QKV
        GEMM (two whole heads of one shard per 256-column tile), residual add +
        RMSNorm in the o_proj and down GEMMs (a row's hidden columns in one
        cluster of 256-column tiles)."""
        m = self.m
        return (self.fused_prefill and self.dtype == torch.bfloat16 and m.head_dim == 128
                and ((m.n_heads + 2 * m.n_kv_heads) // m.tp) % 2 == 0 and m.hidden % 256 == 0
                and m.hidden <= 2048 and (m.n_heads * m.head_dim // m.tp) % 8 == 0
                and (m.intermediate // m.tp) % 8 == 0 and len(self.p.layers) > 0)

    def _prefill_layer(self, l: int, T: int, ctx, first: bool, next_gamma, stream=None):
        """One decoder layer of a prefill in five kernels ([SK] §1, §8).

        On entry y holds input_layernorm(residual) (for the first layer it is
        computed here from the embedding).  On exit the residual holds the
        stream after the layer and y = RMSNorm(residual) * next_gamma (the next
        layer's input_layernorm, or the final norm); with next_gamma None, h
        holds the MLP output and the residual the stream before it, as the
        unfused layer leaves them."""
        m, p = self.m, self.p.layers[l]
        tp = m.tp
        h, res, y = self.h[:T], self.res[:T], self.y[:T]
        q, attn, act = self.q[:T], self.attn[:T], self.act[:T]
        if first:
            with self._around("prefill.add_rmsnorm", l):
                L.add_rmsnorm(h, None, res, p.input_ln, m.eps, y, stream)
        with self._around("prefill.gemm_qkv_norm_rope_store_kv", l):
            L.qkv_gemm_norm_rope_store_kv(y, p.qkv, m.n_heads, m.n_kv_heads, m.head_dim, tp, ctx.positions,
                                          self.cos_sin, p.q_norm, p.k_norm, m.eps, ctx.slot_mapping, self.k_cache[l],
                                          self.v_cache[l], q, self.err, stream)
        with self._around("prefill.attention", l):
            L.attention_prefill(q, self.k_cache[l], self.v_cache[l], ctx.cu_seqlens, ctx.cu_seqlens, ctx.seq_base,
                                ctx.max_seqlen, m.n_heads, m.n_kv_heads, m.head_dim, self.scale, attn, stream)
        with self._around("prefill.gemm_o_add_rmsnorm", l):
            L.gemm_add_rmsnorm(attn, p.o, res, p.post_ln, m.eps, y, tp, stream)
        with self._around("prefill.gemm_gate_up_silu", l):
            L.gemm(y, p.gate_up, act, 2 * m.intermediate, tp, L.QW_GEMM_COLUMN, L.QW_EPI_SILU_MUL, self.workspace,
                   stream)
        if next_gamma is None:
            with self._around("prefill.gemm_down", l):
                L.gemm(act, p.down, h, m.hidden, tp, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_NONE, self.workspace, stream)
        else:
            with self._around("prefill.gemm_down_add_rmsnorm", l):
                L.gemm_add_rmsnorm(act, p.down, res, next_gamma, m.eps, y, tp, stream)

    def norm_fusion_ok(self, T: int) -> bool:
        """Few bf16 tokens: each add+RMSNorm runs as the prologue of the GEMM it feeds."""
        return self.dtype == torch.bfloat16 and T <= 16 and T <= self.res2.shape[0]

    def _res(self, c: int, T: int):
        """Residual after update c of a decode step (two per layer) when norms are fused."""
        return (self.res if c % 2 == 0 else self.res2)[:T]

    # -- one decoder layer ([SK] §1) ------------------------------------------
    def _layer(self, l: int, T: int, ctx, first: bool, decode: bool, stream=None):
        m, p = self.m, self.p.layers[l]
        tp = m.tp
        h, res, y = self.h[:T], self.res[:T], self.y[:T]
        ph = "decode" if decode else "prefill"
        fused = decode and self.norm_fusion_ok(T)
        qkv = self.qkv[:T]
        if fused:
            # residual update 2l here, 2l+1 before gate_up; the buffers alternate
            with self._around(f"{ph}.add_rmsnorm_gemm_qkv", l):
                L.add_rmsnorm_gemm(h, None if first else self._res(2 * l - 1, T), self._res(2 * l, T), p.input_ln,
                                   m.eps, p.qkv, qkv, self.qkv_width, tp, L.QW_EPI_NONE, stream)
        else:
            with self._around(f"{ph}.add_rmsnorm", l):
                L.add_rmsnorm(h, None if first else res, res, p.input_ln, m.eps, y, stream)
            if not decode and self.qkv_epilogue_ok():
                # QK-norm + RoPE + KV store as the QKV GEMM's epilogue: no QKV round trip
                with self._around(f"{ph}.gemm_qkv_norm_rope_store_kv", l):
                    L.qkv_gemm_norm_rope_store_kv(y, p.qkv, m.n_heads, m.n_kv_heads, m.head_dim, tp, ctx.positions,
                                                  self.cos_sin, p.q_norm, p.k_norm, m.eps, ctx.slot_mapping,
                                                  self.k_cache[l], self.v_cache[l], self.q[:T], self.err, stream)
            else:
                with self._around(f"{ph}.gemm_qkv", l):
                    L.gemm(y, p.qkv, qkv, self.qkv_width, tp, L.QW_GEMM_COLUMN, L.QW_EPI_NONE, self.workspace, stream)
        q = self.q[:T]
        attn = self.attn[:T]
        if not decode and self.qkv_epilogue_ok():
            with self._around(f"{ph}.attention", l):
                L.attention_prefill(q, self.k_cache[l], self.v_cache[l], ctx.cu_seqlens, ctx.cu_seqlens, ctx.seq_base,
                                    ctx.max_seqlen, m.n_heads, m.n_kv_heads, m.head_dim, self.scale, attn, stream)
        elif decode and self.dtype == torch.bfloat16 and m.head_dim == 128:
            # QK-norm + RoPE + KV store folded into decode attention.  Sequence b's
            # cache is contiguous from seq_base[b] and this step's k/v go to its last
            # row, so the kernel before (the QKV GEMV) writes none of the cached
            # history: the history can stream in before that kernel finishes.
            with self._around(f"{ph}.attention", l):
                L.attention_decode_rope(qkv, m.n_heads, m.n_kv_heads, m.head_dim, tp, ctx.positions, self.cos_sin,
                                        p.q_norm, p.k_norm, m.eps, ctx.slot_mapping, self.k_cache[l],
                                        self.v_cache[l], self.err, ctx.context_lens, ctx.seq_base, ctx.max_context,
                                        self.scale, attn, self.workspace, stream,
                                        history_ready=self._history_ready)
        else:
            with self._around(f"{ph}.qkv_norm_rope_store_kv", l):
                L.qkv_norm_rope_store_kv(qkv, m.n_heads, m.n_kv_heads, m.head_dim, tp, ctx.positions, self.cos_sin,
                                         p.q_norm, p.k_norm, m.eps, ctx.slot_mapping, self.k_cache[l],
                                         self.v_cache[l], q, self.err, stream)
            with self._around(f"{ph}.attention", l):
                if decode:
                    L.attention_decode(q, self.k_cache[l], self.v_cache[l], ctx.context_lens, ctx.seq_base,
                                       ctx.max_context, m.n_heads, m.n_kv_heads, m.head_dim, self.scale, attn,
                                       self.workspace, stream)
                else:
                    L.attention_prefill(q, self.k_cache[l], self.v_cache[l], ctx.cu_seqlens, ctx.cu_seqlens,
                                        ctx.seq_base, ctx.max_seqlen, m.n_heads, m.n_kv_heads, m.head_dim,
                                        self.scale, attn, stream)
        with self._around(f"{ph}.gemm_o", l):
            L.gemm(attn, p.o, h, m.hidden, tp, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_NONE, self.workspace, stream)
        act = self.act[:T]
        if fused:
            # residual update 2l + 1 as the prologue of gate_up + SiluAndMul
            with self._around(f"{ph}.add_rmsnorm_gemm_gate_up", l):
                L.add_rmsnorm_gemm(h, self._res(2 * l, T), self._res(2 * l + 1, T), p.post_ln, m.eps, p.gate_up, act,
                                   2 * m.intermediate, tp, L.QW_EPI_SILU_MUL, stream)
        else:
            with self._around(f"{ph}.add_rmsnorm", l):
                L.add_rmsnorm(h, res, res, p.post_ln, m.eps, y, stream)
            with self._around(f"{ph}.gemm_gate_up_silu", l):
                L.gemm(y, p.gate_up, act, 2 * m.intermediate, tp, L.QW_GEMM_COLUMN, L.QW_EPI_SILU_MUL,
                       self.workspace, stream)
        with self._around(f"{ph}.gemm_down", l):
            L.gemm(act, p.down, h, m.hidden, tp, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_NONE, self.workspace, stream)

    def fused_decode_ok(self, B: int) -> bool:
        m = self.m
        if not self.fused_decode or self.dtype != torch.bfloat16 or len(self.p.layers) == 0 or B > self.max_seqs:
            return False
        return L.decode_layers_workspace_size(len(self.p.layers), B, m.hidden, m.n_heads, m.n_kv_heads, m.head_dim,
                                              m.intermediate, m.tp, self.max_context) > 0

    def _fused_state(self):
        if self._fused is None:
            m = self.m
            rows = [dict(input_layernorm=p.input_ln, qkv=p.qkv, q_norm=p.q_norm, k_norm=p.k_norm, o_proj=p.o,
                         post_attention_layernorm=p.post_ln, gate_up=p.gate_up, down=p.down,
                         k_cache=self.k_cache[l], v_cache=self.v_cache[l]) for l, p in enumerate(self.p.layers)]
            table = L.decode_layer_table(rows)
            ws = max(L.decode_layers_workspace_size(len(rows), b, m.hidden, m.n_heads, m.n_kv_heads, m.head_dim,
                                                    m.intermediate, m.tp, self.max_context)
                     for b in range(1, min(self.max_seqs, 16) + 1))
            # its counters must be zero before the first call; every call leaves them so
            self._fused = (table, torch.zeros(ws, dtype=torch.uint8, device=self.device))
        return self._fused

    def _decode_fused(self, ctx, stream=None):
        """embedding -> all layers + final add+RMSNorm in one persistent kernel (qw_decode_layers)."""
        m = self.m
        B = ctx.n_tokens
        table, ws = self._fused_state()
        with self._around("decode.embed_vocab", -1):
            L.embed_vocab(ctx.ids, self.p.embed, m.tp, self.h[:B], self.err, stream)
        with self._around("decode.layers", -1):
            L.decode_layers(table, len(self.p.layers), self.h[:B], ctx.positions, ctx.slot_mapping, ctx.context_lens,
                            ctx.seq_base, ctx.max_context, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate, m.tp,
                            self.cos_sin, self.k_cache[0].shape[0], m.eps, self.scale, self.p.final_norm, self.y[:B],
                            ws, self.err, stream)
        return self.y[:B]

    def run_layers(self, ctx, decode: bool, hidden_in: Optional[torch.Tensor] = None, final_norm: bool = True,
                   stream=None):
        """embedding (or hidden_in) -> layers -> optional final add+RMSNorm; returns the hidden buffer view."""
        m = self.m
        T = ctx.n_tokens
        if decode and hidden_in is None and final_norm and self.fused_decode_ok(T):
            return self._decode_fused(ctx, stream)
        if hidden_in is None:
            with self._around(f"{'decode' if decode else 'prefill'}.embed_vocab", -1):
                L.embed_vocab(ctx.ids, self.p.embed, m.tp, self.h[:T], self.err, stream)
        else:
            self.h[:T].copy_(hidden_in)
        nl = len(self.p.layers)
        if not decode and self.prefill_fusion_ok():
            for l in range(nl):
                nxt = self.p.layers[l + 1].input_ln if l + 1 < nl else (self.p.final_norm if final_norm else None)
                self._prefill_layer(l, T, ctx, l == 0, nxt, stream)
            if final_norm:
                return self.y[:T]   # the last down GEMM applied the final norm
            return self.h[:T], self.res[:T]
        for l in range(nl):
            self._layer(l, T, ctx, l == 0, decode, stream)
        nl = len(self.p.layers)
        res = self._res(2 * nl - 1, T) if decode and self.norm_fusion_ok(T) and nl > 0 else self.res[:T]
        if not final_norm:
            return self.h[:T], res
        with self._around("final_norm", -1):
            L.add_rmsnorm(self.h[:T], None if nl == 0 else res, None, self.p.final_norm, m.eps, self.y[:T], stream)
        return self.y[:T]

    def compute_logits(self, hidden: torch.Tensor, last_idx: Optional[torch.Tensor], n_out: int, stream=None):
        """ParallelLMHead ([SK] §6): last token of each sequence in prefill, then greedy argmax."""
        logits = self.logits[:n_out]
        nt = self.next_tokens[:n_out]
        with self._around("lm_head", -1):
            L.lm_head(hidden, last_idx, n_out, self.p.embed, self.m.tp, logits, nt, self.workspace, stream)
        return logits, nt

    def prefill(self, ctx: PrefillContext, stream=None):
        hidden = self.run_layers(ctx, decode=False, stream=stream)
        return self.compute_logits(hidden, ctx.last_idx, ctx.last_idx.shape[0], stream)

    def decode(self, ctx: DecodeContext, stream=None):
        hidden = self.run_layers(ctx, decode=True, stream=stream)
        return self.compute_logits(hidden, None, ctx.n_tokens, stream)
