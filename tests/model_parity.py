"""Run the same seeded batch through the CUDA path and the oracle (test helper)."""
from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

import oracle as O
import seeded_inputs as si


@dataclass
class Trace:
    hidden: List[np.ndarray]      # final (normed) hidden per phase
    logits: List[np.ndarray]      # logits per phase
    tokens: List[np.ndarray]      # argmax per phase


def forced_tokens(m, steps: int, B: int, seed: int = 0) -> torch.Tensor:
    """Seeded decode inputs used by parity runs in place of the greedy feedback."""
    return si.uniform_int(seed, "decode.forced_ids", (steps, B), 0, m.vocab)


def decode_meta(seq_lens, step: int, extra: int):
    """Positions / context lengths / slots of decode step `step` after a prefill of seq_lens."""
    cap = [L + extra for L in seq_lens]
    base = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    pos = np.array([L + step for L in seq_lens], dtype=np.int64)
    return pos, (pos + 1).astype(np.int32), base + pos, base.astype(np.int32)


def run_gpu(m, seq_lens, decode_steps: int, params=None, forced=None, device="cuda", fused_decode=False,
            fwd_out=None, prefill_fusion=False) -> Trace:
    """prefill_fusion: the opt-in prefill epilogues (QK-norm + RoPE + KV store in
    the QKV GEMM, residual add + RMSNorm in the o_proj and down GEMMs)."""
    from qwen3_transformer_forward_gb300 import model as M
    from qwen3_transformer_forward_gb300 import _lib as L
    params = params or M.load_params(m, device=device)
    b = si.prefill_batch(m, seq_lens, extra_capacity=decode_steps)
    B = len(seq_lens)
    fwd = M.Qwen3Forward(m, params, max_tokens=sum(seq_lens), num_slots=b.num_slots, max_seqs=B,
                         max_context=max(seq_lens) + decode_steps)
    fwd.fused_decode = fused_decode
    fwd.fused_qkv = fwd.fused_prefill = prefill_fusion
    if fwd_out is not None:
        fwd_out.append(fwd)
    ctx = M.to_device_prefill(b, device)
    hid, log, tok = [], [], []
    h = fwd.run_layers(ctx, decode=False)
    hid.append(h[ctx.last_idx.long()].double().cpu().numpy())
    lg, nt = fwd.compute_logits(h, ctx.last_idx, B)
    log.append(lg.double().cpu().numpy())
    tok.append(nt.cpu().numpy().copy())
    for s in range(decode_steps):
        pos, cl, slots, base = decode_meta(seq_lens, s, decode_steps)
        ids = forced[s] if forced is not None else torch.from_numpy(tok[-1])
        dctx = M.DecodeContext(ids.to(device), torch.from_numpy(pos).to(device), torch.from_numpy(cl).to(device),
                               torch.from_numpy(slots).to(device), torch.from_numpy(base).to(device), int(cl.max()))
        h = fwd.run_layers(dctx, decode=True)
        hid.append(h.double().cpu().numpy())
        lg, nt = fwd.compute_logits(h, None, B)
        log.append(lg.double().cpu().numpy())
        tok.append(nt.cpu().numpy().copy())
    torch.cuda.synchronize()
    L.device_error()
    return Trace(hid, log, tok)


def run_oracle(m, seq_lens, decode_steps: int, forced=None, weights=None) -> Trace:
    w = weights or O.load_weights(m)
    b = si.prefill_batch(m, seq_lens, extra_capacity=decode_steps)
    B = len(seq_lens)
    cache = O.KVCache(m.n_layers, b.num_slots, m.n_kv_heads, m.head_dim, m.tp)
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    ctx = O.AttnContext(True, b.slot_mapping.numpy(), cu_seqlens=b.cu_seqlens.numpy())
    h = O.model_forward(m, w, b.ids.numpy(), b.positions.numpy(), ctx, cache, cos_sin)
    last = b.last_idx.numpy()
    hid = [h[last]]
    lg = O.compute_logits(m, w.embed, h, m.tp, b.cu_seqlens.numpy())
    log, tok = [lg], [O.greedy(lg)]
    for s in range(decode_steps):
        pos, cl, slots, base = decode_meta(seq_lens, s, decode_steps)
        ids = forced[s].numpy() if forced is not None else tok[-1]
        dctx = O.AttnContext(False, slots, seq_base=base, context_lens=cl)
        h = O.model_forward(m, w, ids, pos, dctx, cache, cos_sin)
        lg = O.compute_logits(m, w.embed, h, m.tp)
        hid.append(h)
        log.append(lg)
        tok.append(O.greedy(lg))
    return Trace(hid, log, tok)


def oracle_prefill_layerwise(m, w, ids, seq_lens, rows):
    """The oracle's prefill of packed sequences, one layer at a time, returning the
    final hidden state and logits of the given token rows.

    Same calls and order as O.model_forward (embedding, decoder layers, final
    add+RMSNorm, lm_head); the only difference is memory: prefill attention reads
    the batch's fresh keys, never the cache, so each layer gets a scratch cache
    that is dropped after it.  Used for long teacher-forced sequences: the
    outputs at position p of a sequence are those of a decode step at p fed the
    same earlier tokens (causality; pinned for the oracle by the prefill/decode
    consistency tests)."""
    ids = np.asarray(ids, dtype=np.int64)
    T = ids.shape[0]
    cu = np.concatenate([[0], np.cumsum(seq_lens)]).astype(np.int64)
    positions = np.concatenate([np.arange(L) for L in seq_lens]).astype(np.int64)
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    h = O.vocab_parallel_embedding(ids, w.embed, m.tp)
    res = None
    for l in range(m.n_layers):
        cache = O.KVCache(1, T, m.n_kv_heads, m.head_dim, m.tp)
        ctx = O.AttnContext(True, np.arange(T), cu_seqlens=cu)
        h, res = O.decoder_layer(m, w.layers[l], 0, positions, h, res, ctx, cache, *cos_sin)
    h, _ = O.add_rms_norm(h[rows], res[rows], w.final_norm, m.eps, m.dtype)
    return h, O.compute_logits(m, w.embed, h, m.tp)


def oracle_decode_layerwise(m, w, ids, positions, context_lens, slots, seq_base, num_slots, history):
    """One decode step of a batch through the oracle, one layer at a time.

    history(l) returns layer l's cache contents before the step as float64
    arrays k, v [num_slots, n_kv_heads, head_dim]; the oracle stores the step's
    own k/v rows and attends over context_lens[b] rows from seq_base[b].  Same
    calls and order as O.model_forward, with one layer's cache alive at a
    time."""
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    h = O.vocab_parallel_embedding(np.asarray(ids, dtype=np.int64), w.embed, m.tp)
    res = None
    nkv_l = m.n_kv_heads // m.tp
    ctx = O.AttnContext(False, np.asarray(slots), seq_base=np.asarray(seq_base), context_lens=np.asarray(context_lens))
    for l in range(m.n_layers):
        cache = O.KVCache(1, num_slots, m.n_kv_heads, m.head_dim, m.tp)
        k, v = history(l)
        for r in range(m.tp):
            cache.k[r][0][:] = k[:, r * nkv_l:(r + 1) * nkv_l]
            cache.v[r][0][:] = v[:, r * nkv_l:(r + 1) * nkv_l]
        del k, v
        h, res = O.decoder_layer(m, w.layers[l], 0, np.asarray(positions), h, res, ctx, cache, *cos_sin)
        del cache
    h, _ = O.add_rms_norm(h, res, w.final_norm, m.eps, m.dtype)
    return h, O.compute_logits(m, w.embed, h, m.tp)
