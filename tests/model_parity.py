"""Run the same seeded batch through the CUDA path and the oracle (test helper)."""
import contextlib
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
            fwd_out=None) -> Trace:
    from qwen3_transformer_forward_gb300 import model as M
    from qwen3_transformer_forward_gb300 import _lib as L
    params = params or M.load_params(m, device=device)
    b = si.prefill_batch(m, seq_lens, extra_capacity=decode_steps)
    B = len(seq_lens)
    fwd = M.Qwen3Forward(m, params, max_tokens=sum(seq_lens), num_slots=b.num_slots, max_seqs=B,
                         max_context=max(seq_lens) + decode_steps)
    fwd.fused_decode = fused_decode
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


@contextlib.contextmanager
def bf16_softmax_weights():
    """Temporarily makes the oracle round its softmax weights to bf16 before the
    PV product (what a flash-style tensor-core kernel does).  Used only to
    measure how much the model's outputs move under that one rounding; the
    oracle proper always uses the exact weights."""
    import oracle.qwen3 as Q
    exact = Q._softmax_rows

    def rounded(s):
        mx = np.max(s, axis=-1, keepdims=True)
        e = np.exp(s - mx)
        return O.bf16_round(e) / np.sum(e, axis=-1, keepdims=True)
    Q._softmax_rows = rounded
    try:
        yield
    finally:
        Q._softmax_rows = exact


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


def argmax_agreement(gpu_logits: np.ndarray, ref_logits: np.ndarray, tol: float):
    """(fraction of rows with equal argmax, rows whose disagreement is NOT a near-tie).

    Where the argmaxes differ, the oracle's logit at the GPU's choice must lie
    within `tol` of the oracle's maximum: the two logits are equal within the
    stated logit tolerance, so either token is a correct greedy choice.
    """
    g = O.greedy(gpu_logits)
    r = O.greedy(ref_logits)
    same = g == r
    rows = np.arange(len(g))
    gap = ref_logits[rows, r] - ref_logits[rows, g]
    bad = (~same) & (gap > tol)
    return float(np.mean(same)), np.nonzero(bad)[0]
