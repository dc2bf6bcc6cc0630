"""ctypes binding of libqw (the C ABI declared in include/qw.h).

Argument marshalling only: every wrapper checks nothing numerical, passes
device pointers, sizes and the current CUDA stream, and raises QwError on a
non-zero status.  There is no fallback: without the built library on a
CUDA device every call fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os
from pathlib import Path
from typing import Optional

import torch

_LIB_PATH = Path(__file__).resolve().parent / "libqw.so"
_lib = None

QW_OK, QW_ERR_INVALID_ARG, QW_ERR_SHAPE, QW_ERR_DTYPE, QW_ERR_CUDA, QW_ERR_TIMEOUT, QW_ERR_WORKSPACE = range(7)
QW_BF16, QW_F32 = 0, 1
QW_GEMM_COLUMN, QW_GEMM_ROW_REDUCE = 0, 1
QW_EPI_NONE, QW_EPI_SILU_MUL = 0, 1

_p, _i64, _i32, _f32, _f64, _sz = C.c_void_p, C.c_int64, C.c_int, C.c_float, C.c_double, C.c_size_t

# name -> (restype, argtypes); mirrors include/qw.h
SIGNATURES = {
    "qw_abi_version": (C.c_int, []),
    "qw_last_error_string": (C.c_char_p, []),
    "qw_device_error": (C.c_int, [_p]),
    "qw_embed_vocab": (C.c_int, [_p, _i64, _p, _i64, _i64, _i32, _p, _p, _i32, _p]),
    "qw_add_rmsnorm": (C.c_int, [_p, _p, _p, _p, _f32, _i64, _i64, _p, _i32, _p]),
    "qw_rope_cos_sin_table": (C.c_int, [_p, _i64, _i32, _f64]),
    "qw_qkv_norm_rope_store_kv": (C.c_int, [_p, _i64, _i32, _i32, _i32, _i32, _p, _p, _i64, _p, _p, _f32, _p, _p,
                                            _p, _i64, _p, _p, _i32, _p]),
    "qw_gemm_add_rmsnorm": (C.c_int, [_p, _p, _i64, _i64, _i64, _i32, _p, _p, _f32, _p, _i32, _p]),
    "qw_qkv_gemm_norm_rope_store_kv": (C.c_int, [_p, _p, _i64, _i64, _i32, _i32, _i32, _i32, _p, _p, _i64, _p, _p,
                                                 _f32, _p, _p, _p, _i64, _p, _p, _i32, _p]),
    "qw_attention_prefill": (C.c_int, [_p, _p, _p, _i64, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _f32, _p, _i32, _p]),
    "qw_attention_decode": (C.c_int, [_p, _p, _p, _i64, _p, _p, _i32, _i32, _i32, _i32, _i32, _f32, _p, _p, _sz,
                                      _i32, _i32, _p]),
    "qw_attention_decode_workspace_size": (C.c_size_t, [_i32, _i32, _i32, _i32]),
    "qw_attention_decode_paged": (C.c_int, [_p, _p, _p, _i64, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32,
                                            _p, _p, _sz, _i32, _i32, _p]),
    "qw_attention_prefill_paged": (C.c_int, [_p, _p, _p, _i64, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                             _f32, _p, _i32, _p]),
    "qw_attention_decode_rope": (C.c_int, [_p, _i32, _i32, _i32, _i32, _p, _p, _i64, _p, _p, _f32, _p, _p, _p, _i64,
                                           _p, _p, _p, _i32, _i32, _f32, _p, _p, _sz, _i32, _i32, _p]),
    "qw_attention_decode_static": (C.c_int, [_p, _p, _p, _i64, _p, _p, _i32, _i32, _i32, _i32, _i32, _f32, _p, _i32,
                                             _p]),
    "qw_attention_decode_static_scratch_bytes": (C.c_size_t, []),
    "qw_gemm": (C.c_int, [_p, _p, _p, _i64, _i64, _i64, _i32, _i32, _i32, _p, _sz, _i32, _p]),
    "qw_gemm_workspace_size": (C.c_size_t, [_i64, _i64, _i64, _i32, _i32, _i32, _i32]),
    "qw_silu_mul": (C.c_int, [_p, _p, _i64, _i64, _i32, _i32, _p]),
    "qw_lm_head": (C.c_int, [_p, _i64, _p, _i64, _p, _i64, _i64, _i32, _p, _p, _p, _sz, _i32, _p]),
    "qw_lm_head_workspace_size": (C.c_size_t, [_i64, _i64, _i64, _i32, _i32]),
    "qw_argmax": (C.c_int, [_p, _i64, _i64, _p, _i32, _p]),
    "qw_sample": (C.c_int, [_p, _i64, _i64, _p, _p, _p, _p, _p, _sz, _i32, _p]),
    "qw_sample_workspace_size": (C.c_size_t, [_i64, _i64]),
    "qw_selftest_wait_timeout": (C.c_int, [_p]),
    "qw_add_rmsnorm_gemm": (C.c_int, [_p, _p, _p, _p, _f32, _p, _p, _i64, _i64, _i64, _i32, _i32, _i32, _p]),
    "qw_decode_layers": (C.c_int, [_p, _i32, _p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _p,
                                   _i64, _i64, _f32, _f32, _p, _p, _p, _p, _sz, _p]),
    "qw_decode_layers_workspace_size": (C.c_size_t, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32]),
}

# field order of qw_decode_layer (include/qw.h)
DECODE_LAYER_FIELDS = ("input_layernorm", "qkv", "q_norm", "k_norm", "o_proj", "post_attention_layernorm", "gate_up",
                       "down", "k_cache", "v_cache")


class QwError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[qw status {code}] {msg}")
        self.code = code


def lib_path() -> Path:
    return _LIB_PATH


def load(path: Optional[os.PathLike] = None):
    """Loads libqw.so (built in-tree by build.py) and declares every signature."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path is not None else _LIB_PATH
    if not p.exists():
        raise QwError(-1, f"{p} is missing: build it with qwen3_transformer_forward_gb300.build.build()")
    lib = C.CDLL(str(p))
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(rc: int):
    if rc != QW_OK:
        raise QwError(rc, load().qw_last_error_string().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return t.data_ptr()


def _dev_ptr(t: Optional[torch.Tensor], name: str):
    if t is None:
        return None
    if not t.is_cuda:
        raise QwError(QW_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise QwError(QW_ERR_INVALID_ARG, f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return QW_BF16
    if t == torch.float32:
        return QW_F32
    raise QwError(QW_ERR_DTYPE, f"unsupported dtype {t}")


# ----------------------------------------------------------------------------
# thin wrappers (same names as the C entry points, without the qw_ prefix)
# ----------------------------------------------------------------------------

def abi_version() -> int:
    return load().qw_abi_version()


def device_error(stream=None):
    _check(load().qw_device_error(_stream(stream)))


def embed_vocab(ids, table, tp, out, err_count=None, stream=None):
    T, H = out.shape
    _check(load().qw_embed_vocab(_dev_ptr(ids, "ids"), T, _dev_ptr(table, "table"), table.shape[0], H, tp,
                                 _dev_ptr(out, "out"), _dev_ptr(err_count, "err_count"), dtype_code(table.dtype),
                                 _stream(stream)))


def add_rmsnorm(x, residual_in, residual_out, gamma, eps, y, stream=None):
    T, H = x.shape
    _check(load().qw_add_rmsnorm(_dev_ptr(x, "x"), _dev_ptr(residual_in, "residual_in"),
                                 _dev_ptr(residual_out, "residual_out"), _dev_ptr(gamma, "gamma"), eps, T, H,
                                 _dev_ptr(y, "y"), dtype_code(x.dtype), _stream(stream)))


def rope_cos_sin_table(max_position: int, rotary_dim: int, theta: float) -> torch.Tensor:
    """Host-side table [max_position, rotary_dim] (float32, CPU tensor)."""
    out = torch.empty((max_position, rotary_dim), dtype=torch.float32)
    _check(load().qw_rope_cos_sin_table(out.data_ptr(), max_position, rotary_dim, theta))
    return out


def qkv_norm_rope_store_kv(qkv, n_heads, n_kv_heads, head_dim, tp, positions, cos_sin, q_gamma, k_gamma, eps,
                           slot_mapping, k_cache, v_cache, q_out, err_count=None, stream=None):
    T = qkv.shape[0]
    _check(load().qw_qkv_norm_rope_store_kv(
        _dev_ptr(qkv, "qkv"), T, n_heads, n_kv_heads, head_dim, tp, _dev_ptr(positions, "positions"),
        _dev_ptr(cos_sin, "cos_sin"), cos_sin.shape[0], _dev_ptr(q_gamma, "q_gamma"), _dev_ptr(k_gamma, "k_gamma"),
        eps, _dev_ptr(slot_mapping, "slot_mapping"), _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"),
        k_cache.shape[0], _dev_ptr(q_out, "q_out"), _dev_ptr(err_count, "err_count"), dtype_code(qkv.dtype),
        _stream(stream)))


def gemm_add_rmsnorm(A, W, residual, gamma, eps, y, tp, stream=None):
    """Row-parallel GEMM whose output is added to the residual in place, then RMSNorm into y (qw_gemm_add_rmsnorm)."""
    M, K = A.shape
    N = residual.shape[1]
    _check(load().qw_gemm_add_rmsnorm(_dev_ptr(A, "A"), _dev_ptr(W, "W"), M, N, K, tp, _dev_ptr(residual, "residual"),
                                      _dev_ptr(gamma, "gamma"), eps, _dev_ptr(y, "y"), dtype_code(A.dtype),
                                      _stream(stream)))


def qkv_gemm_norm_rope_store_kv(A, W, n_heads, n_kv_heads, head_dim, tp, positions, cos_sin, q_gamma, k_gamma, eps,
                                slot_mapping, k_cache, v_cache, q_out, err_count=None, stream=None):
    """Merged QKV GEMM with QK-RMSNorm + RoPE + KV store as its epilogue (qw_qkv_gemm_norm_rope_store_kv)."""
    T, H = A.shape
    _check(load().qw_qkv_gemm_norm_rope_store_kv(
        _dev_ptr(A, "A"), _dev_ptr(W, "W"), T, H, n_heads, n_kv_heads, head_dim, tp, _dev_ptr(positions, "positions"),
        _dev_ptr(cos_sin, "cos_sin"), cos_sin.shape[0], _dev_ptr(q_gamma, "q_gamma"), _dev_ptr(k_gamma, "k_gamma"), eps,
        _dev_ptr(slot_mapping, "slot_mapping"), _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"),
        k_cache.shape[0], _dev_ptr(q_out, "q_out"), _dev_ptr(err_count, "err_count"), dtype_code(A.dtype),
        _stream(stream)))


def attention_prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, seq_base, max_seqlen_q, n_heads, n_kv_heads, head_dim,
                      scale, out, stream=None):
    n_seqs = cu_seqlens_q.shape[0] - 1
    _check(load().qw_attention_prefill(
        _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), k.shape[0], _dev_ptr(cu_seqlens_q, "cu_seqlens_q"),
        _dev_ptr(cu_seqlens_k, "cu_seqlens_k"), _dev_ptr(seq_base, "seq_base"), n_seqs, max_seqlen_q, n_heads,
        n_kv_heads, head_dim, scale, _dev_ptr(out, "out"), dtype_code(q.dtype), _stream(stream)))


def attention_decode_workspace_size(B, max_context, n_heads, head_dim) -> int:
    return load().qw_attention_decode_workspace_size(B, max_context, n_heads, head_dim)


QW_DECODE_HISTORY_READY = 1


def attention_decode(q, k_cache, v_cache, context_lens, seq_base, max_context, n_heads, n_kv_heads, head_dim, scale,
                     out, workspace=None, stream=None, history_ready=False):
    """history_ready: the previous kernel on the stream writes only q and each sequence's last cache row
    (see QW_DECODE_HISTORY_READY in qw.h)."""
    B = q.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().qw_attention_decode(
        _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), k_cache.shape[0],
        _dev_ptr(context_lens, "context_lens"), _dev_ptr(seq_base, "seq_base"), B, max_context, n_heads, n_kv_heads,
        head_dim, scale, _dev_ptr(out, "out"), _dev_ptr(workspace, "workspace"), ws_bytes, dtype_code(q.dtype),
        QW_DECODE_HISTORY_READY if history_ready else 0, _stream(stream)))


def attention_decode_rope(qkv, n_heads, n_kv_heads, head_dim, tp, positions, cos_sin, q_gamma, k_gamma, eps,
                          slot_mapping, k_cache, v_cache, err_count, context_lens, seq_base, max_context, scale, out,
                          workspace, stream=None, history_ready=False):
    """QK-norm + RoPE + KV store of one decode token per sequence, then decode attention, in one launch."""
    B = qkv.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().qw_attention_decode_rope(
        _dev_ptr(qkv, "qkv"), n_heads, n_kv_heads, head_dim, tp, _dev_ptr(positions, "positions"),
        _dev_ptr(cos_sin, "cos_sin"), cos_sin.shape[0], _dev_ptr(q_gamma, "q_gamma"), _dev_ptr(k_gamma, "k_gamma"),
        eps, _dev_ptr(slot_mapping, "slot_mapping"), _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"),
        k_cache.shape[0], _dev_ptr(err_count, "err_count"), _dev_ptr(context_lens, "context_lens"),
        _dev_ptr(seq_base, "seq_base"), B, max_context, scale, _dev_ptr(out, "out"), _dev_ptr(workspace, "workspace"),
        ws_bytes, dtype_code(qkv.dtype), QW_DECODE_HISTORY_READY if history_ready else 0, _stream(stream)))


def attention_decode_paged(q, k_cache, v_cache, context_lens, block_table, block_size, max_context, n_heads,
                           n_kv_heads, head_dim, scale, out, workspace, stream=None, history_ready=False):
    """Decode attention over a paged cache: block_table int32 [B, max_blocks]."""
    B = q.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().qw_attention_decode_paged(
        _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), k_cache.shape[0],
        _dev_ptr(context_lens, "context_lens"), _dev_ptr(block_table, "block_table"), block_table.shape[1],
        block_size, B, max_context, n_heads, n_kv_heads, head_dim, scale, _dev_ptr(out, "out"),
        _dev_ptr(workspace, "workspace"), ws_bytes, dtype_code(q.dtype), QW_DECODE_HISTORY_READY if history_ready else 0,
        _stream(stream)))


def attention_prefill_paged(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, block_size, max_seqlen_q,
                            n_heads, n_kv_heads, head_dim, scale, out, stream=None):
    """Causal prefill attention with every key read from a paged cache (prefix-cache prefill)."""
    n_seqs = cu_seqlens_q.shape[0] - 1
    _check(load().qw_attention_prefill_paged(
        _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), k_cache.shape[0],
        _dev_ptr(cu_seqlens_q, "cu_seqlens_q"), _dev_ptr(cu_seqlens_k, "cu_seqlens_k"),
        _dev_ptr(block_table, "block_table"), block_table.shape[1], block_size, n_seqs, max_seqlen_q, n_heads,
        n_kv_heads, head_dim, scale, _dev_ptr(out, "out"), dtype_code(q.dtype), _stream(stream)))


def attention_decode_static(q, k_cache, v_cache, context_lens, seq_base, max_context, n_heads, n_kv_heads,
                            head_dim, scale, out, stream=None):
    """Decode attention whose split-KV scratch is the library's fixed device array (no workspace)."""
    B = q.shape[0]
    _check(load().qw_attention_decode_static(
        _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), k_cache.shape[0],
        _dev_ptr(context_lens, "context_lens"), _dev_ptr(seq_base, "seq_base"), B, max_context, n_heads, n_kv_heads,
        head_dim, scale, _dev_ptr(out, "out"), dtype_code(q.dtype), _stream(stream)))


def attention_decode_static_scratch_bytes() -> int:
    return load().qw_attention_decode_static_scratch_bytes()


def gemm_workspace_size(M, N, K, tp, mode, epilogue, dtype) -> int:
    return load().qw_gemm_workspace_size(M, N, K, tp, mode, epilogue, dtype_code(dtype))


def gemm(A, W, C_out, N, tp=1, mode=QW_GEMM_COLUMN, epilogue=QW_EPI_NONE, workspace=None, stream=None):
    M, K = A.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().qw_gemm(_dev_ptr(A, "A"), _dev_ptr(W, "W"), _dev_ptr(C_out, "C"), M, N, K, tp, mode, epilogue,
                          _dev_ptr(workspace, "workspace"), ws_bytes, dtype_code(A.dtype), _stream(stream)))


def silu_mul(x, out, tp, stream=None):
    T, I = out.shape
    _check(load().qw_silu_mul(_dev_ptr(x, "x"), _dev_ptr(out, "out"), T, I, tp, dtype_code(x.dtype),
                              _stream(stream)))


def lm_head_workspace_size(n_out, V, H, tp, dtype) -> int:
    return load().qw_lm_head_workspace_size(n_out, V, H, tp, dtype_code(dtype))


def lm_head(hidden, last_idx, n_out, table, tp, logits, next_tokens=None, workspace=None, stream=None):
    T, H = hidden.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().qw_lm_head(_dev_ptr(hidden, "hidden"), T, _dev_ptr(last_idx, "last_idx"), n_out,
                             _dev_ptr(table, "table"), table.shape[0], H, tp, _dev_ptr(logits, "logits"),
                             _dev_ptr(next_tokens, "next_tokens"), _dev_ptr(workspace, "workspace"), ws_bytes,
                             dtype_code(hidden.dtype), _stream(stream)))


def argmax(logits, out, stream=None):
    M, V = logits.shape
    _check(load().qw_argmax(_dev_ptr(logits, "logits"), M, V, _dev_ptr(out, "out"), dtype_code(logits.dtype),
                            _stream(stream)))


def sample_workspace_size(B, V) -> int:
    return load().qw_sample_workspace_size(B, V)


def sample(logits, temperature, top_p, uniforms, out, workspace, stream=None):
    """Temperature / top-p sampling (qw_sample): one token per logits row into out."""
    B, V = logits.shape
    _check(load().qw_sample(_dev_ptr(logits, "logits"), B, V, _dev_ptr(temperature, "temperature"),
                            _dev_ptr(top_p, "top_p"), _dev_ptr(uniforms, "uniforms"), _dev_ptr(out, "out"),
                            _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                            dtype_code(logits.dtype), _stream(stream)))


def selftest_wait_timeout(stream=None):
    """Launches a bounded wait that runs out; the next device_error() raises QW_ERR_TIMEOUT."""
    _check(load().qw_selftest_wait_timeout(_stream(stream)))


class DecodeLayer(C.Structure):
    """qw_decode_layer (include/qw.h): one layer's device pointers."""
    _fields_ = [(f, C.c_void_p) for f in DECODE_LAYER_FIELDS]


def decode_layer_table(layers):
    """Host array of qw_decode_layer records: one dict of CUDA tensors per
    layer (keys DECODE_LAYER_FIELDS).  The tensors must outlive its use."""
    arr = (DecodeLayer * len(layers))()
    for i, lw in enumerate(layers):
        for f in DECODE_LAYER_FIELDS:
            setattr(arr[i], f, _dev_ptr(lw[f], f))
    return arr


def decode_layers_workspace_size(n_layers, B, H, n_heads, n_kv_heads, head_dim, intermediate, tp, max_context) -> int:
    return load().qw_decode_layers_workspace_size(n_layers, B, H, n_heads, n_kv_heads, head_dim, intermediate, tp,
                                                  max_context)


def decode_layers(table, n_layers, x, positions, slot_mapping, context_lens, seq_base, max_context, n_heads,
                  n_kv_heads, head_dim, intermediate, tp, cos_sin, num_slots, eps, scale, final_norm, out,
                  workspace, err_count=None, stream=None):
    B, H = x.shape
    _check(load().qw_decode_layers(
        C.cast(table, C.c_void_p), n_layers, _dev_ptr(x, "x"), _dev_ptr(positions, "positions"),
        _dev_ptr(slot_mapping, "slot_mapping"), _dev_ptr(context_lens, "context_lens"), _dev_ptr(seq_base, "seq_base"),
        B, max_context, H, n_heads, n_kv_heads, head_dim, intermediate, tp, _dev_ptr(cos_sin, "cos_sin"),
        cos_sin.shape[0], num_slots, eps, scale, _dev_ptr(final_norm, "final_norm"), _dev_ptr(out, "out"),
        _dev_ptr(err_count, "err_count"), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def add_rmsnorm_gemm(x, residual_in, residual_out, gamma, eps, W, C, N, tp, epilogue=QW_EPI_NONE, stream=None):
    """C = RMSNorm(x + residual_in) * gamma @ W^T for few tokens; residual_out = x + residual_in."""
    M, K = x.shape
    _check(load().qw_add_rmsnorm_gemm(
        _dev_ptr(x, "x"), _dev_ptr(residual_in, "residual_in"), _dev_ptr(residual_out, "residual_out"),
        _dev_ptr(gamma, "gamma"), eps, _dev_ptr(W, "W"), _dev_ptr(C, "C"), M, N, K, tp, epilogue,
        dtype_code(x.dtype), _stream(stream)))
