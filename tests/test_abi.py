"""Host-side checks of the C ABI (no GPU needed).

The library builds with nvcc for sm_103a, loads, exports every entry point
declared in include/qw.h, rejects bad arguments before touching the device,
and its host-only RoPE table equals the oracle's bit for bit.
"""
import ctypes as C
import os
import re

import numpy as np
import pytest
import torch

import oracle as O
from qwen3_transformer_forward_gb300 import _lib as L
from qwen3_transformer_forward_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "qw.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qw_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert len(syms) >= 15
    for s in syms:
        assert hasattr(lib, s), s
    # and the binding declares a signature for each of them
    assert set(syms) == set(L.SIGNATURES), set(syms) ^ set(L.SIGNATURES)


def test_abi_version(lib):
    assert lib.qw_abi_version() == 9


def test_argument_errors_are_reported_before_launch(lib):
    fake = C.c_void_p(16)   # never dereferenced: every call below fails its host-side check
    # V not divisible by tp
    assert lib.qw_embed_vocab(fake, 4, fake, 10, 64, 4, fake, None, L.QW_BF16, None) == L.QW_ERR_SHAPE
    assert "not divisible" in lib.qw_last_error_string().decode()
    # bad dtype
    assert lib.qw_embed_vocab(fake, 4, fake, 8, 64, 2, fake, None, 7, None) == L.QW_ERR_DTYPE
    # zero tokens is a no-op
    assert lib.qw_embed_vocab(None, 0, fake, 8, 64, 2, fake, None, L.QW_BF16, None) == L.QW_OK
    # null pointer
    assert lib.qw_add_rmsnorm(None, None, None, fake, 1e-6, 3, 64, fake, L.QW_BF16, None) == L.QW_ERR_INVALID_ARG
    # misaligned
    assert lib.qw_add_rmsnorm(C.c_void_p(18), None, None, fake, 1e-6, 3, 64, fake, L.QW_BF16,
                              None) == L.QW_ERR_INVALID_ARG
    # heads not divisible by tp
    assert lib.qw_qkv_norm_rope_store_kv(fake, 3, 16, 8, 128, 3, fake, fake, 64, fake, fake, 1e-6, fake, fake, fake,
                                         10, fake, None, L.QW_BF16, None) == L.QW_ERR_SHAPE
    # gemm: K/tp not a multiple of 8, SiluAndMul with the row layout, N not a multiple of 16
    assert lib.qw_gemm(fake, fake, fake, 4, 64, 36, 2, L.QW_GEMM_ROW_REDUCE, 0, None, 0, L.QW_BF16,
                       None) == L.QW_ERR_SHAPE
    assert lib.qw_gemm(fake, fake, fake, 4, 64, 64, 1, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_SILU_MUL, None, 0, L.QW_BF16,
                       None) == L.QW_ERR_INVALID_ARG
    assert lib.qw_gemm(fake, fake, fake, 4, 60, 64, 1, L.QW_GEMM_COLUMN, 0, None, 0, L.QW_BF16,
                       None) == L.QW_ERR_SHAPE
    # attention: head_dim must be 128 (bf16) or <= 64; decode group must be 1/2/4/8
    assert lib.qw_attention_prefill(fake, fake, fake, 64, fake, fake, None, 2, 8, 16, 8, 96, 0.1, fake, L.QW_BF16,
                                    None) == L.QW_ERR_SHAPE
    assert lib.qw_attention_prefill(fake, fake, fake, 64, fake, fake, None, 2, 8, 16, 8, 128, 0.1, fake, L.QW_F32,
                                    None) == L.QW_ERR_SHAPE
    assert lib.qw_attention_decode(fake, fake, fake, 100, fake, fake, 2, 8, 12, 4, 128, 0.1, fake, None, 0,
                                   L.QW_BF16, 0, None) == L.QW_ERR_SHAPE
    # decode without the workspace it needs
    need = lib.qw_attention_decode_workspace_size(8, 4096, 16, 128)
    assert need > 0
    assert lib.qw_attention_decode(fake, fake, fake, 100, fake, fake, 8, 4096, 16, 8, 128, 0.1, fake, None, 0,
                                   L.QW_BF16, 0, None) == L.QW_ERR_WORKSPACE
    # unknown flags
    assert lib.qw_attention_decode(fake, fake, fake, 100, fake, fake, 8, 4096, 16, 8, 128, 0.1, fake, None, 0,
                                   L.QW_BF16, 2, None) == L.QW_ERR_INVALID_ARG
    # paged decode / prefill: bf16, head_dim 128, block size a multiple of the key tile, context within the table
    pd = lambda bs, maxb, mc, table, dt: (fake, fake, fake, 100, fake, table, maxb, bs, 8, mc, 16, 8, 128, 0.1, fake,  # noqa: E731
                                          None, 0, dt, 0, None)
    assert lib.qw_attention_decode_paged(*pd(256, 4, 1024, fake, L.QW_F32)) == L.QW_ERR_DTYPE
    assert lib.qw_attention_decode_paged(*pd(100, 4, 400, fake, L.QW_BF16)) == L.QW_ERR_SHAPE
    assert lib.qw_attention_decode_paged(*pd(256, 4, 1025, fake, L.QW_BF16)) == L.QW_ERR_SHAPE
    assert lib.qw_attention_decode_paged(*pd(256, 4, 1024, None, L.QW_BF16)) == L.QW_ERR_INVALID_ARG
    assert lib.qw_attention_decode_paged(*pd(256, 4, 1024, fake, L.QW_BF16)) == L.QW_ERR_WORKSPACE
    pp = lambda bs, table, hd: (fake, fake, fake, 100, fake, fake, table, 4, bs, 2, 64, 16, 8, hd, 0.1, fake,  # noqa: E731
                                L.QW_BF16, None)
    assert lib.qw_attention_prefill_paged(*pp(64, fake, 128)) == L.QW_ERR_SHAPE      # block size below the 128-key tile
    assert lib.qw_attention_prefill_paged(*pp(256, fake, 64)) == L.QW_ERR_SHAPE
    assert lib.qw_attention_prefill_paged(*pp(256, None, 128)) == L.QW_ERR_INVALID_ARG
    # decode attention with the QK-norm + RoPE + KV store folded in: bf16, head_dim 128, tp | heads
    rope = lambda hd, nh, nkv, tp, dt, flags, ws, wsb: (fake, nh, nkv, hd, tp, fake, fake, 4096, fake, fake, 1e-6,  # noqa: E731
                                                        fake, fake, fake, 100, None, fake, fake, 8, 2048, 0.1, fake,
                                                        ws, wsb, dt, flags, None)
    assert lib.qw_attention_decode_rope(*rope(128, 16, 8, 2, L.QW_F32, 0, None, 0)) == L.QW_ERR_DTYPE
    assert lib.qw_attention_decode_rope(*rope(64, 16, 8, 2, L.QW_BF16, 0, None, 0)) == L.QW_ERR_SHAPE
    assert lib.qw_attention_decode_rope(*rope(128, 16, 8, 3, L.QW_BF16, 0, None, 0)) == L.QW_ERR_SHAPE
    assert lib.qw_attention_decode_rope(*rope(128, 12, 4, 2, L.QW_BF16, 0, None, 0)) == L.QW_ERR_SHAPE
    assert lib.qw_attention_decode_rope(*rope(128, 16, 8, 2, L.QW_BF16, 4, None, 0)) == L.QW_ERR_INVALID_ARG
    assert lib.qw_attention_decode_rope(*rope(128, 16, 8, 2, L.QW_BF16, 0, None, 0)) == L.QW_ERR_WORKSPACE
    # one-kernel decode step: at most 16 tokens, head_dim 128, group size 1/2/4/8
    args = lambda B, hd, nh, nkv: (fake, 28, fake, fake, fake, fake, fake, B, 100, 1024, nh, nkv, hd, 3072, 2, fake,  # noqa: E731
                                   4096, 100, 1e-6, 0.1, fake, fake, None, fake, 1 << 30, None)
    assert lib.qw_decode_layers(*args(17, 128, 16, 8)) == L.QW_ERR_SHAPE
    assert lib.qw_decode_layers(*args(8, 64, 16, 8)) == L.QW_ERR_SHAPE
    assert lib.qw_decode_layers(*args(8, 128, 12, 4)) == L.QW_ERR_SHAPE
    assert lib.qw_decode_layers_workspace_size(28, 17, 1024, 16, 8, 128, 3072, 2, 2048) == 0
    # fused add + RMSNorm + GEMM: at most 16 tokens, residual_out distinct from x
    assert lib.qw_add_rmsnorm_gemm(fake, None, None, fake, 1e-6, fake, fake, 17, 64, 64, 1, 0, L.QW_BF16,
                                   None) == L.QW_ERR_SHAPE
    assert lib.qw_add_rmsnorm_gemm(fake, fake, fake, fake, 1e-6, fake, fake, 4, 64, 64, 1, 0, L.QW_BF16,
                                   None) == L.QW_ERR_INVALID_ARG
    # 16 tokens of K = 8192 normed rows do not fit in shared memory
    assert lib.qw_add_rmsnorm_gemm(fake, None, None, fake, 1e-6, fake, fake, 16, 64, 8192, 1, 0, L.QW_BF16,
                                   None) == L.QW_ERR_SHAPE
    # QKV GEMM with the QK-norm / RoPE / KV-store epilogue: bf16, head_dim 128, an even number of heads per shard
    qg = lambda nh, nkv, hd, tp, dt: (fake, fake, 300, 1024, nh, nkv, hd, tp, fake, fake, 4096, fake, fake, 1e-6,  # noqa: E731
                                      fake, fake, fake, 100, fake, None, dt, None)
    assert lib.qw_qkv_gemm_norm_rope_store_kv(*qg(16, 8, 128, 2, L.QW_F32)) == L.QW_ERR_DTYPE
    assert lib.qw_qkv_gemm_norm_rope_store_kv(*qg(16, 8, 64, 2, L.QW_BF16)) == L.QW_ERR_SHAPE
    assert lib.qw_qkv_gemm_norm_rope_store_kv(*qg(16, 8, 128, 3, L.QW_BF16)) == L.QW_ERR_SHAPE
    assert lib.qw_qkv_gemm_norm_rope_store_kv(*qg(5, 1, 128, 1, L.QW_BF16)) == L.QW_ERR_SHAPE   # 7 heads: odd
    # row-parallel GEMM + residual add + RMSNorm: bf16, N a multiple of 256 up to 2048, y not the residual
    ga = lambda N, K, tp, y, dt: (fake, fake, 300, N, K, tp, C.c_void_p(32), fake, 1e-6, y, dt, None)  # noqa: E731
    assert lib.qw_gemm_add_rmsnorm(*ga(1024, 2048, 2, fake, L.QW_F32)) == L.QW_ERR_DTYPE
    assert lib.qw_gemm_add_rmsnorm(*ga(1000, 2048, 2, fake, L.QW_BF16)) == L.QW_ERR_SHAPE
    assert lib.qw_gemm_add_rmsnorm(*ga(4096, 2048, 2, fake, L.QW_BF16)) == L.QW_ERR_SHAPE
    assert lib.qw_gemm_add_rmsnorm(*ga(1024, 2052, 2, fake, L.QW_BF16)) == L.QW_ERR_SHAPE
    assert lib.qw_gemm_add_rmsnorm(*ga(1024, 2048, 2, C.c_void_p(32), L.QW_BF16)) == L.QW_ERR_INVALID_ARG
    # sampler: bf16 only, V a multiple of 8, a workspace of the queried size
    assert lib.qw_sample(fake, 4, 151936, fake, fake, fake, fake, fake, 1 << 30, L.QW_F32, None) == L.QW_ERR_DTYPE
    assert lib.qw_sample(fake, 4, 100, fake, fake, fake, fake, fake, 1 << 30, L.QW_BF16, None) == L.QW_ERR_INVALID_ARG
    assert lib.qw_sample(fake, 4, 151936, fake, fake, fake, fake, None, 0, L.QW_BF16, None) == L.QW_ERR_WORKSPACE
    need = lib.qw_sample_workspace_size(4, 151936)
    assert need >= 64 * 1024 + 4 * 65536 * 4
    assert lib.qw_sample(fake, 4, 151936, fake, fake, fake, fake, fake, need - 1, L.QW_BF16, None) == L.QW_ERR_WORKSPACE
    assert lib.qw_sample(None, 0, 151936, None, None, None, None, None, 0, L.QW_BF16, None) == L.QW_OK
    # lm_head: V not divisible by tp
    assert lib.qw_lm_head(fake, 4, None, 4, fake, 10, 64, 4, fake, None, None, 0, L.QW_BF16,
                          None) == L.QW_ERR_SHAPE


@pytest.mark.parametrize("max_pos,d,theta", [(64, 16, 1e6), (2200, 128, 1e6), (300, 8, 1e4)])
def test_rope_table_equals_oracle(lib, max_pos, d, theta):
    t = L.rope_cos_sin_table(max_pos, d, theta).double().numpy()
    cos_t, sin_t = O.rope_cos_sin(max_pos, d, theta)
    assert np.array_equal(t[:, : d // 2], cos_t)
    assert np.array_equal(t[:, d // 2:], sin_t)


def test_workspace_sizes(lib):
    # GEMMs keep split-K partials on chip: no workspace at any size
    assert L.gemm_workspace_size(2048, 4096, 1024, 2, L.QW_GEMM_COLUMN, 0, torch.bfloat16) == 0
    assert L.gemm_workspace_size(8, 1024, 3072, 2, L.QW_GEMM_ROW_REDUCE, 0, torch.bfloat16) == 0
    assert L.lm_head_workspace_size(8, 151936, 1024, 2, torch.bfloat16) >= 64 * 1024 + 8 * 1024 * 2
    assert L.attention_decode_workspace_size(64, 2048, 16, 128) > 0
    # max_context 0 (every sequence empty) still plans one key tile per pair
    assert L.attention_decode_workspace_size(8, 0, 16, 128) > 0
    assert L.attention_decode_workspace_size(8, -1, 16, 128) == 0
