"""Runs one libqw kernel on a fixed, seeded problem, for profiling (e.g. with ncu).

    python -m qwen3_transformer_forward_gb300.kernel_cases <case> [--reps N]

Cases (sizes of the Qwen3-0.6B decode and prefill steps):
  attn_decode_b64    decode attention, 64 sequences x 1152 keys, 16 q / 8 kv heads of 128
  attn_decode_b8     decode attention, 8 sequences x 2176 keys
  gemm_down_m8       down_proj with 8 tokens: [8, 3072] x [2, 1024, 1536]^T, row split
  gemm_qkv_m8        QKV with 8 tokens: [8, 1024] x [4096, 1024]^T
  gemm_gate_up_m8    gate_up + SiluAndMul with 8 tokens
  gemm_gate_up_prefill  gate_up + SiluAndMul with 16384 tokens
  attn_prefill_8x2048   causal prefill attention, 8 sequences x 2048
  qkv_rope_prefill   QK-norm + RoPE + KV store for 16384 tokens
"""
from __future__ import annotations

import argparse

import torch

from . import _lib as L
from . import build


def _rand(shape, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(0)
    return (torch.randn(*shape, device="cuda", generator=g) * scale).to(torch.bfloat16)


def make_case(name):
    H, I, nh, nkv, hd = 1024, 3072, 16, 8, 128
    if name.startswith("attn_decode"):
        B, ctx, cap = (64, 1152, 2048) if name.endswith("b64") else (8, 2176, 2176)
        kc, vc = _rand((B * cap, nkv, hd)), _rand((B * cap, nkv, hd))
        q, out = _rand((B, nh, hd)), torch.empty(B, nh * hd, dtype=torch.bfloat16, device="cuda")
        cl = torch.full((B,), ctx, dtype=torch.int32, device="cuda")
        sb = torch.arange(B, dtype=torch.int32, device="cuda") * cap
        ws = torch.zeros(L.attention_decode_workspace_size(B, cap, nh, hd) + 16, dtype=torch.uint8, device="cuda")
        return lambda: L.attention_decode(q, kc, vc, cl, sb, cap, nh, nkv, hd, hd ** -0.5, out, ws)
    if name == "gemm_down_m8":
        a, w, c = _rand((8, I)), _rand((2, H, I // 2), 0.02), torch.empty(8, H, dtype=torch.bfloat16, device="cuda")
        return lambda: L.gemm(a, w, c, H, 2, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_NONE)
    if name == "gemm_qkv_m8":
        a, w, c = _rand((8, H)), _rand((4096, H), 0.02), torch.empty(8, 4096, dtype=torch.bfloat16, device="cuda")
        return lambda: L.gemm(a, w, c, 4096, 2, L.QW_GEMM_COLUMN, L.QW_EPI_NONE)
    if name in ("gemm_gate_up_m8", "gemm_gate_up_prefill"):
        M = 8 if name.endswith("m8") else 16384
        a, w, c = _rand((M, H)), _rand((2 * I, H), 0.02), torch.empty(M, I, dtype=torch.bfloat16, device="cuda")
        return lambda: L.gemm(a, w, c, 2 * I, 2, L.QW_GEMM_COLUMN, L.QW_EPI_SILU_MUL)
    if name == "attn_prefill_8x2048":
        T = 8 * 2048
        q, k, v = _rand((T, nh, hd)), _rand((T, nkv, hd)), _rand((T, nkv, hd))
        cu = torch.arange(0, T + 1, 2048, dtype=torch.int32, device="cuda")
        out = torch.empty(T, nh * hd, dtype=torch.bfloat16, device="cuda")
        return lambda: L.attention_prefill(q, k, v, cu, cu, None, 2048, nh, nkv, hd, hd ** -0.5, out)
    if name == "qkv_rope_prefill":
        T = 16384
        qkv = _rand((T, (nh + 2 * nkv) * hd))
        pos = torch.arange(T, device="cuda", dtype=torch.int64) % 2048
        cs = L.rope_cos_sin_table(4096, hd, 1e6).cuda()
        g = torch.ones(hd, dtype=torch.bfloat16, device="cuda")
        kc, vc = torch.zeros(T, nkv, hd, dtype=torch.bfloat16, device="cuda"), torch.zeros(
            T, nkv, hd, dtype=torch.bfloat16, device="cuda")
        slots = torch.arange(T, device="cuda", dtype=torch.int64)
        qo = torch.empty(T, nh * hd, dtype=torch.bfloat16, device="cuda")
        return lambda: L.qkv_norm_rope_store_kv(qkv, nh, nkv, hd, 2, pos, cs, g, g, 1e-6, slots, kc, vc, qo)
    raise SystemExit(f"unknown case {name}")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)
    build.build()
    L.load()
    fn = make_case(args.case)
    for _ in range(args.reps):
        fn()
    torch.cuda.synchronize()
    L.device_error()


if __name__ == "__main__":
    main()
