"""Seeded synthetic inputs shared by the CUDA path and the CPU oracle.

This module holds no arithmetic of the Qwen3 forward pass.  It only turns a
(seed, stream name, element index) triple into reproducible bits, and knows
the workload shapes (model sizes, batch layout, slot layout).

Every value is produced with integer operations plus at most one IEEE
correctly-rounded fp32 multiply, so the same call yields bit-identical
tensors on the CPU and on a GPU.  That is why the "normal" draws are an
Irwin-Hall sum of four 16-bit uniforms (mean 0, variance matched to sigma,
support +-3.46 sigma) rather than Box-Muller: no transcendental function
whose last bit could differ between devices is involved.

Hash: MurmurHash3's 32-bit finaliser ``fmix32`` (A. Appleby, public domain),
evaluated on int64 tensors with the 32x32-bit products split into 16-bit
halves so that no intermediate exceeds 2**49.
"""
from __future__ import annotations

import math
import zlib

import torch

from .workloads import (  # noqa: F401  (re-exported)
    ModelShape,
    PrefillBatch,
    DecodeBatch,
    WORKLOADS,
    workload,
    prefill_batch,
    decode_batch,
    decode_context_lens,
    kv_history,
    embed_ids,
    checkpoint_tensor,
    weight_names,
    weight_shape,
    QWEN3_0_6B,
    TINY,
)

MASK32 = 0xFFFFFFFF
_CHUNK = 1 << 24


def _fmix32_py(h: int) -> int:
    h &= MASK32
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & MASK32
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & MASK32
    h ^= h >> 16
    return h


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & MASK32


def _fmix32(h: torch.Tensor) -> torch.Tensor:
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    h = h ^ (h >> 16)
    return h


def stream_key(seed: int, name: str) -> int:
    """32-bit key of one named random stream under one seed."""
    return _fmix32_py((seed * 0x9E3779B9) ^ _fmix32_py(zlib.crc32(name.encode())))


def hash_words(seed: int, name: str, idx: torch.Tensor):
    """Two independent 32-bit words (as int64 tensors) for each element index."""
    key = stream_key(seed, name)
    lo = idx & MASK32
    hi = idx >> 32
    a = _fmix32(lo ^ key)
    a = _fmix32(a ^ hi ^ 0x9E3779B9)
    b = _fmix32(a ^ 0x7F4A7C15)
    return a, b


_IH_STD = math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0)
_DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32, "fp32": torch.float32,
           torch.bfloat16: torch.bfloat16, torch.float32: torch.float32}


def _as_dtype(dtype):
    return _DTYPES[dtype]


def normal_at(seed: int, name: str, idx: torch.Tensor, sigma: float, dtype) -> torch.Tensor:
    """Approximately N(0, sigma^2) values at the given flat element indices."""
    a, b = hash_words(seed, name, idx)
    s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16)
    z = (s - 131070).to(torch.float32)
    c = torch.tensor(sigma / _IH_STD, dtype=torch.float32, device=idx.device)
    return (z * c).to(_as_dtype(dtype))


def normal(seed: int, name: str, shape, sigma: float, dtype, device="cpu") -> torch.Tensor:
    """A tensor of the given shape filled with seeded approximately-normal values."""
    shape = tuple(int(s) for s in shape)
    n = math.prod(shape)
    out = torch.empty(n, dtype=_as_dtype(dtype), device=device)
    for s0 in range(0, n, _CHUNK):
        s1 = min(n, s0 + _CHUNK)
        idx = torch.arange(s0, s1, dtype=torch.int64, device=device)
        out[s0:s1] = normal_at(seed, name, idx, sigma, dtype)
    return out.view(shape)


def uniform_int(seed: int, name: str, shape, low: int, high: int, device="cpu") -> torch.Tensor:
    """int64 tensor of values in [low, high)."""
    shape = tuple(int(s) for s in shape)
    n = math.prod(shape)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    a, _ = hash_words(seed, name, idx)
    return (a % (high - low) + low).view(shape)


def uniform01(seed: int, name: str, shape, device="cpu") -> torch.Tensor:
    """float32 values in the open interval (0, 1): (2 k + 1) * 2^-24 for k the top 23
    bits of a hash word, exact in fp32 (an integer below 2^24 and a power-of-two multiply)."""
    shape = tuple(int(s) for s in shape)
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s0 in range(0, n, _CHUNK):
        s1 = min(n, s0 + _CHUNK)
        idx = torch.arange(s0, s1, dtype=torch.int64, device=device)
        a, _ = hash_words(seed, name, idx)
        out[s0:s1] = ((a >> 9) * 2 + 1).to(torch.float32) * (2.0 ** -24)
    return out.view(shape)


def uniform_word(seed: int, name: str, shape, device="cpu") -> torch.Tensor:
    """Raw 32-bit words (int64 tensor in [0, 2**32))."""
    shape = tuple(int(s) for s in shape)
    n = math.prod(shape)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    _, b = hash_words(seed, name, idx)
    return b.view(shape)
