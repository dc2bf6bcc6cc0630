"""Workload shapes and seeded batch layouts (no arithmetic of the model).

Five workloads, all drawn with seed 0:

* ``tiny_fp32_prefill`` - 1-layer Qwen3-style decoder in fp32: vocab 512,
  hidden 64, 4 q / 2 kv heads of 16, intermediate 128, two emulated shards,
  prefill of 2 sequences x 16 tokens.
* ``embed_lm_head`` - the vocab-sharded embedding and lm_head only, bf16,
  vocab 151936 x 1024, shards 1/2/4, 8192 ids (5 % on shard boundaries) and
  8192 hidden vectors N(0,1).
* ``layer_prefill`` - one Qwen3-0.6B-shaped decoder layer, bf16, two shards,
  prefill 4 x 512 tokens with N(0,1) hidden inputs.
* ``model_decode`` - the 28-layer Qwen3-0.6B shape, one decode step for 64
  sequences whose context lengths are uniform in [256, 2048]; the cache
  history is seeded N(0,1).
* ``model_prefill_decode`` - the same model with two shards: prefill
  8 x 2048 tokens, then 128 greedy decode steps.

KV-cache addressing is contiguous per sequence: sequence b owns slots
[seq_base[b], seq_base[b] + capacity[b]) and the token at position p is
stored in slot seq_base[b] + p.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch


@dataclass(frozen=True)
class ModelShape:
    vocab: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    n_layers: int
    tp: int = 1
    dtype: str = "bf16"
    eps: float = 1e-6
    rope_theta: float = 1e6
    max_position: int = 40960
    weight_sigma: float = 0.02
    # 0.0 means every RMSNorm gamma is exactly 1.0 (the workloads' setting);
    # tests use > 0 to draw gamma = 1 + N(0, sigma) so that gamma matters.
    gamma_sigma: float = 0.0

    @property
    def q_size(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_size(self) -> int:
        return self.n_kv_heads * self.head_dim

    def replace(self, **kw) -> "ModelShape":
        return dataclasses.replace(self, **kw)


QWEN3_0_6B = ModelShape(vocab=151936, hidden=1024, n_heads=16, n_kv_heads=8, head_dim=128,
                        intermediate=3072, n_layers=28)
TINY = ModelShape(vocab=512, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, intermediate=128,
                  n_layers=1, tp=2, dtype="f32", max_position=128)


@dataclass(frozen=True)
class Workload:
    name: str
    model: ModelShape
    seq_lens: Sequence[int] = ()
    decode_steps: int = 0
    batch: int = 0
    ctx_low: int = 0
    ctx_high: int = 0
    tps: Sequence[int] = (1,)
    n_tokens: int = 0
    boundary_fraction: float = 0.0
    seed: int = 0


WORKLOADS = {
    "tiny_fp32_prefill": Workload("tiny_fp32_prefill", TINY, seq_lens=(16, 16)),
    "embed_lm_head": Workload("embed_lm_head", QWEN3_0_6B.replace(n_layers=0), tps=(1, 2, 4),
                              n_tokens=8192, boundary_fraction=0.05),
    "layer_prefill": Workload("layer_prefill", QWEN3_0_6B.replace(n_layers=1, tp=2),
                              seq_lens=(512,) * 4),
    "model_decode": Workload("model_decode", QWEN3_0_6B, batch=64, ctx_low=256, ctx_high=2048),
    "model_prefill_decode": Workload("model_prefill_decode", QWEN3_0_6B.replace(tp=2),
                                     seq_lens=(2048,) * 8, decode_steps=128),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


# ----------------------------------------------------------------------------
# weights (checkpoint form: separate q/k/v and gate/up, unsharded)
# ----------------------------------------------------------------------------

def weight_names(layer: int):
    p = f"layer{layer}."
    return [p + n for n in ("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj")]


def weight_shape(m: ModelShape, name: str):
    base = name.split(".")[-1]
    return {
        "embed_tokens": (m.vocab, m.hidden),
        "q_proj": (m.q_size, m.hidden),
        "k_proj": (m.kv_size, m.hidden),
        "v_proj": (m.kv_size, m.hidden),
        "o_proj": (m.hidden, m.q_size),
        "gate_proj": (m.intermediate, m.hidden),
        "up_proj": (m.intermediate, m.hidden),
        "down_proj": (m.hidden, m.intermediate),
        "input_layernorm": (m.hidden,),
        "post_attention_layernorm": (m.hidden,),
        "q_norm": (m.head_dim,),
        "k_norm": (m.head_dim,),
        "norm": (m.hidden,),
    }[base]


def checkpoint_tensor(m: ModelShape, name: str, seed: int = 0, device="cpu") -> torch.Tensor:
    """One unsharded parameter, as a checkpoint would hold it."""
    from . import normal
    shape = weight_shape(m, name)
    base = name.split(".")[-1]
    if base in ("input_layernorm", "post_attention_layernorm", "q_norm", "k_norm", "norm"):
        if m.gamma_sigma == 0.0:
            return torch.ones(shape, dtype=_dt(m.dtype), device=device)
        g = normal(seed, name, shape, m.gamma_sigma, "f32", device) + 1.0
        return g.to(_dt(m.dtype))
    return normal(seed, name, shape, m.weight_sigma, m.dtype, device)


def _dt(d):
    return torch.bfloat16 if d == "bf16" else torch.float32


# ----------------------------------------------------------------------------
# batches
# ----------------------------------------------------------------------------

@dataclass
class PrefillBatch:
    seq_lens: List[int]
    ids: torch.Tensor            # int64 [T]
    positions: torch.Tensor      # int64 [T]
    cu_seqlens: torch.Tensor     # int32 [S+1]
    slot_mapping: torch.Tensor   # int64 [T]
    seq_base: torch.Tensor       # int32 [S]
    capacity: List[int]
    num_slots: int
    last_idx: torch.Tensor       # int32 [S]  (cu_seqlens[1:] - 1)


@dataclass
class DecodeBatch:
    ids: torch.Tensor            # int64 [B]
    positions: torch.Tensor      # int64 [B]   (context_lens - 1)
    context_lens: torch.Tensor   # int32 [B]   (keys visible, including this token)
    slot_mapping: torch.Tensor   # int64 [B]
    seq_base: torch.Tensor       # int32 [B]
    num_slots: int


def prefill_batch(m: ModelShape, seq_lens: Sequence[int], seed: int = 0, extra_capacity: int = 0,
                  stream: str = "prefill.ids") -> PrefillBatch:
    from . import uniform_int
    seq_lens = [int(s) for s in seq_lens]
    T = sum(seq_lens)
    ids = uniform_int(seed, stream, (T,), 0, m.vocab)
    positions = torch.cat([torch.arange(L, dtype=torch.int64) for L in seq_lens]) if T else \
        torch.zeros(0, dtype=torch.int64)
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(seq_lens, dtype=torch.int64), 0).to(torch.int32)
    capacity = [L + extra_capacity for L in seq_lens]
    base = [0]
    for c in capacity[:-1]:
        base.append(base[-1] + c)
    seq_base = torch.tensor(base, dtype=torch.int32)
    slots = torch.cat([torch.arange(L, dtype=torch.int64) + base[b] for b, L in enumerate(seq_lens)]) \
        if T else torch.zeros(0, dtype=torch.int64)
    return PrefillBatch(seq_lens, ids, positions, cu, slots, seq_base, capacity, sum(capacity),
                        (cu[1:] - 1).to(torch.int32))


def decode_context_lens(seed: int, batch: int, low: int, high: int) -> List[int]:
    """Context lengths (including the token being decoded), uniform in [low, high]."""
    from . import uniform_int
    return [int(v) for v in uniform_int(seed, "decode.context_lens", (batch,), low, high + 1)]


def decode_batch(m: ModelShape, context_lens: Sequence[int], seed: int = 0,
                 capacity: Optional[Sequence[int]] = None, stream: str = "decode.ids") -> DecodeBatch:
    from . import uniform_int
    context_lens = [int(c) for c in context_lens]
    B = len(context_lens)
    capacity = list(capacity) if capacity is not None else list(context_lens)
    base = [0]
    for c in capacity[:-1]:
        base.append(base[-1] + c)
    ids = uniform_int(seed, stream, (B,), 0, m.vocab)
    pos = torch.tensor([c - 1 for c in context_lens], dtype=torch.int64)
    slots = torch.tensor([base[b] + context_lens[b] - 1 for b in range(B)], dtype=torch.int64)
    return DecodeBatch(ids, pos, torch.tensor(context_lens, dtype=torch.int32), slots,
                       torch.tensor(base, dtype=torch.int32), sum(capacity))


def kv_history(m: ModelShape, layer: int, which: str, slots: torch.Tensor, seed: int = 0) -> torch.Tensor:
    """Synthetic cache history: N(0,1) values of [len(slots), n_kv_heads, head_dim] at those slots."""
    from . import normal_at
    D = m.kv_size
    idx = (slots.to(torch.int64)[:, None] * D + torch.arange(D, dtype=torch.int64, device=slots.device)[None, :])
    v = normal_at(seed, f"layer{layer}.{which}_cache_history", idx.reshape(-1), 1.0, m.dtype)
    return v.view(len(slots), m.n_kv_heads, m.head_dim)


def embed_ids(m: ModelShape, n: int, boundary_fraction: float, seed: int = 0) -> torch.Tensor:
    """Token ids uniform over the vocab, with a fraction replaced by shard-boundary ids."""
    from . import uniform_int, uniform_word
    ids = uniform_int(seed, "embed.ids", (n,), 0, m.vocab)
    if boundary_fraction > 0:
        V = m.vocab
        bnd = sorted({0, V - 1} | {k * V // 4 - 1 for k in (1, 2, 3)} | {k * V // 4 for k in (1, 2, 3)})
        bnd_t = torch.tensor(bnd, dtype=torch.int64)
        w = uniform_word(seed, "embed.boundary_pick", (n,))
        pick = w < int(boundary_fraction * 2 ** 32)
        which = uniform_int(seed, "embed.boundary_which", (n,), 0, len(bnd))
        ids = torch.where(pick, bnd_t[which], ids)
    return ids
