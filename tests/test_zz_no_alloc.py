"""The decode-attention entry point that needs no device allocation from its caller.

Some callers cannot allocate device memory: a plugin that its host framework
gives only input and output pointers (the framework owns the allocator), or a
serving loop that fixes all device memory at start-up.  qw_attention_decode_static
serves them by keeping its split-KV scratch in a fixed array inside the
library.  This test calls it through the C ABI twice in a row, with different
inputs each time (so stale scratch from the first call would show), and checks
each result against qw_attention_decode with a caller-provided workspace: the
two run the same kernels with the same partition and merge order, so the
results must be identical bit for bit.  It also checks that a
batch too big for the fixed array is refused before anything runs.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_transformer_forward_gb300 import build
    build.build()
    from qwen3_transformer_forward_gb300 import _lib
    _lib.load()
    return _lib


def _case(name, ctx, dtype="bf16"):
    nh, nkv, hd = 16, 8, 128
    B = len(ctx)
    cap = [c + 1 for c in ctx]
    base = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int32)
    S = int(sum(cap))
    kc = si.normal(0, f"{name}.k", (S, nkv, hd), 1.0, dtype).cuda()
    vc = si.normal(0, f"{name}.v", (S, nkv, hd), 1.0, dtype).cuda()
    q = si.normal(0, f"{name}.q", (B, nh, hd), 1.0, dtype).cuda()
    cl = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    sb = torch.tensor(base, device="cuda")
    return q, kc, vc, cl, sb, max(ctx), nh, nkv, hd


def test_static_scratch_matches_workspace_version_twice(L):
    for name, ctx in (("noalloc.a", [2176] * 8), ("noalloc.b", [1, 700, 65, 2048, 3000])):
        q, kc, vc, cl, sb, mc, nh, nkv, hd = _case(name, ctx)
        assert 0 < L.attention_decode_workspace_size(len(ctx), mc, nh, hd) <= L.attention_decode_static_scratch_bytes()
        ref = torch.empty(len(ctx), nh * hd, dtype=q.dtype, device="cuda")
        ws = torch.zeros(L.attention_decode_workspace_size(len(ctx), mc, nh, hd), dtype=torch.uint8, device="cuda")
        L.attention_decode(q, kc, vc, cl, sb, mc, nh, nkv, hd, hd ** -0.5, ref, ws)
        got = torch.empty_like(ref)
        L.attention_decode_static(q, kc, vc, cl, sb, mc, nh, nkv, hd, hd ** -0.5, got)
        torch.cuda.synchronize()
        L.device_error()
        # the same kernels with the same partition and a fixed merge order: bit for bit
        assert torch.equal(got, ref), f"{name}: static scratch result differs from the workspace result"
        assert not torch.isnan(got.float()).any()


def test_static_scratch_rejects_batches_beyond_its_size(L):
    from qwen3_transformer_forward_gb300._lib import QW_ERR_WORKSPACE, QwError
    # 256 sequences of 16 q heads over 8 kv heads: one (m, l, o) slot per
    # (CTA, pair) plus one per pair, (8 x SMs + 256 x 16) x (128 + 2) floats,
    # is over 2 MiB
    B, mc, nh, nkv, hd = 256, 64, 16, 8, 128
    assert L.attention_decode_workspace_size(B, mc, nh, hd) > L.attention_decode_static_scratch_bytes()
    q = torch.zeros(B, nh, hd, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(8, nkv, hd, dtype=torch.bfloat16, device="cuda")
    cl = torch.ones(B, dtype=torch.int32, device="cuda")
    sb = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.full((B, nh * hd), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(QwError) as e:
        L.attention_decode_static(q, kv, kv, cl, sb, mc, nh, nkv, hd, hd ** -0.5, out)
    assert e.value.code == QW_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)            # nothing ran
