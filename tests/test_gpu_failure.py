"""Failure detection without a GPU fault (needs a GB300).

Every wait in the tensor-core kernels is bounded.  A wait that runs out
records a code in a device error word, and the kernel returns; the host then
reports QW_ERR_TIMEOUT from qw_device_error.  This test makes one such wait
run out on purpose (an mbarrier that nothing completes), then checks three
things: the status arrives, it clears once read, and the context still runs
kernels afterwards.  Nothing traps, faults or hangs: the wait gives up after
2 s.
"""
import pytest
import torch

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


def test_bounded_wait_runs_out_and_is_reported(L):
    L.device_error()                      # a clean start
    L.selftest_wait_timeout()
    with pytest.raises(L.QwError) as e:
        L.device_error()
    assert e.value.code == L.QW_ERR_TIMEOUT
    assert "gemm 0x100" in str(e.value)
    L.device_error()                      # reading the words cleared them
    # the context still runs kernels: an argmax over distinct values
    g = torch.Generator().manual_seed(0)
    logits = torch.stack([torch.randperm(64, generator=g) for _ in range(3)]).to(torch.bfloat16).cuda()
    out = torch.empty(3, dtype=torch.int64, device="cuda")
    L.argmax(logits, out)
    L.device_error()
    assert torch.equal(out.cpu(), logits.float().argmax(dim=1).cpu())
