"""The tensor-core kernels' bounded waits, timed out on purpose without a fault or a hang:
a one-CTA kernel waits on an mbarrier that nothing completes, gives up after its short
limit, sets its bit in the status word and returns; the context stays usable (a layer
computed next still matches the oracle) and the bit clears on reset."""
import pytest
import torch

from implicit_gemm_conv2d_gb300 import binding

from .gpu_cases import L1, Case, check, to_np

pytestmark = pytest.mark.gpu


def test_wait_timeout_sets_status_and_context_survives():
    binding.conv_device_status(reset=True)
    assert binding.conv_device_status() == 0
    binding.conv_wait_selftest(1000)
    torch.cuda.synchronize()
    st = binding.conv_device_status()
    assert st & binding.STATUS_WAIT_SELFTEST
    assert st & ~binding.STATUS_WAIT_SELFTEST == 0   # no real kernel timed out
    c = Case(37, **L1, dtype="f32")
    y = c.gpu_fwd()
    torch.cuda.synchronize()
    ref, den = c.ref_fwd()
    check(to_np(y), ref, den, "f32", "fwd after the wait self-test")
    binding.conv_device_status(reset=True)
    assert binding.conv_device_status() == 0
