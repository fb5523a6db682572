"""conv_bwd_filter_noalloc: the weight gradient for callers that cannot
allocate device memory (hosts that own every byte but the inputs and outputs,
code that must not allocate mid-step).  Its split-K partials live in the
library's fixed scratch array instead of a caller workspace.

Each case runs two calls in a row through the C ABI and checks, per call:
  - the oracle's fp64 result on the same inputs, element by element, within
    the normalised-error tolerance the other GPU tests use;
  - the existing conv_bwd_filter entry point's result, within the same
    tolerance (both are normalised by the oracle's sum of |terms|);
and that the two calls give bit-identical outputs (the shared array keeps
the previous call's contents; nothing of it may leak into the result).
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
from implicit_gemm_conv2d_gb300 import binding

from .gpu_cases import L1, L2, TOL, Case, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layer,B", [("L1", 1024), ("L2", 1024), ("L1", 7)])
def test_noalloc_matches_oracle_and_bwd_filter(layer, B, dtype):
    c = Case(B, **(L1 if layer == "L1" else L2), dtype=dtype)
    y = c.gpu_fwd()
    existing = c.gpu_wgrad(y)  # the existing entry point, caller-provided workspace
    torch.cuda.synchronize()
    existing_np = to_np(existing)
    ref, den = c.ref_wgrad(to_np(y))
    outs = []
    for call in range(2):
        dw = torch.full_like(existing, float("nan"))
        binding.conv_bwd_filter_noalloc(c.desc, c.x, c.dy, y if c.relu else None, dw)
        torch.cuda.synchronize()
        out = to_np(dw)
        assert np.isfinite(out).all(), f"call {call}: output not fully written"
        err = oracle.normalised_error(out, ref, den)
        assert err <= TOL[dtype], f"call {call}: normalised error vs the oracle {err:.3e} > {TOL[dtype]}"
        err = oracle.normalised_error(out, existing_np, den)
        assert err <= TOL[dtype], f"call {call}: normalised difference vs conv_bwd_filter {err:.3e}"
        outs.append(dw)
    view = torch.int16 if dtype == "bf16" else torch.int32
    assert torch.equal(outs[0].view(view), outs[1].view(view)), "two calls in a row differ"


def test_noalloc_rejects_partials_beyond_the_scratch():
    # One split of OC x round_up(IC*K*K, 4) fp32 partials would need 26 MB > 16 MiB.
    d = binding.make_desc(2, 512, 512, 5, 5, 5, 1, 0, torch.float32)
    x = torch.zeros((2, 512, 5, 5), device="cuda")
    dy = torch.zeros((2, 512, 1, 1), device="cuda")
    dw = torch.zeros((512, 512, 5, 5), device="cuda")
    with pytest.raises(binding.ConvError) as ei:
        binding.conv_bwd_filter_noalloc(d, x, dy, None, dw)
    assert ei.value.status == -3


def test_noalloc_empty_batch_writes_zeros():
    d = binding.make_desc(0, 59, 128, 11, 15, 5, 3, 1, torch.float32)
    dw = torch.full((128, 59, 5, 5), 3.0, device="cuda")
    e = torch.empty(0, device="cuda")
    binding.conv_bwd_filter_noalloc(d, e, e, e, dw)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw).item() == 0
