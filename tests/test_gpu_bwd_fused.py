"""conv_bwd: the whole backward of the layer -- d_input, wgrad and optionally the bias
gradient -- in one launch (PufferLib PR #522 times "backward" as wgrad plus d_input).  Checked
through the C ABI: dx bit for bit against conv_bwd_data; dw and db against the fp64 oracle and
dw against conv_bwd_filter within the tolerance (conv_bwd splits the batch into fewer ranges);
run to run bit identity; the two-call path, both where the batch is large enough for the
standalone kernels (layer 1 from 4096 samples) and when a family other than the tensor cores is
forced; an undersized workspace rejected."""
import numpy as np
import pytest
import torch

import oracle
from implicit_gemm_conv2d_gb300 import binding

from .gpu_cases import L1, L2, TOL, Case, check, to_np

pytestmark = pytest.mark.gpu

SHAPES = {"L1": L1, "L2": L2, "odd": dict(IC=3, OC=5, H=7, W=9, K=2, S=2, relu=True),
          "k_eq_input": dict(IC=7, OC=33, H=5, W=5, K=5, S=2, relu=True),
          "p1_relu_oc64": dict(IC=16, OC=64, H=4, W=4, K=3, S=2, relu=True)}


@pytest.fixture(autouse=True)
def _restore_algo():
    yield
    for op in range(4):
        binding.conv_set_algo(op, binding.ALGO_AUTO)


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def run_bwd(c: Case, y, with_bias):
    dx = torch.full((c.B, c.IC, c.H, c.W), float("nan"), dtype=c.x.dtype, device="cuda")
    dw = torch.full((c.OC, c.IC, c.K, c.K), float("nan"), dtype=c.x.dtype, device="cuda")
    db = torch.full((c.OC,), float("nan"), dtype=c.x.dtype, device="cuda") if with_bias else None
    ws = torch.empty(max(16, binding.conv_bwd_workspace_size(c.desc)), dtype=torch.uint8, device="cuda")
    binding.conv_bwd(c.desc, c.x, c.dy, c.w, y if c.relu else None, dx, dw, db, ws)
    return dx, dw, db


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [1, 37, 1024, 4096])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_fused_backward(layer, B, dtype):
    c = Case(B, **SHAPES[layer], dtype=dtype)
    q = binding.conv_query(binding.OP_BWD, c.desc)
    fused = not (layer == "L1" and B >= 4096)  # fewer than two waves of d_input items
    if fused:
        assert q["algo"] == binding.ALGO_TC and q["launches"] == 3 and q["workspace"] > 0, q
    else:
        assert q["algo"] == binding.ALGO_AUTO and q["workspace"] > 0, q
    y = c.gpu_fwd()
    dx, dw, db = run_bwd(c, y, with_bias=True)
    dx0 = c.gpu_dgrad(y)
    dw0 = c.gpu_wgrad(y)
    torch.cuda.synchronize()
    assert binding.conv_device_status(reset=True) == 0
    assert torch.equal(_bits(dx), _bits(dx0)), "dx differs from conv_bwd_data"
    yn = to_np(y)
    if B <= 1024:
        ref, den = c.ref_dgrad(yn)
        check(to_np(dx), ref, den, dtype, f"{layer} B={B} {dtype} fused dx")
    ref, den = c.ref_wgrad(yn)
    check(to_np(dw), ref, den, dtype, f"{layer} B={B} {dtype} fused dw")
    check(to_np(dw), to_np(dw0), den, dtype, f"{layer} B={B} {dtype} fused dw vs conv_bwd_filter")
    ref, den = oracle.conv_bwd_bias(c.inp["dy"], yn if c.relu else None, c.relu)
    check(to_np(db), ref, den, dtype, f"{layer} B={B} {dtype} fused db")
    # run to run
    dx2, dw2, db2 = run_bwd(c, y, with_bias=True)
    torch.cuda.synchronize()
    for a, b in ((dx, dx2), (dw, dw2), (db, db2)):
        assert torch.equal(_bits(a), _bits(b))


@pytest.mark.parametrize("shape", ["odd", "k_eq_input", "p1_relu_oc64"])
def test_fused_backward_odd_shapes(shape):
    c = Case(5, **SHAPES[shape], dtype="f32")
    y = c.gpu_fwd()
    dx, dw, db = run_bwd(c, y, with_bias=False)
    torch.cuda.synchronize()
    yn = to_np(y)
    ref, den = c.ref_dgrad(yn)
    check(to_np(dx), ref, den, "f32", f"{shape} fused dx")
    ref, den = c.ref_wgrad(yn)
    check(to_np(dw), ref, den, "f32", f"{shape} fused dw")


def test_backward_two_call_path():
    """With the FFMA family forced, conv_bwd runs d_input and wgrad one after the other."""
    for op in (binding.OP_BWD_DATA, binding.OP_BWD_FILTER):
        binding.conv_set_algo(op, binding.ALGO_FFMA)
    c = Case(29, **L1, dtype="f32")
    assert binding.conv_query(binding.OP_BWD, c.desc)["algo"] == binding.ALGO_AUTO
    y = c.gpu_fwd()
    dx, dw, db = run_bwd(c, y, with_bias=True)
    torch.cuda.synchronize()
    yn = to_np(y)
    ref, den = c.ref_dgrad(yn)
    check(to_np(dx), ref, den, "f32", "two-call dx")
    ref, den = c.ref_wgrad(yn)
    check(to_np(dw), ref, den, "f32", "two-call dw")
    ref, den = oracle.conv_bwd_bias(c.inp["dy"], yn, True)
    check(to_np(db), ref, den, "f32", "two-call db")


def test_fused_backward_rejects_small_workspace():
    c = Case(64, **L1, dtype="f32")
    y = c.gpu_fwd()
    need = binding.conv_bwd_workspace_size(c.desc)
    dx, dw = torch.empty_like(c.x), torch.empty_like(c.w)
    with pytest.raises(binding.ConvError) as ei:
        binding.conv_bwd(c.desc, c.x, c.dy, c.w, y, dx, dw, None, torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
    assert ei.value.status == -5
