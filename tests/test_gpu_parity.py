"""GPU parity: the library's forward, d_input and wgrad, called through the C
ABI, against the fp64 oracle on the same seeded inputs, element by element,
within the normalised-error tolerances of tests/gpu_cases.py.  Covers both
layers of PufferLib PR #522's encoder at B = 1, a ragged 37 and the full
1024, both dtypes, every kernel family, odd shapes that exercise tile tails,
and the degenerate cases (empty batch, 1x1 kernel, kernel as large as the
input)."""
import numpy as np
import pytest
import torch

from implicit_gemm_conv2d_gb300 import binding

from .gpu_cases import L1, L2, Case, check, to_np

pytestmark = pytest.mark.gpu

SHAPES = {
    "L1": L1,
    "L2": L2,
    "odd": dict(IC=3, OC=5, H=7, W=9, K=2, S=2, relu=True),
    "wide_oc_p16": dict(IC=4, OC=200, H=6, W=6, K=3, S=1, relu=False),
    "kk_above_128": dict(IC=2, OC=8, H=13, W=12, K=12, S=1, relu=True),
    "k1": dict(IC=16, OC=24, H=3, W=5, K=1, S=1, relu=False),
    # 1x1 with 128 channels per d_input k-tile (the widest its plan encodes)
    "k1_wide": dict(IC=160, OC=64, H=4, W=5, K=1, S=1, relu=True),
    "k_eq_input": dict(IC=7, OC=33, H=5, W=5, K=5, S=2, relu=True),
    "stride_gt_k": dict(IC=5, OC=20, H=10, W=11, K=2, S=3, relu=False),
    # layer 1's input size, kernel and stride (the d_input gather compiled for them) without the
    # ReLU, one full k-tile of 5 channels and a ragged one of 2
    "l1_geometry_ic7": dict(IC=7, OC=16, H=11, W=15, K=5, S=3, relu=False),
    # one output position per sample and 64 channels: d_input stages dy and y (ReLU) of a sample
    # tile through shared memory by bulk copies (128 samples per tile: B = 200 is one full tile
    # and a ragged one)
    "p1_relu_oc64": dict(IC=16, OC=64, H=4, W=4, K=3, S=2, relu=True),
}


@pytest.fixture(autouse=True)
def _restore_algo():
    yield
    for op in range(3):
        binding.conv_set_algo(op, binding.ALGO_AUTO)


def run_and_check(c: Case, label: str):
    y = c.gpu_fwd()
    dx = c.gpu_dgrad(y)
    dw = c.gpu_wgrad(y)
    torch.cuda.synchronize()
    yn = to_np(y)
    ref, den = c.ref_fwd()
    e1 = check(yn, ref, den, c.dtype, f"{label} fwd")
    ref, den = c.ref_dgrad(yn)
    e2 = check(to_np(dx), ref, den, c.dtype, f"{label} dgrad")
    ref, den = c.ref_wgrad(yn)
    e3 = check(to_np(dw), ref, den, c.dtype, f"{label} wgrad")
    return e1, e2, e3


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [1, 37, 1024])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_encoder_layers(layer, B, dtype):
    run_and_check(Case(B, **SHAPES[layer], dtype=dtype), f"{layer} B={B} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [s for s in SHAPES if s not in ("L1", "L2")])
def test_odd_shapes(shape, dtype):
    run_and_check(Case(5, **SHAPES[shape], dtype=dtype), f"{shape} {dtype}")


@pytest.mark.parametrize("algo", [binding.ALGO_DIRECT, binding.ALGO_FFMA])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_each_family(layer, dtype, algo):
    for op in range(3):
        binding.conv_set_algo(op, algo)
    c = Case(29, **SHAPES[layer], dtype=dtype)
    for op in range(3):
        assert binding.conv_query(op, c.desc)["algo"] == algo
    run_and_check(c, f"{layer} {dtype} algo={algo}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_bit_identical_run_to_run(layer, dtype):
    c = Case(1024, **SHAPES[layer], dtype=dtype)
    outs = []
    for _ in range(2):
        y = c.gpu_fwd()
        outs.append((y, c.gpu_dgrad(y), c.gpu_wgrad(y)))
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                           b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))


def test_layer1_unread_column_has_zero_gradient():
    c = Case(64, **L1, dtype="f32")
    y = c.gpu_fwd()
    dx = c.gpu_dgrad(y)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dx[..., 14]).item() == 0
    assert torch.count_nonzero(dx[..., :14]).item() > 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_empty_batch(dtype):
    c = Case(1, **L1, dtype=dtype)
    d0 = binding.make_desc(0, 59, 128, 11, 15, 5, 3, 1, c.x.dtype)
    dw = torch.full((128, 59, 5, 5), 7.0, dtype=c.x.dtype, device="cuda")
    n = binding.conv_bwd_filter_workspace_size(d0)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    binding.conv_bwd_filter(d0, c.x[:0], c.dy[:0], c.dy[:0], dw, ws)
    binding.conv_fwd(d0, c.x[:0], c.w, torch.empty(0, device="cuda", dtype=c.x.dtype))
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw).item() == 0


def test_workspace_too_small_is_rejected():
    c = Case(64, **L1, dtype="f32")
    y = c.gpu_fwd()
    need = binding.conv_bwd_filter_workspace_size(c.desc)
    assert need > 0
    dw = torch.empty((128, 59, 5, 5), device="cuda")
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.ConvError) as ei:
        binding.conv_bwd_filter(c.desc, c.x, c.dy, y, dw, small)
    assert ei.value.status == -5
    with pytest.raises(binding.ConvError):
        binding.conv_bwd_filter(c.desc, c.x, c.dy, y, dw, None)


def test_query_reports_plan():
    c = Case(1024, **L1, dtype="f32")
    q = binding.conv_query(binding.OP_BWD_FILTER, c.desc)
    assert q["launches"] == 2 and q["splits"] >= 1 and q["workspace"] > 0
    # the forward and d_input are one launch each in every family (the tensor-core kernels
    # format the weights themselves and reduce K ranges inside a cluster)
    for op in (binding.OP_FWD, binding.OP_BWD_DATA):
        q = binding.conv_query(op, c.desc)
        assert q["launches"] == 1 and q["workspace"] == 0 and q["grid"] >= 1


def test_outputs_fully_overwritten():
    """Each call overwrites its whole output: pre-fill with NaN and compare."""
    c = Case(37, **L1, dtype="f32")
    y = torch.full((37, 128, 3, 4), float("nan"), device="cuda")
    binding.conv_fwd(c.desc, c.x, c.w, y)
    dx = torch.full((37, 59, 11, 15), float("nan"), device="cuda")
    binding.conv_bwd_data(c.desc, c.dy, c.w, y, dx)
    dw = torch.full((128, 59, 5, 5), float("nan"), device="cuda")
    ws = torch.full((binding.conv_bwd_filter_workspace_size(c.desc) // 4,), float("nan"), device="cuda")
    binding.conv_bwd_filter(c.desc, c.x, c.dy, y, dw, ws)
    torch.cuda.synchronize()
    for t in (y, dx, dw):
        assert not torch.isnan(t).any()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [3, 200])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_tc_forward(shape, B, dtype):
    """tcgen05 forward (bf16: kind::f16; fp32: 3xTF32) against the oracle."""
    binding.conv_set_algo(binding.OP_FWD, binding.ALGO_TC)
    c = Case(B, **SHAPES[shape], dtype=dtype)
    assert binding.conv_query(binding.OP_FWD, c.desc)["algo"] == binding.ALGO_TC
    y = c.gpu_fwd()
    torch.cuda.synchronize()
    ref, den = c.ref_fwd()
    check(to_np(y), ref, den, dtype, f"tc fwd {shape} B={B} {dtype}")
    assert binding.conv_device_status(reset=True) == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_tc_forward_full_batch(layer, dtype):
    binding.conv_set_algo(binding.OP_FWD, binding.ALGO_TC)
    c = Case(1024, **SHAPES[layer], dtype=dtype)
    y = c.gpu_fwd()
    torch.cuda.synchronize()
    ref, den = c.ref_fwd()
    check(to_np(y), ref, den, dtype, f"tc fwd {layer} B=1024 {dtype}")
    y2 = c.gpu_fwd()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16 if dtype == "bf16" else torch.int32),
                       y2.view(torch.int16 if dtype == "bf16" else torch.int32))
    assert binding.conv_device_status(reset=True) == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [3, 200, 1024])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_tc_wgrad(shape, B, dtype):
    """tcgen05 wgrad split-K partials + reduction against the oracle."""
    if B == 1024 and shape not in ("L1", "L2"):
        pytest.skip("full batch only for the encoder layers")
    binding.conv_set_algo(binding.OP_BWD_FILTER, binding.ALGO_TC)
    c = Case(B, **SHAPES[shape], dtype=dtype)
    try:
        q = binding.conv_query(binding.OP_BWD_FILTER, c.desc)
    except binding.ConvError:
        pytest.skip("shape outside the tensor-core wgrad kernel's limits")
    assert q["algo"] == binding.ALGO_TC
    y = c.gpu_fwd()
    dw = c.gpu_wgrad(y)
    torch.cuda.synchronize()
    yn = to_np(y)
    ref, den = c.ref_wgrad(yn)
    check(to_np(dw), ref, den, dtype, f"tc wgrad {shape} B={B} {dtype}")
    assert binding.conv_device_status(reset=True) == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [2048, 2051])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_tc_wgrad_large_batch(shape, B, dtype):
    """From 2048 samples bf16 wgrad keeps g in tensor memory and the patches in shared memory
    (k-tiles of up to 256 rows); fp32 keeps the patches in tensor memory.  Both against the
    oracle, a full and a ragged last chunk, and run to run bit identity."""
    binding.conv_set_algo(binding.OP_BWD_FILTER, binding.ALGO_TC)
    c = Case(B, **SHAPES[shape], dtype=dtype)
    try:
        binding.conv_query(binding.OP_BWD_FILTER, c.desc)
    except binding.ConvError:
        pytest.skip("shape outside the tensor-core wgrad kernel's limits")
    y = c.gpu_fwd()
    dw = c.gpu_wgrad(y)
    dw2 = c.gpu_wgrad(y)
    torch.cuda.synchronize()
    assert binding.conv_device_status(reset=True) == 0
    ref, den = c.ref_wgrad(to_np(y))
    check(to_np(dw), ref, den, dtype, f"tc wgrad {shape} B={B} {dtype}")
    assert torch.equal(_bits(dw), _bits(dw2))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [3, 200, 1024])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_tc_dgrad(shape, B, dtype):
    """tcgen05 d_input (resident W^T chunk, TMEM accumulator, shared-memory col2im)."""
    if B == 1024 and shape not in ("L1", "L2"):
        pytest.skip("full batch only for the encoder layers")
    c = Case(B, **SHAPES[shape], dtype=dtype)
    binding.conv_set_algo(binding.OP_BWD_DATA, binding.ALGO_TC)
    try:
        q = binding.conv_query(binding.OP_BWD_DATA, c.desc)
    except binding.ConvError:
        pytest.skip("shape outside the tensor-core d_input kernel's limits")
    assert q["algo"] == binding.ALGO_TC
    y = c.gpu_fwd()
    dx = c.gpu_dgrad(y)
    torch.cuda.synchronize()
    yn = to_np(y)
    ref, den = c.ref_dgrad(yn)
    check(to_np(dx), ref, den, dtype, f"tc dgrad {shape} B={B} {dtype}")
    assert binding.conv_device_status(reset=True) == 0


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [1, 37, 1024])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_workspace_path(layer, B, dtype):
    """conv_fwd_ws / conv_bwd_data_ws (weights packed once into the caller's workspace) against
    the oracle, and bit for bit against conv_fwd / conv_bwd_data (weights formatted in the
    kernel): both build the same operand tiles."""
    c = Case(B, **SHAPES[layer], dtype=dtype)
    assert binding.conv_fwd_workspace_size(c.desc) > 0 and binding.conv_bwd_data_workspace_size(c.desc) > 0
    y = c.gpu_fwd_ws()
    dx = c.gpu_dgrad_ws(y)
    y0 = c.gpu_fwd()
    dx0 = c.gpu_dgrad(y)
    torch.cuda.synchronize()
    yn = to_np(y)
    ref, den = c.ref_fwd()
    check(yn, ref, den, dtype, f"{layer} B={B} {dtype} fwd_ws")
    ref, den = c.ref_dgrad(yn)
    check(to_np(dx), ref, den, dtype, f"{layer} B={B} {dtype} dgrad_ws")
    assert torch.equal(_bits(y), _bits(y0)), "conv_fwd_ws and conv_fwd differ"
    assert torch.equal(_bits(dx), _bits(dx0)), "conv_bwd_data_ws and conv_bwd_data differ"
    assert binding.conv_device_status(reset=True) == 0


@pytest.mark.parametrize("shape", [s for s in SHAPES if s not in ("L1", "L2")])
def test_workspace_path_odd_shapes(shape):
    c = Case(5, **SHAPES[shape], dtype="f32")
    y = c.gpu_fwd_ws()
    dx = c.gpu_dgrad_ws(y)
    torch.cuda.synchronize()
    yn = to_np(y)
    ref, den = c.ref_fwd()
    check(yn, ref, den, "f32", f"{shape} fwd_ws")
    ref, den = c.ref_dgrad(yn)
    check(to_np(dx), ref, den, "f32", f"{shape} dgrad_ws")


def test_workspace_path_rejects_small_workspace():
    c = Case(64, **L1, dtype="f32")
    y = torch.empty((64, 128, 3, 4), device="cuda")
    for size_fn, call in ((binding.conv_fwd_workspace_size,
                           lambda ws: binding.conv_fwd_ws(c.desc, c.x, c.w, None, y, ws)),
                          (binding.conv_bwd_data_workspace_size,
                           lambda ws: binding.conv_bwd_data_ws(c.desc, c.dy, c.w, y, torch.empty_like(c.x), ws))):
        need = size_fn(c.desc)
        assert need > 0
        with pytest.raises(binding.ConvError) as ei:
            call(torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
        assert ei.value.status == -5
        with pytest.raises(binding.ConvError):
            call(None)
