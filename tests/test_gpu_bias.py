"""GPU parity of the per-channel conv bias, through the C ABI, against the fp64
oracle on the same seeded inputs: the forward with the bias (every forward
kernel family, including the tensor-core epilogue and its split-K reduce, both
dtypes, both layers of PufferLib PR #522's encoder, ragged and odd shapes) and
the bias gradient (column-sum and one-warp-per-channel kernels; the vectorised
and scalar column paths; one and several channel windows), at the batch the
PR's "n3_conv_bias_grad" blocks use (B = 32768), for an empty batch, and run to
run.  Tolerances are those of tests/gpu_cases.py; the bias gradient's
denominator is sum |g| over the terms it adds."""
import numpy as np
import pytest
import torch

import oracle
from implicit_gemm_conv2d_gb300 import binding, synth

from .gpu_cases import L1, L2, TORCH_DT, check, to_dev, to_np

pytestmark = pytest.mark.gpu

SHAPES = {
    "L1": L1,
    "L2": L2,
    "odd": dict(IC=3, OC=5, H=7, W=9, K=2, S=2, relu=True),            # OC*P = 60: scalar columns
    "wide_oc_p16": dict(IC=4, OC=200, H=6, W=6, K=3, S=1, relu=False),
    "k1": dict(IC=16, OC=24, H=3, W=5, K=1, S=1, relu=False),
    "stride_gt_k": dict(IC=5, OC=20, H=10, W=11, K=2, S=3, relu=False),
    "two_windows": dict(IC=2, OC=200, H=10, W=10, K=1, S=1, relu=True),  # OC*P = 20000 > one window
    "long_rows": dict(IC=1, OC=3, H=120, W=120, K=1, S=1, relu=False),   # P = 14400: direct kernel
}


@pytest.fixture(autouse=True)
def _restore_algo():
    yield
    for op in range(4):
        binding.conv_set_algo(op, binding.ALGO_AUTO)


class BiasCase:
    def __init__(self, B, IC, OC, H, W, K, S, relu, dtype="f32", need=("x", "w", "dy", "bias")):
        self.B, self.IC, self.OC, self.H, self.W, self.K, self.S = B, IC, OC, H, W, K, S
        self.relu, self.dtype = bool(relu), dtype
        self.inp = synth.conv_inputs(B, IC, OC, H, W, K, S, dtype=dtype, need=need)
        self.dev = {k: to_dev(v, dtype) for k, v in self.inp.items()}
        self.desc = binding.make_desc(B, IC, OC, H, W, K, S, relu, TORCH_DT[dtype])
        self.OH, self.OW = binding.out_dims(self.desc)

    def gpu_fwd(self, bias=True):
        y = torch.empty((self.B, self.OC, self.OH, self.OW), dtype=TORCH_DT[self.dtype], device="cuda")
        d = self.dev
        if bias:
            binding.conv_fwd_bias(self.desc, d["x"], d["w"], d["bias"], y)
        else:
            binding.conv_fwd(self.desc, d["x"], d["w"], y)
        return y

    def gpu_bgrad(self, y):
        db = torch.full((self.OC,), float("nan"), dtype=TORCH_DT[self.dtype], device="cuda")
        binding.conv_bwd_bias(self.desc, self.dev["dy"], y if self.relu else None, db)
        return db

    def ref_fwd(self):
        return oracle.conv_fwd(self.inp["x"], self.inp["w"], self.S, self.relu, bias=self.inp["bias"])

    def ref_bgrad(self, y_np):
        return oracle.conv_bwd_bias(self.inp["dy"], y_np if self.relu else None, self.relu)


def fwd_and_bgrad(c: BiasCase, label: str):
    y = c.gpu_fwd()
    db = c.gpu_bgrad(y)
    torch.cuda.synchronize()
    yn = to_np(y)
    ref, den = c.ref_fwd()
    check(yn, ref, den, c.dtype, f"{label} fwd+bias")
    ref, den = c.ref_bgrad(yn)
    check(to_np(db), ref, den, c.dtype, f"{label} bias grad")
    assert binding.conv_device_status(reset=True) == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [1, 37, 1024])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_encoder_layers_with_bias(layer, B, dtype):
    fwd_and_bgrad(BiasCase(B, **SHAPES[layer], dtype=dtype), f"{layer} B={B} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bias_in_tensor_core_epilogue(dtype):
    """On 152 SMs, layer 1 at B = 1024 and 4096 has enough column tiles for the tensor-core
    forward to run without K ranges, so the bias is added in its epilogue; layer 2 at
    B = 1024 splits K over a thread-block cluster and the cluster's reduction adds it (both
    checked by test_encoder_layers_with_bias at B = 1024; here layer 1 at B = 4096 too).
    Either way the forward is one launch."""
    c = BiasCase(4096, **L1, dtype=dtype)
    q = binding.conv_query(binding.OP_FWD, c.desc)
    assert q["algo"] == binding.ALGO_TC and q["launches"] == 1 and q["splits"] == 1
    q1 = binding.conv_query(binding.OP_FWD, BiasCase(1024, **L1, dtype=dtype, need=("dy",)).desc)
    assert q1["launches"] == 1 and q1["splits"] == 1
    q2 = binding.conv_query(binding.OP_FWD, BiasCase(1024, **L2, dtype=dtype, need=("dy",)).desc)
    assert q2["launches"] == 1 and q2["splits"] > 1
    fwd_and_bgrad(c, f"L1 B=4096 {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [s for s in SHAPES if s not in ("L1", "L2")])
def test_odd_shapes_with_bias(shape, dtype):
    fwd_and_bgrad(BiasCase(5, **SHAPES[shape], dtype=dtype), f"{shape} {dtype}")


@pytest.mark.parametrize("algo", [binding.ALGO_DIRECT, binding.ALGO_FFMA, binding.ALGO_TC])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_forward_bias_each_family(layer, dtype, algo):
    binding.conv_set_algo(binding.OP_FWD, algo)
    c = BiasCase(29, **SHAPES[layer], dtype=dtype)
    assert binding.conv_query(binding.OP_FWD, c.desc)["algo"] == algo
    y = c.gpu_fwd()
    torch.cuda.synchronize()
    ref, den = c.ref_fwd()
    check(to_np(y), ref, den, dtype, f"{layer} {dtype} algo={algo} fwd+bias")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_bias_grad_direct_kernel(layer, dtype):
    binding.conv_set_algo(binding.OP_BWD_BIAS, binding.ALGO_DIRECT)
    c = BiasCase(37, **SHAPES[layer], dtype=dtype)
    assert binding.conv_query(binding.OP_BWD_BIAS, c.desc)["algo"] == binding.ALGO_DIRECT
    fwd_and_bgrad(c, f"{layer} {dtype} direct")


def test_bias_grad_plans():
    c = BiasCase(1024, **L1, dtype="f32", need=("dy",))
    q = binding.conv_query(binding.OP_BWD_BIAS, c.desc)
    assert q["algo"] == binding.ALGO_FFMA and q["launches"] == 1 and q["splits"] in (2, 4, 8)
    c = BiasCase(2, **SHAPES["long_rows"], dtype="f32", need=("dy",))
    assert binding.conv_query(binding.OP_BWD_BIAS, c.desc)["algo"] == binding.ALGO_DIRECT


@pytest.mark.parametrize("layer,dtype", [("L1", "f32"), ("L2", "f32"), ("L2", "bf16")])
def test_bias_grad_at_the_pages_batch(layer, dtype):
    """B = 32768, the batch of the PR's bias-gradient blocks (its gradient has 50.3 M
    elements for layer 1 and 8.4 M for layer 2), without the mask, as timed there."""
    shape = dict(SHAPES[layer], relu=False)
    c = BiasCase(32768, **shape, dtype=dtype, need=("dy",))
    db = torch.empty((c.OC,), dtype=TORCH_DT[dtype], device="cuda")
    binding.conv_bwd_bias(c.desc, c.dev["dy"], None, db)
    torch.cuda.synchronize()
    assert c.dev["dy"].numel() == 32768 * 128 * c.OH * c.OW
    ref, den = oracle.conv_bwd_bias(c.inp["dy"], None, False)
    check(to_np(db), ref, den, dtype, f"{layer} B=32768 {dtype} bias grad")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bias_grad_empty_batch_writes_zeros(dtype):
    d0 = binding.make_desc(0, 59, 128, 11, 15, 5, 3, 1, TORCH_DT[dtype])
    db = torch.full((128,), 7.0, dtype=TORCH_DT[dtype], device="cuda")
    empty = torch.empty(0, dtype=TORCH_DT[dtype], device="cuda")
    binding.conv_bwd_bias(d0, empty, empty, db)
    torch.cuda.synchronize()
    assert torch.count_nonzero(db).item() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_bias_bit_identical_run_to_run(layer, dtype):
    c = BiasCase(1024, **SHAPES[layer], dtype=dtype)
    outs = []
    for _ in range(2):
        y = c.gpu_fwd()
        outs.append((y, c.gpu_bgrad(y)))
    torch.cuda.synchronize()
    iv = torch.int16 if dtype == "bf16" else torch.int32
    for a, b in zip(*outs):
        assert torch.equal(a.view(iv), b.view(iv))


def test_zero_bias_matches_plain_forward():
    """conv_fwd_bias with an all-zero bias gives conv_fwd's bits (x + 0 = x in fp32)."""
    c = BiasCase(64, **L1, dtype="f32")
    c.dev["bias"].zero_()
    a = c.gpu_fwd(bias=True)
    b = c.gpu_fwd(bias=False)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def wgrad_and_bias(c: BiasCase, label: str, y=None):
    """conv_bwd_filter_bias: dw bit for bit as conv_bwd_filter, db against the oracle."""
    y = c.gpu_fwd() if y is None else y
    ym = y if c.relu else None
    d = c.dev
    ws = torch.empty(max(16, binding.conv_bwd_filter_workspace_size(c.desc)), dtype=torch.uint8, device="cuda")
    dw_ref = torch.empty((c.OC, c.IC, c.K, c.K), dtype=TORCH_DT[c.dtype], device="cuda")
    binding.conv_bwd_filter(c.desc, d["x"], d["dy"], ym, dw_ref, ws)
    dw = torch.full_like(dw_ref, float("nan"))
    db = torch.full((c.OC,), float("nan"), dtype=TORCH_DT[c.dtype], device="cuda")
    binding.conv_bwd_filter_bias(c.desc, d["x"], d["dy"], ym, dw, db, ws)
    torch.cuda.synchronize()
    assert torch.equal(_bits(dw), _bits(dw_ref)), f"{label}: dw differs from conv_bwd_filter's"
    ref, den = c.ref_bgrad(to_np(y))
    check(to_np(db), ref, den, c.dtype, f"{label} fused bias grad")
    assert binding.conv_device_status(reset=True) == 0
    return db


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [1, 37, 1024])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_bias_grad_fused_into_wgrad(layer, B, dtype):
    c = BiasCase(B, **SHAPES[layer], dtype=dtype)
    assert binding.conv_query(binding.OP_BWD_FILTER, c.desc)["algo"] == binding.ALGO_TC
    db = wgrad_and_bias(c, f"{layer} B={B} {dtype}")
    # run to run: bit-identical
    db2 = wgrad_and_bias(c, f"{layer} B={B} {dtype} again")
    assert torch.equal(_bits(db), _bits(db2))


@pytest.mark.parametrize("shape", ["odd", "wide_oc_p16", "k1", "stride_gt_k", "two_windows"])
def test_bias_grad_fused_odd_shapes(shape):
    wgrad_and_bias(BiasCase(5, **SHAPES[shape], dtype="f32"), shape)


@pytest.mark.parametrize("algo", [binding.ALGO_FFMA, binding.ALGO_DIRECT])
def test_bias_grad_with_other_wgrad_families(algo):
    """The FFMA and direct wgrad families run the bias-gradient kernel after the weight gradient."""
    binding.conv_set_algo(binding.OP_BWD_FILTER, algo)
    c = BiasCase(29, **L1, dtype="f32")
    assert binding.conv_query(binding.OP_BWD_FILTER, c.desc)["algo"] == algo
    wgrad_and_bias(c, f"L1 algo={algo}")


def test_bias_grad_fused_empty_batch():
    c = BiasCase(1, **L1, dtype="f32")
    d0 = binding.make_desc(0, 59, 128, 11, 15, 5, 3, 1, torch.float32)
    dw = torch.full((128, 59, 5, 5), 7.0, device="cuda")
    db = torch.full((128,), 7.0, device="cuda")
    e = torch.empty(0, device="cuda")
    ws = torch.empty(max(16, binding.conv_bwd_filter_workspace_size(d0)), dtype=torch.uint8, device="cuda")
    binding.conv_bwd_filter_bias(d0, e, e, e, dw, db, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw).item() == 0 and torch.count_nonzero(db).item() == 0
