"""The two-layer encoder stack of PufferLib PR #522 end to end in bf16: layer 1
(11x15 -> 3x4, K=5, S=3, ReLU) feeding layer 2 (3x4 -> 1x2, K=3, S=1), full
forward + backward chain, over a batch sweep B in {256, 1024, 4096, 16384}.

Each GPU call is checked stage by stage against the oracle fed that call's
actual GPU inputs (the GPU's y1 feeds layer 2, the GPU's dy1 feeds layer 1's
backward), within the bf16 tolerance.  At the larger batches the oracle runs
on a sample of the batch (forward / d_input are per-sample) and on a sample of
output channels (wgrad's dw[oc] depends only on dy[:, oc])."""
import numpy as np
import pytest
import torch

import oracle
from implicit_gemm_conv2d_gb300 import binding, synth

from .gpu_cases import TOL, to_dev, to_np

pytestmark = pytest.mark.gpu

L1 = dict(IC=59, OC=128, H=11, W=15, K=5, S=3)
L2 = dict(IC=128, OC=128, H=3, W=4, K=3, S=1)


def _ws(desc):
    return torch.empty(max(16, binding.conv_bwd_filter_workspace_size(desc)), dtype=torch.uint8, device="cuda")


def _check(out, ref, den, what):
    err = oracle.normalised_error(out, ref, den)
    assert err <= TOL["bf16"], f"{what}: normalised error {err:.3e}"


@pytest.mark.parametrize("B", [256, 1024, 4096, 16384])
def test_two_layer_chain_bf16(B):
    dt = torch.bfloat16
    i1 = synth.conv_inputs(B, L1["IC"], L1["OC"], L1["H"], L1["W"], L1["K"], L1["S"], dtype="bf16",
                           need=("x", "w"))
    w2 = synth.conv_inputs(1, L2["IC"], L2["OC"], L2["H"], L2["W"], L2["K"], L2["S"], dtype="bf16",
                           w_stream=synth.STREAM_W2, need=("w",))["w"]
    dy2 = synth.conv_inputs(B, L2["IC"], L2["OC"], L2["H"], L2["W"], L2["K"], L2["S"], dtype="bf16",
                            need=("dy",))["dy"]
    x1, W1, W2, DY2 = to_dev(i1["x"], "bf16"), to_dev(i1["w"], "bf16"), to_dev(w2, "bf16"), to_dev(dy2, "bf16")
    d1 = binding.make_desc(B, **L1, relu=1, dtype=dt)
    d2 = binding.make_desc(B, **L2, relu=0, dtype=dt)
    y1 = torch.empty((B, 128, 3, 4), dtype=dt, device="cuda")
    y2 = torch.empty((B, 128, 1, 2), dtype=dt, device="cuda")
    dw2 = torch.empty_like(W2)
    dy1 = torch.empty_like(y1)
    dw1 = torch.empty_like(W1)
    dx1 = torch.empty_like(x1)
    binding.conv_fwd(d1, x1, W1, y1)
    binding.conv_fwd(d2, y1, W2, y2)
    binding.conv_bwd_filter(d2, y1, DY2, None, dw2, _ws(d2))
    binding.conv_bwd_data(d2, DY2, W2, None, dy1)
    binding.conv_bwd_filter(d1, x1, dy1, y1, dw1, _ws(d1))
    binding.conv_bwd_data(d1, dy1, W1, y1, dx1)
    torch.cuda.synchronize()
    assert binding.conv_device_status(reset=True) == 0

    rng = np.random.default_rng(B)
    samples = np.arange(B) if B <= 1024 else np.sort(rng.choice(B, 256, replace=False))
    chans = np.arange(128) if B <= 1024 else np.sort(rng.choice(128, 8, replace=False))
    x1n, y1n, y2n = i1["x"], to_np(y1), to_np(y2)
    dy1n = to_np(dy1)
    # layer-1 forward, layer-2 forward (on the GPU's y1)
    ref, den = oracle.conv_fwd(x1n[samples], i1["w"], 3, True)
    _check(y1n[samples], ref, den, f"B={B} layer1 fwd")
    ref, den = oracle.conv_fwd(y1n[samples], w2, 1, False)
    _check(y2n[samples], ref, den, f"B={B} layer2 fwd")
    # layer-2 backward
    ref, den = oracle.conv_bwd_data(dy2[samples], w2, None, 3, 4, 1, False)
    _check(dy1n[samples], ref, den, f"B={B} layer2 dgrad")
    ref, den = oracle.conv_bwd_filter(y1n, dy2[:, chans], None, 3, 1, False)
    _check(to_np(dw2)[chans], ref, den, f"B={B} layer2 wgrad")
    # layer-1 backward on the GPU's dy1, masked by the GPU's y1
    ref, den = oracle.conv_bwd_data(dy1n[samples], i1["w"], y1n[samples], 11, 15, 3, True)
    st = torch.from_numpy(samples).to("cuda")
    dx1s = to_np(dx1.index_select(0, st))
    _check(dx1s, ref, den, f"B={B} layer1 dgrad")
    ref, den = oracle.conv_bwd_filter(x1n, dy1n[:, chans], y1n[:, chans], 5, 3, True)
    _check(to_np(dw1)[chans], ref, den, f"B={B} layer1 wgrad")
    assert np.isfinite(dx1s).all()


@pytest.fixture(autouse=True)
def _restore_algo():
    yield
    for op in range(6):
        binding.conv_set_algo(op, binding.ALGO_AUTO)


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


@pytest.mark.parametrize("dtype,B", [("bf16", 256), ("bf16", 1024), ("bf16", 4096), ("bf16", 16384),
                                     ("f32", 256), ("f32", 1024), ("f32", 4096)])
def test_fused_forward_chain(dtype, B):
    """conv_fwd_chain2: both layers' forward in one kernel, layer 1's output tile kept in shared
    memory as layer 2's input.  Checked stage by stage against the oracle (layer 2 fed the
    GPU's y1), y1 bit for bit against conv_fwd, and y2 against conv_fwd on that y1."""
    from .gpu_cases import TORCH_DT
    tdt = TORCH_DT[dtype]
    i1 = synth.conv_inputs(B, L1["IC"], L1["OC"], L1["H"], L1["W"], L1["K"], L1["S"], dtype=dtype,
                           need=("x", "w", "bias"))
    w2 = synth.conv_inputs(1, L2["IC"], L2["OC"], L2["H"], L2["W"], L2["K"], L2["S"], dtype=dtype,
                           w_stream=synth.STREAM_W2, need=("w",))["w"]
    x1, W1, W2, b1 = to_dev(i1["x"], dtype), to_dev(i1["w"], dtype), to_dev(w2, dtype), to_dev(i1["bias"], dtype)
    d1 = binding.make_desc(B, **L1, relu=1, dtype=tdt)
    d2 = binding.make_desc(B, **L2, relu=0, dtype=tdt)
    # bf16: fused while every CTA gets at most one group of 10 samples, else two forward calls;
    # fp32: two forward calls unless the tensor-core family is forced (then fused likewise)
    if dtype == "f32":
        assert binding.conv_query_chain2(d1, d2)["algo"] == binding.ALGO_AUTO
        binding.conv_set_algo(binding.OP_FWD, binding.ALGO_TC)
    q = binding.conv_query_chain2(d1, d2)
    fused = (B + 9) // 10 <= torch.cuda.get_device_properties(0).multi_processor_count
    assert (q["algo"] == binding.ALGO_TC and q["launches"] == 3) if fused else q["algo"] == binding.ALGO_AUTO, q
    ws = torch.empty(binding.conv_fwd_chain2_workspace_size(d1, d2), dtype=torch.uint8, device="cuda")
    y1 = torch.full((B, 128, 3, 4), float("nan"), dtype=tdt, device="cuda")
    y2 = torch.full((B, 128, 1, 2), float("nan"), dtype=tdt, device="cuda")
    binding.conv_fwd_chain2(d1, d2, x1, W1, b1, W2, None, y1, y2, ws)
    y1_ref = torch.empty_like(y1)
    binding.conv_fwd_bias(d1, x1, W1, b1, y1_ref)
    y2_ref = torch.empty_like(y2)
    binding.conv_fwd(d2, y1, W2, y2_ref)
    torch.cuda.synchronize()
    assert binding.conv_device_status(reset=True) == 0
    # The chain's layer 1 sums K in one range; so does conv_fwd_bias unless its plan splits K
    # (fewer column tiles than half the SMs), in which case the two agree within tolerance.
    if binding.conv_query(binding.OP_FWD, d1)["splits"] == 1:
        assert torch.equal(_bits(y1), _bits(y1_ref)), "y1 differs from conv_fwd_bias"
    rng = np.random.default_rng(B + 7)
    samples = np.arange(B) if B <= 1024 else np.sort(rng.choice(B, 256, replace=False))
    y1n, y2n = to_np(y1), to_np(y2)
    assert np.isfinite(y2n).all() and np.isfinite(y1n).all()
    ref, den = oracle.conv_fwd(i1["x"][samples], i1["w"], 3, True, bias=i1["bias"])
    e1 = oracle.normalised_error(y1n[samples], ref, den)
    assert e1 <= TOL[dtype], f"B={B} {dtype} chain layer1: {e1:.3e}"
    ref, den = oracle.conv_fwd(y1n[samples], w2, 1, False)
    e2 = oracle.normalised_error(y2n[samples], ref, den)
    assert e2 <= TOL[dtype], f"B={B} {dtype} chain layer2: {e2:.3e}"
    e3 = oracle.normalised_error(y2n, to_np(y2_ref), oracle.conv_fwd(y1n, w2, 1, False)[1])
    assert e3 <= TOL[dtype], f"B={B} {dtype} chain layer2 vs conv_fwd: {e3:.3e}"
    e4 = oracle.normalised_error(y1n, to_np(y1_ref), oracle.conv_fwd(i1["x"], i1["w"], 3, True, bias=i1["bias"])[1])
    assert e4 <= TOL[dtype], f"B={B} {dtype} chain layer1 vs conv_fwd_bias: {e4:.3e}"


def test_fused_forward_chain_ragged_and_run_to_run():
    """A batch that leaves the last group partial (37 = 3 groups of 10 + 7), twice: bit-identical."""
    B, dtype = 37, "f32"
    i1 = synth.conv_inputs(B, L1["IC"], L1["OC"], L1["H"], L1["W"], L1["K"], L1["S"], dtype=dtype, need=("x", "w"))
    w2 = synth.conv_inputs(1, L2["IC"], L2["OC"], L2["H"], L2["W"], L2["K"], L2["S"], dtype=dtype,
                           w_stream=synth.STREAM_W2, need=("w",))["w"]
    x1, W1, W2 = to_dev(i1["x"], dtype), to_dev(i1["w"], dtype), to_dev(w2, dtype)
    d1 = binding.make_desc(B, **L1, relu=1, dtype=torch.float32)
    d2 = binding.make_desc(B, **L2, relu=0, dtype=torch.float32)
    ws = torch.empty(binding.conv_fwd_chain2_workspace_size(d1, d2), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        y1 = torch.full((B, 128, 3, 4), float("nan"), device="cuda")
        y2 = torch.full((B, 128, 1, 2), float("nan"), device="cuda")
        binding.conv_fwd_chain2(d1, d2, x1, W1, None, W2, None, y1, y2, ws)
        outs.append((y1, y2))
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(_bits(a), _bits(b))
    y1n, y2n = to_np(outs[0][0]), to_np(outs[0][1])
    ref, den = oracle.conv_fwd(i1["x"], i1["w"], 3, True)
    assert oracle.normalised_error(y1n, ref, den) <= TOL[dtype]
    ref, den = oracle.conv_fwd(y1n, w2, 1, False)
    assert oracle.normalised_error(y2n, ref, den) <= TOL[dtype]


def test_chain_descriptors_must_chain():
    d1 = binding.make_desc(8, **L1, relu=1, dtype=torch.float32)
    bad = binding.make_desc(8, 64, 128, 3, 4, 3, 1, 0, torch.float32)  # IC != layer 1's OC
    with pytest.raises(binding.ConvError) as ei:
        binding.conv_query_chain2(d1, bad)
    assert ei.value.status == -2


@pytest.mark.parametrize("dtype,B", [("f32", 37), ("f32", 1024), ("bf16", 37), ("bf16", 1024)])
def test_backward_chain(dtype, B):
    """conv_bwd_chain2: layer 2's backward with dx2 kept in the workspace, then layer 1's on it.
    Stage by stage against the oracle: layer 2 on the GPU's y1 / y2, layer 1 on dx2 as
    conv_bwd_data computes it (the same kernels, bit for bit); without dx1 only layer 1's wgrad
    runs.  Biases' gradients included."""
    from .gpu_cases import TORCH_DT
    tdt = TORCH_DT[dtype]
    i1 = synth.conv_inputs(B, L1["IC"], L1["OC"], L1["H"], L1["W"], L1["K"], L1["S"], dtype=dtype, need=("x", "w"))
    w2 = synth.conv_inputs(1, L2["IC"], L2["OC"], L2["H"], L2["W"], L2["K"], L2["S"], dtype=dtype,
                           w_stream=synth.STREAM_W2, need=("w",))["w"]
    dy2 = synth.conv_inputs(B, L2["IC"], L2["OC"], L2["H"], L2["W"], L2["K"], L2["S"], dtype=dtype,
                            need=("dy",))["dy"]
    x1, W1, W2, DY2 = to_dev(i1["x"], dtype), to_dev(i1["w"], dtype), to_dev(w2, dtype), to_dev(dy2, dtype)
    d1 = binding.make_desc(B, **L1, relu=1, dtype=tdt)
    d2 = binding.make_desc(B, **L2, relu=1, dtype=tdt)  # a ReLU on layer 2 too: both masks
    y1 = torch.empty((B, 128, 3, 4), dtype=tdt, device="cuda")
    y2 = torch.empty((B, 128, 1, 2), dtype=tdt, device="cuda")
    binding.conv_fwd(d1, x1, W1, y1)
    binding.conv_fwd(d2, y1, W2, y2)
    ws = torch.empty(binding.conv_bwd_chain2_workspace_size(d1, d2), dtype=torch.uint8, device="cuda")
    nan = float("nan")
    dx1 = torch.full_like(x1, nan)
    dw1, dw2 = torch.full_like(W1, nan), torch.full_like(W2, nan)
    db1 = torch.full((128,), nan, dtype=tdt, device="cuda")
    db2 = torch.full((128,), nan, dtype=tdt, device="cuda")
    binding.conv_bwd_chain2(d1, d2, x1, W1, y1, W2, y2, DY2, dx1, dw1, db1, dw2, db2, ws)
    # without dx1 (and without the biases): layer 1's wgrad only
    dw1b = torch.full_like(W1, nan)
    dw2b = torch.full_like(W2, nan)
    binding.conv_bwd_chain2(d1, d2, x1, W1, y1, W2, y2, DY2, None, dw1b, None, dw2b, None, ws)
    dx2 = torch.empty_like(y1)
    binding.conv_bwd_data(d2, DY2, W2, y2, dx2)
    torch.cuda.synchronize()
    assert binding.conv_device_status(reset=True) == 0
    y1n, y2n, dx2n = to_np(y1), to_np(y2), to_np(dx2)
    # layer 2
    ref, den = oracle.conv_bwd_filter(y1n, dy2, y2n, 3, 1, True)
    for out in (dw2, dw2b):
        _check_dt(to_np(out), ref, den, dtype, f"B={B} {dtype} chain dw2")
    ref, den = oracle.conv_bwd_bias(dy2, y2n, True)
    _check_dt(to_np(db2), ref, den, dtype, f"B={B} {dtype} chain db2")
    ref, den = oracle.conv_bwd_data(dy2, w2, y2n, 3, 4, 1, True)
    _check_dt(dx2n, ref, den, dtype, f"B={B} {dtype} layer-2 dx (conv_bwd_data)")
    # layer 1 on that dx2, masked by y1
    ref, den = oracle.conv_bwd_filter(i1["x"], dx2n, y1n, 5, 3, True)
    for out in (dw1, dw1b):
        _check_dt(to_np(out), ref, den, dtype, f"B={B} {dtype} chain dw1")
    ref, den = oracle.conv_bwd_bias(dx2n, y1n, True)
    _check_dt(to_np(db1), ref, den, dtype, f"B={B} {dtype} chain db1")
    ref, den = oracle.conv_bwd_data(dx2n, i1["w"], y1n, 11, 15, 3, True)
    _check_dt(to_np(dx1), ref, den, dtype, f"B={B} {dtype} chain dx1")


def _check_dt(out, ref, den, dtype, what):
    assert np.isfinite(out).all(), what
    err = oracle.normalised_error(out, ref, den)
    assert err <= TOL[dtype], f"{what}: normalised error {err:.3e}"
