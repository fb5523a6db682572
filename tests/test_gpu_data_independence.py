"""Both encoder layers at B=16384 in fp32 and bf16 with x and w scaled by 1/8
and by 8, and with binary32 subnormals planted in a seeded 1% of x and w: the
results stay within tolerance of the oracle and the runtime does not depend
on the data (cf. the cut-cross-entropy issue "Runtime of kernel seems
dependant on input data distribution", whose kernel slowed down ~3x when its
inputs were scaled by 1/8).

Scaling by a power of two is exact, so the scaled inputs are made on the
device from the seeded base inputs.  The oracle checks a sample of the batch
(forward / d_input) and of the output channels (wgrad)."""
import numpy as np
import pytest
import torch

import oracle
from implicit_gemm_conv2d_gb300 import binding, synth

from .gpu_cases import TOL, TORCH_DT, to_dev, to_np

pytestmark = pytest.mark.gpu

LAYERS = {"L1": dict(IC=59, OC=128, H=11, W=15, K=5, S=3, relu=1),
          "L2": dict(IC=128, OC=128, H=3, W=4, K=3, S=1, relu=0)}
B = 16384


def _time_ops(run, reps=15):
    ts = {}
    for name, fn in run.items():
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        ts[name] = float(np.median([a.elapsed_time(b) for a, b in ev]))
    return ts


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layer", ["L1", "L2"])
def test_scaled_and_subnormal_inputs(layer, dtype):
    sh = LAYERS[layer]
    tdt = TORCH_DT[dtype]
    base = synth.conv_inputs(B, sh["IC"], sh["OC"], sh["H"], sh["W"], sh["K"], sh["S"], dtype=dtype)
    sub = synth.conv_inputs(B, sh["IC"], sh["OC"], sh["H"], sh["W"], sh["K"], sh["S"], dtype=dtype,
                            subnormal=True, need=("x", "w"))
    desc = binding.make_desc(B, **sh, dtype=tdt)
    OH, OW = binding.out_dims(desc)
    dy = to_dev(base["dy"], dtype)
    rng = np.random.default_rng(5)
    samples = np.sort(rng.choice(B, 96, replace=False))
    chans = np.sort(rng.choice(sh["OC"], 6, replace=False))
    st = torch.from_numpy(samples).to("cuda")
    times = {}
    for variant in ("base", "x1/8", "x8", "subnormal"):
        if variant == "subnormal":
            xh, wh = sub["x"], sub["w"]
        else:
            s = {"base": 1.0, "x1/8": 0.125, "x8": 8.0}[variant]
            xh, wh = base["x"] * np.float32(s), base["w"] * np.float32(s)
        x, w = to_dev(xh, dtype), to_dev(wh, dtype)
        y = torch.empty((B, sh["OC"], OH, OW), dtype=tdt, device="cuda")
        dx = torch.empty_like(x)
        dw = torch.empty_like(w)
        ws = torch.empty(max(16, binding.conv_bwd_filter_workspace_size(desc)), dtype=torch.uint8, device="cuda")
        ym = y if sh["relu"] else None
        run = {"fwd": lambda: binding.conv_fwd(desc, x, w, y),
               "dgrad": lambda: binding.conv_bwd_data(desc, dy, w, ym, dx),
               "wgrad": lambda: binding.conv_bwd_filter(desc, x, dy, ym, dw, ws)}
        times[variant] = _time_ops(run)
        torch.cuda.synchronize()
        assert binding.conv_device_status(reset=True) == 0
        yn = to_np(y)
        ref, den = oracle.conv_fwd(xh[samples], wh, sh["S"], sh["relu"])
        e = oracle.normalised_error(yn[samples], ref, den)
        assert e <= TOL[dtype], (variant, "fwd", e)
        ref, den = oracle.conv_bwd_data(base["dy"][samples], wh, yn[samples] if sh["relu"] else None,
                                        sh["H"], sh["W"], sh["S"], sh["relu"])
        e = oracle.normalised_error(to_np(dx.index_select(0, st)), ref, den)
        assert e <= TOL[dtype], (variant, "dgrad", e)
        ref, den = oracle.conv_bwd_filter(xh, base["dy"][:, chans], yn[:, chans] if sh["relu"] else None,
                                          sh["K"], sh["S"], sh["relu"])
        e = oracle.normalised_error(to_np(dw)[chans], ref, den)
        assert e <= TOL[dtype], (variant, "wgrad", e)
        del x, w, y, dx, dw, ws
    print(f"\n{layer} {dtype} B={B} median ms:", {v: {k: round(t, 4) for k, t in d.items()} for v, d in times.items()})
    for variant in ("x1/8", "x8", "subnormal"):
        for op in ("fwd", "dgrad", "wgrad"):
            r = times[variant][op] / times["base"][op]
            assert 0.85 < r < 1.15, f"{layer} {dtype} {op} runtime with {variant} inputs is {r:.2f}x the base"
