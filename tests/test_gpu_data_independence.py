"""Both encoder layers at B=16384 in fp32 and bf16 with x and w scaled by 1/8
and by 8, and with binary32 subnormals planted in a seeded 1% of x and w: the
results stay within tolerance of the oracle and the runtime does not depend
on the data (cf. the cut-cross-entropy issue "Runtime of kernel seems
dependant on input data distribution", whose kernel slowed down ~3x when its
inputs were scaled by 1/8).

Pass condition per operation: the median time of every variant within +-3 %
of the unscaled run's median.  Timing protocol, chosen so that only the data
differs between variants: all four variants' buffers are resident at once;
each repetition times every (operation, variant) pair once, in an order
rotated from one repetition to the next; L2 is flushed (a 512 MiB write)
before every timed call, so each one starts cold; CUDA events on the
launching stream bracket the call alone.  The medians and ratios are printed
(run pytest with -s to see them).

Scaling by a power of two is exact, so the scaled inputs are made from the
seeded base inputs.  The oracle checks a sample of the batch (forward /
d_input) and of the output channels (wgrad)."""
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
VARIANTS = ("base", "x1/8", "x8", "subnormal")
OPS = ("fwd", "dgrad", "wgrad")
REPS = 61
RATIO_BAND = (0.97, 1.03)


def _time_interleaved(runs, flush):
    """Median ms per (variant, op) over REPS repetitions; each repetition times every
    pair once, cold L2, in a rotated order."""
    pairs = [(v, o) for o in OPS for v in VARIANTS]
    for v, o in pairs:  # warm-up: plans, first-touch
        runs[v][o]()
    torch.cuda.synchronize()
    ev = {pr: [] for pr in pairs}
    for r in range(REPS):
        order = pairs[r % len(pairs):] + pairs[:r % len(pairs)]
        for pr in order:
            binding.conv_l2_flush(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            runs[pr[0]][pr[1]]()
            b.record()
            ev[pr].append((a, b))
        if r % 8 == 7:
            torch.cuda.synchronize()  # bound the events in flight
    torch.cuda.synchronize()
    return {pr: float(np.median([a.elapsed_time(b) for a, b in e])) for pr, e in ev.items()}


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
    host, runs, keep = {}, {}, []
    for variant in VARIANTS:
        if variant == "subnormal":
            xh, wh = sub["x"], sub["w"]
        else:
            s = {"base": 1.0, "x1/8": 0.125, "x8": 8.0}[variant]
            xh, wh = base["x"] * np.float32(s), base["w"] * np.float32(s)
        host[variant] = (xh, wh)
        x, w = to_dev(xh, dtype), to_dev(wh, dtype)
        y = torch.empty((B, sh["OC"], OH, OW), dtype=tdt, device="cuda")
        dx = torch.empty_like(x)
        dw = torch.empty_like(w)
        ws = torch.empty(max(16, binding.conv_bwd_filter_workspace_size(desc)), dtype=torch.uint8, device="cuda")
        ym = y if sh["relu"] else None
        runs[variant] = {
            "fwd": (lambda x=x, w=w, y=y: binding.conv_fwd(desc, x, w, y)),
            "dgrad": (lambda w=w, ym=ym, dx=dx: binding.conv_bwd_data(desc, dy, w, ym, dx)),
            "wgrad": (lambda x=x, ym=ym, dw=dw, ws=ws: binding.conv_bwd_filter(desc, x, dy, ym, dw, ws)),
        }
        keep.append((x, w, y, dx, dw, ws))
    # Parity of every variant.
    for variant, (x, w, y, dx, dw, ws) in zip(VARIANTS, keep):
        xh, wh = host[variant]
        for o in OPS:
            runs[variant][o]()
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
    # Runtime independence.
    flush = torch.empty((512 << 20) // 4, dtype=torch.float32, device="cuda")
    med = _time_interleaved(runs, flush)
    torch.cuda.synchronize()
    assert binding.conv_device_status(reset=True) == 0
    bad = []
    for o in OPS:
        line = [f"DATAIND {layer} {dtype} B={B} {o}: base {med[('base', o)] * 1e3:.2f} us"]
        for v in VARIANTS[1:]:
            r = med[(v, o)] / med[("base", o)]
            line.append(f"{v} {med[(v, o)] * 1e3:.2f} us ({r:.4f})")
            if not (RATIO_BAND[0] <= r <= RATIO_BAND[1]):
                bad.append(f"{o} {v} {r:.4f}")
        print("; ".join(line))
    assert not bad, f"{layer} {dtype}: median runtime outside +-3 % of the unscaled run: {bad}"
