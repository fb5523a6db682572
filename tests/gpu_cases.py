"""Helpers for the GPU parity tests: seeded inputs on the device, the library's
three results through the C ABI, and the oracle's results on the same inputs.

Tolerances (normalised error |out - ref| / sum|terms|, max over elements):
  fp32  1e-5   (fp32 FFMA accumulation: typical error ~1e-7 of the
                denominator; worst-case recursive-summation bound Kred * 2^-24)
  bf16  8e-3   (one bf16 output rounding <= 2^-8 relative plus fp32
                accumulation; inputs are the same bf16 values on both sides)
Where the denominator is 0 the output must equal the reference exactly.
"""
import numpy as np
import torch

import oracle
from implicit_gemm_conv2d_gb300 import binding, synth

TOL = {"f32": 1e-5, "bf16": 8e-3}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}

L1 = dict(IC=59, OC=128, H=11, W=15, K=5, S=3, relu=True)   # layer 1 of the PR's encoder
L2 = dict(IC=128, OC=128, H=3, W=4, K=3, S=1, relu=False)   # layer 2


def to_dev(a: np.ndarray, dtype: str):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device="cuda").to(TORCH_DT[dtype]).contiguous()


def to_np(t) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


class Case:
    def __init__(self, B, IC, OC, H, W, K, S, relu, dtype="f32", seed=synth.SEED, scale=1.0,
                 subnormal=False):
        self.B, self.IC, self.OC, self.H, self.W, self.K, self.S = B, IC, OC, H, W, K, S
        self.relu, self.dtype = bool(relu), dtype
        self.inp = synth.conv_inputs(B, IC, OC, H, W, K, S, dtype=dtype, seed=seed, scale=scale,
                                     subnormal=subnormal)
        self.x = to_dev(self.inp["x"], dtype)
        self.w = to_dev(self.inp["w"], dtype)
        self.dy = to_dev(self.inp["dy"], dtype)
        self.desc = binding.make_desc(B, IC, OC, H, W, K, S, relu, TORCH_DT[dtype])

    # ---- library (C ABI) ----
    def gpu_fwd(self):
        OH, OW = binding.out_dims(self.desc)
        y = torch.empty((self.B, self.OC, OH, OW), dtype=TORCH_DT[self.dtype], device="cuda")
        binding.conv_fwd(self.desc, self.x, self.w, y)
        return y

    def gpu_dgrad(self, y):
        dx = torch.empty((self.B, self.IC, self.H, self.W), dtype=TORCH_DT[self.dtype], device="cuda")
        binding.conv_bwd_data(self.desc, self.dy, self.w, y if self.relu else None, dx)
        return dx

    def gpu_fwd_ws(self):
        """conv_fwd_ws: the forward with a caller-provided workspace (packed weights)."""
        OH, OW = binding.out_dims(self.desc)
        y = torch.empty((self.B, self.OC, OH, OW), dtype=TORCH_DT[self.dtype], device="cuda")
        ws = torch.empty(max(binding.conv_fwd_workspace_size(self.desc), 16), dtype=torch.uint8, device="cuda")
        binding.conv_fwd_ws(self.desc, self.x, self.w, None, y, ws)
        return y

    def gpu_dgrad_ws(self, y):
        dx = torch.empty((self.B, self.IC, self.H, self.W), dtype=TORCH_DT[self.dtype], device="cuda")
        ws = torch.empty(max(binding.conv_bwd_data_workspace_size(self.desc), 16), dtype=torch.uint8, device="cuda")
        binding.conv_bwd_data_ws(self.desc, self.dy, self.w, y if self.relu else None, dx, ws)
        return dx

    def gpu_wgrad(self, y):
        dw = torch.empty((self.OC, self.IC, self.K, self.K), dtype=TORCH_DT[self.dtype], device="cuda")
        n = binding.conv_bwd_filter_workspace_size(self.desc)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
        binding.conv_bwd_filter(self.desc, self.x, self.dy, y if self.relu else None, dw, ws)
        return dw

    # ---- oracle on the same inputs (mask source: the y the GPU call receives) ----
    def ref_fwd(self, samples=None):
        x = self.inp["x"] if samples is None else self.inp["x"][samples]
        return oracle.conv_fwd(x, self.inp["w"], self.S, self.relu)

    def ref_dgrad(self, y_np, samples=None):
        dy = self.inp["dy"] if samples is None else self.inp["dy"][samples]
        y = None if not self.relu else (y_np if samples is None else y_np[samples])
        return oracle.conv_bwd_data(dy, self.inp["w"], y, self.H, self.W, self.S, self.relu)

    def ref_wgrad(self, y_np, channels=None):
        dy, y = self.inp["dy"], y_np
        if channels is not None:
            dy = dy[:, channels]
            y = None if y is None else y[:, channels]
        return oracle.conv_bwd_filter(self.inp["x"], dy, y if self.relu else None, self.K, self.S,
                                      self.relu)


def check(out, ref, den, dtype, what):
    err = oracle.normalised_error(out, ref, den)
    assert err <= TOL[dtype], f"{what}: normalised error {err:.3e} > {TOL[dtype]:.0e}"
    return err
