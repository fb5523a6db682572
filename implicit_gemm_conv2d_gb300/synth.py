"""Seeded synthetic inputs for the conv2d layer (x, w, dy), shared by the tests,
the benchmark and the oracle checks.  This module holds random-number
generation and value formatting only: no convolution arithmetic.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: draw ``i`` of stream
``s`` is ``mix(s0 + (i + 1) * GAMMA)`` with ``s0 = mix(seed ^ (s << 32))``.
Uniforms take the top 53 bits.  Normals use the Box-Muller transform
(cosine branch), draws ``2i`` and ``2i + 1`` for element ``i``.

Distributions (the layer-1 / layer-2 workloads of PufferLib PR #522 with the
synthetic value recipe used throughout this project):
  x  ~ N(0, 1)                            stream 1
  w  ~ U(-a, a),  a = 1 / sqrt(IC*K*K)    stream 2
  dy ~ N(0, 1)                            stream 3
  bias ~ U(-a, a), the same a              stream 7 (only when asked for)
Values are rounded to fp32 (round-to-nearest-even); bf16 inputs round those
fp32 values once more to bf16 with round-to-nearest-even.  The arrays returned
are float32 holding exactly the values the layer receives in either dtype.
"""
from __future__ import annotations

import math

import numpy as np

SEED = 0x5EED2026
GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

STREAM_X, STREAM_W, STREAM_DY, STREAM_SUB_X, STREAM_SUB_W, STREAM_W2, STREAM_BIAS = 1, 2, 3, 4, 5, 6, 7


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_state(seed: int, stream: int) -> np.uint64:
    s = np.array([(seed ^ (stream << 32)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix(s)[0]


def splitmix64(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """Draws start .. start+n-1 of the given stream as uint64."""
    s0 = stream_state(seed, stream)
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(s0 + i * GAMMA)


def _u53(z: np.ndarray) -> np.ndarray:
    """[0, 1) from the top 53 bits."""
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, _CHUNK):
        m = min(_CHUNK, n - lo)
        z = splitmix64(seed, stream, 2 * lo, 2 * m)
        u1 = _u53(z[0::2]) + (1.0 / 9007199254740992.0)  # (0, 1]
        u2 = _u53(z[1::2])
        out[lo:lo + m] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return out


def uniform_pm(seed: int, stream: int, n: int, a: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, _CHUNK):
        m = min(_CHUNK, n - lo)
        out[lo:lo + m] = a * (2.0 * _u53(splitmix64(seed, stream, lo, m)) - 1.0)
    return out


def round_bf16_bits(f32: np.ndarray) -> np.ndarray:
    """IEEE-754 round-to-nearest-even from binary32 to bfloat16 (the upper 16
    bits of binary32), returned as uint16 bit patterns.  NaN stays NaN."""
    b = np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(f32)
    if np.any(nan):
        r[nan] = ((b[nan] >> np.uint32(16)) | np.uint32(0x40)).astype(np.uint16)
    return r


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_dtype_values(v64: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 draws -> float32 array holding exactly the values of ``dtype``."""
    f32 = v64.astype(np.float32)
    if dtype == "f32":
        return f32
    if dtype == "bf16":
        return bf16_bits_to_f32(round_bf16_bits(f32))
    raise ValueError(f"unknown dtype {dtype!r}")


def plant_subnormals(f32: np.ndarray, seed: int, stream: int, frac: float = 0.01) -> np.ndarray:
    """Replace a seeded ``frac`` of the entries by +-2**u, u uniform over the
    integers in [-149, -127) (binary32 subnormals)."""
    flat = f32.reshape(-1).copy()
    n = flat.size
    for lo in range(0, n, _CHUNK):
        m = min(_CHUNK, n - lo)
        z = splitmix64(seed, stream, 3 * lo, 3 * m)
        sel = _u53(z[0::3]) < frac
        neg = (z[1::3] >> np.uint64(63)) == 1
        e = -149 + np.floor(_u53(z[2::3]) * 22.0).astype(np.int64)
        val = np.ldexp(np.where(neg, -1.0, 1.0), e).astype(np.float32)
        seg = flat[lo:lo + m]
        seg[sel] = val[sel]
    return flat.reshape(f32.shape)


def out_hw(H: int, W: int, K: int, S: int) -> tuple[int, int]:
    """Output spatial size (no padding): floor((n - K) / S) + 1 per axis."""
    return (H - K) // S + 1, (W - K) // S + 1


def conv_inputs(B: int, IC: int, OC: int, H: int, W: int, K: int, S: int, dtype: str = "f32",
                seed: int = SEED, scale: float = 1.0, subnormal: bool = False,
                w_stream: int = STREAM_W, need=("x", "w", "dy")) -> dict:
    """Seeded x (B,IC,H,W), w (OC,IC,K,K), dy (B,OC,OH,OW) as float32 arrays
    holding values exact in ``dtype``.  ``scale`` multiplies x and w before
    rounding; ``subnormal`` plants binary32 subnormals in x and w (before the
    bf16 rounding, which flushes the smallest of them to zero)."""
    OH, OW = out_hw(H, W, K, S)
    out = {}
    if "x" in need:
        x = normal(seed, STREAM_X, B * IC * H * W) * scale
        xf = x.astype(np.float32).reshape(B, IC, H, W)
        if subnormal:
            xf = plant_subnormals(xf, seed, STREAM_SUB_X)
        out["x"] = xf if dtype == "f32" else to_dtype_values(xf.astype(np.float64), dtype)
    if "w" in need:
        a = 1.0 / math.sqrt(IC * K * K)
        w = uniform_pm(seed, w_stream, OC * IC * K * K, a) * scale
        wf = w.astype(np.float32).reshape(OC, IC, K, K)
        if subnormal:
            wf = plant_subnormals(wf, seed, STREAM_SUB_W)
        out["w"] = wf if dtype == "f32" else to_dtype_values(wf.astype(np.float64), dtype)
    if "dy" in need:
        dy = normal(seed, STREAM_DY, B * OC * OH * OW)
        out["dy"] = to_dtype_values(dy, dtype).reshape(B, OC, OH, OW)
    if "bias" in need:
        a = 1.0 / math.sqrt(IC * K * K)
        out["bias"] = to_dtype_values(uniform_pm(seed, STREAM_BIAS, OC, a) * scale, dtype)
    return out
