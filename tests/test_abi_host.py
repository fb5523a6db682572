"""The C ABI on the host (no GPU needed): the library builds and loads,
exports every function include/conv.h declares, validates arguments before
touching CUDA, and its fast-divmod routine matches '/' and '%' exhaustively
for the divisors the two layers use."""
import concurrent.futures as cf
import ctypes
import os
import re

import pytest

from implicit_gemm_conv2d_gb300 import binding, build

from . import oracle_pins

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "conv.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(conv_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/conv.h but not exported"
    assert sorted(binding.EXPORTS) == names


def test_version_and_status_strings(L):
    assert binding.conv_version().count(".") == 2
    for code in range(-6, 1):
        assert binding.status_string(code).startswith("CONV_")
    assert binding.status_string(-99) == "unknown conv status"


def desc(**kw):
    base = dict(B=1024, IC=59, OC=128, H=11, W=15, K=5, S=3, relu=1, dtype=0)
    base.update(kw)
    return binding.ConvDesc(*(base[k] for k in ("B", "IC", "OC", "H", "W", "K", "S", "relu", "dtype")))


def test_out_dims_match_printed_shapes(L):
    for B, IC, OC, H, W, K, S, OH, OW, relu in oracle_pins.printed_shapes():
        d = desc(B=B, IC=IC, OC=OC, H=H, W=W, K=K, S=S, relu=relu)
        assert binding.out_dims(d) == (OH, OW)


@pytest.mark.parametrize("bad", [dict(H=4), dict(W=4), dict(K=0), dict(S=0), dict(IC=0), dict(OC=0),
                                 dict(B=-1), dict(relu=2), dict(dtype=7)])
def test_invalid_descriptor(L, bad):
    d = desc(**bad)
    fake = ctypes.c_void_p(0x1000)
    assert L.conv_fwd(ctypes.byref(d), fake, fake, fake, None) == -2
    assert L.conv_bwd_data(ctypes.byref(d), fake, fake, fake, fake, None) == -2
    assert L.conv_bwd_filter(ctypes.byref(d), fake, fake, fake, fake, fake, 1 << 30, None) == -2
    assert L.conv_bwd_filter_workspace_size(ctypes.byref(d)) == 0
    assert L.conv_fwd_bias(ctypes.byref(d), fake, fake, fake, fake, None) == -2
    assert L.conv_bwd_bias(ctypes.byref(d), fake, fake, fake, None) == -2
    assert L.conv_fwd_ws(ctypes.byref(d), fake, fake, None, fake, fake, 1 << 30, None) == -2
    assert L.conv_bwd_data_ws(ctypes.byref(d), fake, fake, fake, fake, fake, 1 << 30, None) == -2
    assert L.conv_bwd_filter_bias(ctypes.byref(d), fake, fake, fake, fake, fake, fake, 1 << 30, None) == -2
    assert L.conv_fwd_chain2(ctypes.byref(d), ctypes.byref(d), fake, fake, None, fake, None, fake, fake, fake,
                             1 << 30, None) == -2
    assert L.conv_fwd_chain2_workspace_size(ctypes.byref(d), ctypes.byref(d)) == 0
    assert L.conv_bwd_chain2(ctypes.byref(d), ctypes.byref(d), *([fake] * 11), fake, 1 << 30, None) == -2
    assert L.conv_bwd_chain2_workspace_size(ctypes.byref(d), ctypes.byref(d)) == 0
    assert L.conv_bwd(ctypes.byref(d), fake, fake, fake, fake, fake, fake, None, fake, 1 << 30, None) == -2
    assert L.conv_bwd_workspace_size(ctypes.byref(d)) == 0
    assert L.conv_fwd_workspace_size(ctypes.byref(d)) == 0
    assert L.conv_bwd_data_workspace_size(ctypes.byref(d)) == 0
    oh, ow = ctypes.c_int32(), ctypes.c_int32()
    assert L.conv_out_dims(ctypes.byref(d), ctypes.byref(oh), ctypes.byref(ow)) == -2


def test_too_large_for_int32_indexing(L):
    d = desc(B=16384 * 14)  # 2.2e9 input elements
    fake = ctypes.c_void_p(0x1000)
    assert L.conv_fwd(ctypes.byref(d), fake, fake, fake, None) == -3


def test_null_and_alignment_checked_before_cuda(L):
    d = desc()
    ok, odd = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1008)
    assert L.conv_fwd(None, ok, ok, ok, None) == -1
    assert L.conv_fwd(ctypes.byref(d), None, ok, ok, None) == -1
    assert L.conv_fwd(ctypes.byref(d), ok, ok, None, None) == -1
    assert L.conv_fwd(ctypes.byref(d), ok, odd, ok, None) == -4
    assert L.conv_bwd_data(ctypes.byref(d), ok, ok, None, ok, None) == -1  # relu needs y
    assert L.conv_bwd_data(ctypes.byref(d), ok, ok, odd, ok, None) == -4
    assert L.conv_bwd_filter(ctypes.byref(d), ok, ok, None, ok, ok, 1 << 30, None) == -1
    assert L.conv_bwd_filter(ctypes.byref(d), ok, ok, ok, odd, ok, 1 << 30, None) == -4
    assert L.conv_bwd_filter(ctypes.byref(d), ok, ok, ok, ok, odd, 1 << 30, None) == -4
    d0 = desc(relu=0)
    assert L.conv_bwd_data(ctypes.byref(d0), ok, ok, None, None, None) == -1
    # The bias entry points.
    assert L.conv_fwd_bias(ctypes.byref(d), ok, ok, None, ok, None) == -1   # bias required
    assert L.conv_fwd_bias(ctypes.byref(d), ok, ok, odd, ok, None) == -4
    assert L.conv_fwd_bias(ctypes.byref(d), None, ok, ok, ok, None) == -1
    assert L.conv_bwd_bias(None, ok, ok, ok, None) == -1
    assert L.conv_bwd_bias(ctypes.byref(d), ok, ok, None, None) == -1      # db required
    assert L.conv_bwd_bias(ctypes.byref(d), ok, None, ok, None) == -1      # relu needs y
    assert L.conv_bwd_bias(ctypes.byref(d), None, ok, ok, None) == -1
    assert L.conv_bwd_bias(ctypes.byref(d), ok, ok, odd, None) == -4
    assert L.conv_bwd_bias(ctypes.byref(d), odd, ok, ok, None) == -4
    assert L.conv_bwd_bias(ctypes.byref(d), ok, odd, ok, None) == -4
    # The fused backward: dw and w required, y with relu, everything aligned.
    assert L.conv_bwd(ctypes.byref(d), ok, ok, ok, ok, ok, None, None, ok, 1 << 30, None) == -1
    assert L.conv_bwd(ctypes.byref(d), ok, ok, ok, None, ok, ok, None, ok, 1 << 30, None) == -1
    assert L.conv_bwd(ctypes.byref(d), ok, ok, ok, ok, ok, ok, odd, ok, 1 << 30, None) == -4
    assert L.conv_bwd(ctypes.byref(d), ok, ok, ok, ok, odd, ok, None, ok, 1 << 30, None) == -4
    # The fused weight + bias gradients: db required and aligned.
    assert L.conv_bwd_filter_bias(ctypes.byref(d), ok, ok, ok, ok, None, ok, 1 << 30, None) == -1
    assert L.conv_bwd_filter_bias(ctypes.byref(d), ok, ok, ok, ok, odd, ok, 1 << 30, None) == -4
    assert L.conv_bwd_filter_bias(ctypes.byref(d), ok, ok, None, ok, ok, ok, 1 << 30, None) == -1  # relu needs y
    # The workspace-taking forward / d_input: the same checks, plus the workspace's alignment.
    assert L.conv_fwd_ws(ctypes.byref(d), None, ok, None, ok, ok, 1 << 30, None) == -1
    assert L.conv_fwd_ws(ctypes.byref(d), ok, ok, None, ok, odd, 1 << 30, None) == -4
    assert L.conv_fwd_ws(ctypes.byref(d), ok, ok, odd, ok, ok, 1 << 30, None) == -4
    assert L.conv_bwd_data_ws(ctypes.byref(d), ok, ok, None, ok, ok, 1 << 30, None) == -1  # relu needs y
    assert L.conv_bwd_data_ws(ctypes.byref(d), ok, ok, ok, ok, odd, 1 << 30, None) == -4


def test_chain_descriptors_checked_before_cuda(L):
    d1 = desc()
    d2 = desc(IC=128, H=3, W=4, K=3, S=1, relu=0)
    ok = ctypes.c_void_p(0x1000)
    fake = ctypes.c_void_p(0x1000)
    # layer 2's input must be layer 1's output
    for bad in (desc(IC=64, H=3, W=4, K=3, S=1), desc(IC=128, H=4, W=4, K=3, S=1), desc(B=7, IC=128, H=3, W=4, K=3, S=1),
                desc(IC=128, H=3, W=4, K=3, S=1, dtype=1)):
        assert L.conv_fwd_chain2(ctypes.byref(d1), ctypes.byref(bad), fake, fake, None, fake, None, fake, fake, fake,
                                 1 << 30, None) == -2
    assert L.conv_fwd_chain2(None, ctypes.byref(d2), ok, ok, None, ok, None, ok, ok, ok, 1 << 30, None) == -1
    assert L.conv_fwd_chain2(ctypes.byref(d1), ctypes.byref(d2), None, ok, None, ok, None, ok, ok, ok, 1 << 30,
                             None) == -1
    odd = ctypes.c_void_p(0x1008)
    assert L.conv_fwd_chain2(ctypes.byref(d1), ctypes.byref(d2), ok, ok, None, ok, None, ok, odd, ok, 1 << 30,
                             None) == -4
    # the backward chain: the same descriptor check, then the required pointers
    for bad in (desc(IC=64, H=3, W=4, K=3, S=1), desc(B=7, IC=128, H=3, W=4, K=3, S=1)):
        assert L.conv_bwd_chain2(ctypes.byref(d1), ctypes.byref(bad), *([fake] * 11), fake, 1 << 30, None) == -2
        assert L.conv_bwd_chain2_workspace_size(ctypes.byref(d1), ctypes.byref(bad)) == 0
    args = [ok] * 11  # x1 w1 y1 w2 y2 dy2 dx1 dw1 db1 dw2 db2
    for i in (1, 2, 3, 5, 7, 9):  # w1, y1, w2, dy2, dw1, dw2 are required
        a = list(args)
        a[i] = None
        assert L.conv_bwd_chain2(ctypes.byref(d1), ctypes.byref(d2), *a, ok, 1 << 30, None) == -1, i
    assert L.conv_bwd_chain2(ctypes.byref(d1), ctypes.byref(d2), *args, odd, 1 << 30, None) == -4


def test_empty_batch_is_a_no_op(L):
    d = desc(B=0)
    assert L.conv_fwd(ctypes.byref(d), None, None, None, None) == 0
    assert L.conv_bwd_data(ctypes.byref(d), None, None, None, None, None) == 0
    assert L.conv_fwd_bias(ctypes.byref(d), None, None, None, None, None) == 0
    assert L.conv_bwd_bias(ctypes.byref(d), None, None, None, None) == -1  # db is still written


def test_wait_selftest_arguments_checked_before_cuda(L):
    assert L.conv_wait_selftest(0, None) == -3
    assert L.conv_wait_selftest(1000001, None) == -3


def test_set_algo_validation(L):
    assert L.conv_set_algo(6, 0) == -3
    assert L.conv_set_algo(4, 0) == 0   # the workspace-taking forward shares the forward's choice
    assert L.conv_set_algo(5, 0) == 0   # ... and d_input's
    assert L.conv_set_algo(-1, 0) == -3
    assert L.conv_set_algo(0, 9) == -3
    assert L.conv_set_algo(0, 0) == 0
    # The bias gradient has the column-sum kernel (auto) and the direct kernel only.
    assert L.conv_set_algo(3, 2) == -3
    assert L.conv_set_algo(3, 3) == -3
    assert L.conv_set_algo(3, 1) == 0
    assert L.conv_set_algo(3, 0) == 0


# Divisors the two layers use: P, OW, K*K, K, W, H*W and IC*K*K for
# layer 1 (11x15, K5, S3 -> 3x4) and layer 2 (3x4, K3, S1 -> 1x2).
LAYER_DIVISORS = sorted({12, 4, 25, 5, 15, 165, 1475, 2, 9, 3, 1152, 1})


def test_fastdivmod_exhaustive_for_layer_divisors(L):
    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        jobs = {d: ex.submit(binding.conv_fastdivmod_check, d, 0, 1 << 31) for d in LAYER_DIVISORS}
        for d, j in jobs.items():
            assert j.result() == 0, f"fast divmod wrong for divisor {d}"


def test_fastdivmod_random_divisors(L):
    import numpy as np
    rng = np.random.default_rng(0)
    divs = list(rng.integers(1, 1 << 31, size=300)) + [2**k for k in range(31)] + [2**k + 1 for k in range(1, 31)] \
        + [2**k - 1 for k in range(2, 32)]
    for d in divs:
        d = int(min(d, (1 << 31) - 1))
        lo = int(rng.integers(0, (1 << 31) - 20000))
        assert binding.conv_fastdivmod_check(d, lo, lo + 20000) == 0, d
        assert binding.conv_fastdivmod_check(d, (1 << 31) - 20000, 1 << 31) == 0, d
        assert binding.conv_fastdivmod_check(d, 0, 2000) == 0, d
    assert binding.conv_fastdivmod_check(0, 0, 10) == 2**64 - 1
