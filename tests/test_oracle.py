"""The fp64 oracle against its pins (CPU only).  See tests/oracle_pins.py for
what each pin checks and why it is independent of the oracle."""
import numpy as np
import pytest

import oracle

from . import oracle_pins as pins


def test_brute_force_small_shapes():
    pins.pin_brute()


def test_1x1_stride1_is_matmul():
    pins.pin_matmul()


def test_delta_input_returns_kernel():
    pins.pin_delta()


def test_zero_weight_leaves_bias():
    pins.pin_zero_weight()


def test_adjoint_identity():
    pins.pin_adjoint()


def test_finite_differences():
    pins.pin_fd()


def test_printed_output_sizes():
    pins.pin_shapes()


def test_printed_bias_grad_sizes():
    pins.pin_bias_grad_shapes()


def test_layer1_column14_unread():
    pins.pin_unread()


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((9, 5, 11, 15))
    w = rng.standard_normal((6, 5, 5, 5))
    y1, d1 = oracle.conv_fwd(x, w, 3, True, nthreads=1)
    y7, d7 = oracle.conv_fwd(x, w, 3, True, nthreads=7)
    assert y1.tobytes() == y7.tobytes() and d1.tobytes() == d7.tobytes()
    dy = rng.standard_normal(y1.shape)
    a = oracle.conv_bwd_data(dy, w, y1, 11, 15, 3, True, nthreads=1)
    b = oracle.conv_bwd_data(dy, w, y1, 11, 15, 3, True, nthreads=5)
    assert a[0].tobytes() == b[0].tobytes()
    a = oracle.conv_bwd_filter(x, dy, y1, 5, 3, True, nthreads=1)
    b = oracle.conv_bwd_filter(x, dy, y1, 5, 3, True, nthreads=4)
    assert a[0].tobytes() == b[0].tobytes()


def test_relu_semantics():
    """y = acc if acc > 0 else +0; the backward mask is y > 0, so a zero output
    passes no gradient."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal((3, 2, 5, 5))
    w = rng.standard_normal((4, 2, 3, 3))
    pre, _ = oracle.conv_fwd(x, w, 1, False)
    y, _ = oracle.conv_fwd(x, w, 1, True)
    assert np.array_equal(y, np.where(pre > 0, pre, 0.0))
    assert not np.any(np.signbit(y))
    dy = np.ones_like(y)
    dw_masked, _ = oracle.conv_bwd_filter(x, dy, y, 3, 1, True)
    dw_by_hand, _ = oracle.conv_bwd_filter(x, dy * (y > 0), None, 3, 1, False)
    assert np.array_equal(dw_masked, dw_by_hand)


def test_denominator_bounds_output():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((2, 3, 7, 7))
    w = rng.standard_normal((5, 3, 3, 3))
    y, den = oracle.conv_fwd(x, w, 2, False)
    assert np.all(np.abs(y) <= den * (1 + 1e-15))


def test_normalised_error_helper():
    ref = np.array([1.0, 0.0, 2.0])
    den = np.array([2.0, 0.0, 4.0])
    assert oracle.normalised_error(np.array([1.5, 0.0, 2.0]), ref, den) == 0.25
    assert oracle.normalised_error(np.array([1.0, 1e-30, 2.0]), ref, den) == float("inf")


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.conv_fwd(np.zeros((1, 1, 2, 2)), np.zeros((1, 1, 3, 3)), 1, False)
