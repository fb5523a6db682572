"""Checks that pin the fp64 oracle to facts outside itself.  Each ``pin_*``
function raises AssertionError on failure and takes ``lib`` (a build of
oracle/conv_ref.c bound with ``oracle.bind``; None = the normal build), so the
planted-mistake tests can run the same pins against a mutated oracle.

Pins, per the layer's definitions (PufferLib PR #522, layer-1/layer-2 bench
blocks) and the mathematics of a linear map:
  brute      exact agreement with an independent im2col-matrix formulation on
             small integer inputs (tests/brute.py), outputs and denominators,
             with and without the bias, and the bias gradient;
  matmul     K=1, S=1 reduces to y[b,:,p] = w[:,:,0,0] @ x[b,:,p];
  delta      a one-hot input returns the (flipped-window) kernel entries;
  adjoint    <conv(x,w), g> = <x, dgrad(g,w)> = <w, wgrad(x,g)> (and the
             ReLU-masked form of it);
  fd         central finite differences of L = <relu(conv(x,w) + bias), dy>
             in x, w and the bias;
  zero_w     with w = 0 the forward is act(bias) at every sample and position;
  shapes     the output sizes printed on the page (tests/golden), and the
             bias-gradient sizes its bias blocks print;
  unread     layer 1's input column w=14 is never read: dx is exactly 0
             there and changing x there changes nothing.
"""
import itertools
import os

import numpy as np

import oracle

from . import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _ints(rng, shape, lo=-3, hi=3):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64)


def brute_cases(n=160, seed=7):
    """Seeded subset of B in {1,2,3}, IC in {1,3}, OC in {1,2}, H,W in [K,K+5],
    K in {1,2,3,5}, S in {1,2,3}, relu in {0,1}, plus the corner cases."""
    rng = np.random.default_rng(seed)
    full = list(itertools.product([1, 2, 3], [1, 3], [1, 2], range(6), range(6),
                                  [1, 2, 3, 5], [1, 2, 3], [0, 1]))
    pick = [full[i] for i in rng.choice(len(full), size=n, replace=False)]
    corners = [(1, 1, 1, 0, 0, 5, 3, 1), (3, 3, 2, 5, 5, 5, 3, 1), (2, 3, 2, 0, 5, 3, 1, 0),
               (1, 3, 2, 5, 0, 2, 2, 1), (3, 1, 1, 3, 4, 1, 1, 0), (2, 3, 2, 1, 2, 3, 3, 1)]
    out = []
    for B, IC, OC, dh, dw, K, S, relu in pick + corners:
        out.append((B, IC, OC, K + dh, K + dw, K, S, relu))
    return out


def pin_brute(lib=None, cases=None):
    rng = np.random.default_rng(11)
    for B, IC, OC, H, W, K, S, relu in (cases or brute_cases()):
        x = _ints(rng, (B, IC, H, W))
        w = _ints(rng, (OC, IC, K, K))
        y, den = oracle.conv_fwd(x, w, S, relu, nthreads=2, lib=lib)
        yb, denb, _ = brute.fwd(x, w, S, relu)
        assert y.shape == yb.shape, (B, IC, OC, H, W, K, S, relu)
        assert np.array_equal(y, yb), ("fwd", B, IC, OC, H, W, K, S, relu)
        assert np.array_equal(den, denb), ("fwd den", B, IC, OC, H, W, K, S, relu)
        dy = _ints(rng, y.shape)
        dx, dden = oracle.conv_bwd_data(dy, w, y, H, W, S, relu, nthreads=2, lib=lib)
        dxb, ddenb = brute.dgrad(dy, w, y, H, W, S, relu)
        assert np.array_equal(dx, dxb), ("dgrad", B, IC, OC, H, W, K, S, relu)
        assert np.array_equal(dden, ddenb), ("dgrad den", B, IC, OC, H, W, K, S, relu)
        dw, wden = oracle.conv_bwd_filter(x, dy, y, K, S, relu, nthreads=2, lib=lib)
        dwb, wdenb = brute.wgrad(x, dy, y, K, S, relu)
        assert np.array_equal(dw, dwb), ("wgrad", B, IC, OC, H, W, K, S, relu)
        assert np.array_equal(wden, wdenb), ("wgrad den", B, IC, OC, H, W, K, S, relu)
        # The bias: forward with it, and its gradient (masked by the biased output).
        bias = _ints(rng, (OC,), -4, 4)
        yb_, den_ = oracle.conv_fwd(x, w, S, relu, nthreads=2, lib=lib, bias=bias)
        ybb, denbb, _ = brute.fwd(x, w, S, relu, bias=bias)
        assert np.array_equal(yb_, ybb), ("fwd bias", B, IC, OC, H, W, K, S, relu)
        assert np.array_equal(den_, denbb), ("fwd bias den", B, IC, OC, H, W, K, S, relu)
        db, bden = oracle.conv_bwd_bias(dy, yb_, relu, nthreads=2, lib=lib)
        dbb, bdenb = brute.bgrad(dy, yb_, relu)
        assert np.array_equal(db, dbb), ("bias grad", B, IC, OC, H, W, K, S, relu)
        assert np.array_equal(bden, bdenb), ("bias grad den", B, IC, OC, H, W, K, S, relu)


def pin_matmul(lib=None):
    rng = np.random.default_rng(3)
    for B, IC, OC, H, W in [(2, 5, 7, 3, 4), (1, 16, 3, 1, 1), (3, 2, 9, 5, 2)]:
        x = rng.standard_normal((B, IC, H, W))
        w = rng.standard_normal((OC, IC, 1, 1))
        y, _ = oracle.conv_fwd(x, w, 1, False, lib=lib)
        ref = np.einsum("oi,bip->bop", w[:, :, 0, 0], x.reshape(B, IC, -1)).reshape(B, OC, H, W)
        assert np.allclose(y, ref, rtol=1e-13, atol=1e-13), "1x1 stride-1 != matmul"


def pin_delta(lib=None):
    rng = np.random.default_rng(5)
    for B, IC, OC, H, W, K, S in [(2, 3, 4, 11, 15, 5, 3), (1, 2, 3, 3, 4, 3, 1), (2, 2, 2, 7, 6, 2, 2)]:
        w = rng.standard_normal((OC, IC, K, K))
        OH, OW = (H - K) // S + 1, (W - K) // S + 1
        for _ in range(6):
            b0, ic0, h0, w0 = (rng.integers(B), rng.integers(IC), rng.integers(H), rng.integers(W))
            x = np.zeros((B, IC, H, W))
            x[b0, ic0, h0, w0] = 1.0
            y, _ = oracle.conv_fwd(x, w, S, False, lib=lib)
            want = np.zeros_like(y)
            for oh in range(OH):
                for ow in range(OW):
                    kh, kw = h0 - oh * S, w0 - ow * S
                    if 0 <= kh < K and 0 <= kw < K:
                        want[b0, :, oh, ow] = w[:, ic0, kh, kw]
            assert np.array_equal(y, want), "delta input does not return the kernel"


def pin_zero_weight(lib=None):
    """w = 0 leaves only the bias: y[b, oc, p] = act(bias[oc]) exactly, den = |bias[oc]|;
    the bias gradient of an all-ones dy is then B*P where bias > 0 (relu) or everywhere."""
    rng = np.random.default_rng(17)
    for B, IC, OC, H, W, K, S in [(3, 2, 5, 11, 15, 5, 3), (2, 4, 3, 3, 4, 3, 1)]:
        x = rng.standard_normal((B, IC, H, W))
        w = np.zeros((OC, IC, K, K))
        bias = rng.standard_normal(OC)
        bias[0] = 0.0
        OH, OW = (H - K) // S + 1, (W - K) // S + 1
        for relu in (False, True):
            y, den = oracle.conv_fwd(x, w, S, relu, lib=lib, bias=bias)
            act = np.where(bias > 0, bias, 0.0) if relu else bias
            assert np.array_equal(y, np.broadcast_to(act[None, :, None, None], y.shape)), "w=0: y != act(bias)"
            assert np.array_equal(den, np.broadcast_to(np.abs(bias)[None, :, None, None], y.shape))
            db, bden = oracle.conv_bwd_bias(np.ones_like(y), y, relu, lib=lib)
            want = np.where((bias > 0) | (not relu), float(B * OH * OW), 0.0)
            assert np.array_equal(db, want) and np.array_equal(bden, want), "bias grad of ones"


def pin_adjoint(lib=None):
    rng = np.random.default_rng(9)
    for (B, IC, OC, H, W, K, S) in [(3, 4, 5, 11, 15, 5, 3), (4, 6, 5, 3, 4, 3, 1), (2, 3, 2, 9, 8, 3, 2)]:
        x = rng.standard_normal((B, IC, H, W))
        w = rng.standard_normal((OC, IC, K, K))
        for relu in (False, True):
            y, _ = oracle.conv_fwd(x, w, S, relu, lib=lib)
            dy = rng.standard_normal(y.shape)
            dx, _ = oracle.conv_bwd_data(dy, w, y, H, W, S, relu, lib=lib)
            dw, _ = oracle.conv_bwd_filter(x, dy, y, K, S, relu, lib=lib)
            lhs = float(np.sum(y * dy))
            a = float(np.sum(x * dx))
            c = float(np.sum(w * dw))
            scale = float(np.sum(np.abs(y * dy))) + 1e-300
            assert abs(lhs - a) <= 1e-12 * scale, ("adjoint <y,dy> vs <x,dx>", relu, lhs, a)
            assert abs(lhs - c) <= 1e-12 * scale, ("adjoint <y,dy> vs <w,dw>", relu, lhs, c)
            # The bias enters as a broadcast over (b, oh, ow); its adjoint is the sum
            # over them: <broadcast(v), g> = <v, bias_grad(g)> for any v.
            v = rng.standard_normal(OC)
            g = dy * (y > 0) if relu else dy
            db, _ = oracle.conv_bwd_bias(dy, y, relu, lib=lib)
            lhs = float(np.sum(v[None, :, None, None] * g))
            rhs = float(np.sum(v * db))
            scale = float(np.sum(np.abs(v[None, :, None, None] * g))) + 1e-300
            assert abs(lhs - rhs) <= 1e-12 * scale, ("adjoint of the bias broadcast", relu, lhs, rhs)


def pin_fd(lib=None):
    rng = np.random.default_rng(13)
    B, IC, OC, H, W, K, S = 2, 3, 4, 11, 15, 5, 3
    x = rng.standard_normal((B, IC, H, W))
    w = rng.standard_normal((OC, IC, K, K)) * 0.3
    dy = rng.standard_normal((B, OC, 3, 4))
    pre, _ = oracle.conv_fwd(x, w, S, False, lib=lib)
    y, _ = oracle.conv_fwd(x, w, S, True, lib=lib)
    dx, _ = oracle.conv_bwd_data(dy, w, y, H, W, S, True, lib=lib)
    dw, _ = oracle.conv_bwd_filter(x, dy, y, K, S, True, lib=lib)
    h = 1e-5

    def loss(xx, ww):
        yy, _ = oracle.conv_fwd(xx, ww, S, True, lib=lib)
        return float(np.sum(yy * dy))

    margin = np.min(np.abs(pre))
    # The loss is piecewise linear; the difference is exact while no
    # pre-activation crosses zero, which |pre| > margin >> h guarantees.
    assert margin > 1e-3, "seed gives a pre-activation too close to the ReLU kink"
    checked = 0
    for _ in range(24):
        idx = tuple(int(rng.integers(d)) for d in x.shape)
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd = (loss(xp, w) - loss(xm, w)) / (2 * h)
        assert abs(fd - dx[idx]) <= 1e-6 * (1 + abs(dx[idx])), ("fd dx", idx, fd, dx[idx])
        checked += 1
    for _ in range(24):
        idx = tuple(int(rng.integers(d)) for d in w.shape)
        wp, wm = w.copy(), w.copy()
        wp[idx] += h
        wm[idx] -= h
        fd = (loss(x, wp) - loss(x, wm)) / (2 * h)
        assert abs(fd - dw[idx]) <= 1e-6 * (1 + abs(dw[idx])), ("fd dw", idx, fd, dw[idx])
        checked += 1
    assert checked == 48
    # The bias: L(bias) = <relu(conv(x,w) + bias), dy> with its gradient from the oracle.
    bias = rng.standard_normal(OC) * 0.05
    pre_b, _ = oracle.conv_fwd(x, w, S, False, lib=lib, bias=bias)
    assert np.min(np.abs(pre_b)) > 1e-3, "seed gives a biased pre-activation too close to the kink"
    yb, _ = oracle.conv_fwd(x, w, S, True, lib=lib, bias=bias)
    db, _ = oracle.conv_bwd_bias(dy, yb, True, lib=lib)

    def loss_b(bb):
        yy, _ = oracle.conv_fwd(x, w, S, True, lib=lib, bias=bb)
        return float(np.sum(yy * dy))

    for oc in range(OC):
        bp, bm = bias.copy(), bias.copy()
        bp[oc] += h
        bm[oc] -= h
        fd = (loss_b(bp) - loss_b(bm)) / (2 * h)
        assert abs(fd - db[oc]) <= 1e-6 * (1 + abs(db[oc])), ("fd db", oc, fd, db[oc])


def printed_shapes():
    rows = []
    with open(os.path.join(GOLDEN, "pr522_layer_shapes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(tuple(int(t) for t in line.split()))
    return rows


def pin_shapes(lib=None):
    rows = printed_shapes()
    assert len(rows) == 2
    rng = np.random.default_rng(1)
    for B, IC, OC, H, W, K, S, OH, OW, relu in rows:
        assert oracle.out_dim(H, K, S) == OH and oracle.out_dim(W, K, S) == OW
        x = rng.standard_normal((2, IC, H, W))
        w = rng.standard_normal((OC, IC, K, K))
        y, _ = oracle.conv_fwd(x, w, S, relu, lib=lib)
        assert y.shape == (2, OC, OH, OW)


def pin_bias_grad_shapes(lib=None):
    """The page's bias-gradient headers name each layer's OC and OH*OW and the element
    count of the gradient; the layer shapes above must produce exactly those, and the
    oracle's bias gradient must take that gradient to one value per output channel."""
    layers = {i + 1: row for i, row in enumerate(printed_shapes())}
    rows = []
    with open(os.path.join(GOLDEN, "pr522_bias_grad_shapes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(tuple(int(t) for t in line.split()))
    assert len(rows) == 2
    rng = np.random.default_rng(19)
    for layer, B, OC, spatial, elems in rows:
        _, IC, OC_l, H, W, K, S, OH, OW, relu = layers[layer]
        OHo, OWo = oracle.out_dim(H, K, S), oracle.out_dim(W, K, S)
        assert OC == OC_l and OHo * OWo == spatial and B * OC * spatial == elems
        dy = rng.standard_normal((2, OC, OHo, OWo))
        db, _ = oracle.conv_bwd_bias(dy, None, False, lib=lib)
        assert db.shape == (OC,)


def pin_unread(lib=None):
    """Layer 1 (11x15, K=5, S=3): windows start at w = 0, 3, 6, 9 and end at 13,
    so column 14 feeds no output."""
    rng = np.random.default_rng(2)
    B, IC, OC, H, W, K, S = 2, 4, 3, 11, 15, 5, 3
    x = rng.standard_normal((B, IC, H, W))
    w = rng.standard_normal((OC, IC, K, K))
    y, _ = oracle.conv_fwd(x, w, S, True, lib=lib)
    x2 = x.copy()
    x2[..., 14] = rng.standard_normal(x2[..., 14].shape) * 100
    y2, _ = oracle.conv_fwd(x2, w, S, True, lib=lib)
    assert np.array_equal(y, y2)
    dy = rng.standard_normal(y.shape)
    for relu in (True, False):
        dx, den = oracle.conv_bwd_data(dy, w, y, H, W, S, relu, lib=lib)
        assert np.all(dx[..., 14] == 0) and np.all(den[..., 14] == 0)
    assert np.all(den[..., :14] > 0)  # without the mask every other column is reached


ALL_PINS = [pin_brute, pin_matmul, pin_delta, pin_zero_weight, pin_adjoint, pin_fd, pin_shapes,
            pin_bias_grad_shapes, pin_unread]
