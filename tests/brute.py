"""Independent second formulation of the conv2d layer, used only to pin the
oracle: the patch matrix (im2col) is materialised by strided slicing and
multiplied with numpy matmul; d_input scatters the patch-matrix gradient back
by the transpose of the same slicing; the bias rides in the matmul as a row of
ones, and its gradient is a product with vectors of ones.  No loop order, index formula or helper
is shared with oracle/conv_ref.c.
"""
import numpy as np


def out_hw(H, W, K, S):
    return (H - K) // S + 1, (W - K) // S + 1


def patches(x, K, S):
    """Xcol[b, ic*K*K + kh*K + kw, oh*OW + ow] = x[b, ic, oh*S + kh, ow*S + kw]."""
    B, IC, H, W = x.shape
    OH, OW = out_hw(H, W, K, S)
    cols = np.empty((B, IC, K, K, OH, OW), dtype=np.float64)
    for kh in range(K):
        for kw in range(K):
            cols[:, :, kh, kw] = x[:, :, kh:kh + S * (OH - 1) + 1:S, kw:kw + S * (OW - 1) + 1:S]
    return cols.reshape(B, IC * K * K, OH * OW)


def unpatch(cols, IC, H, W, K, S):
    """Adjoint of ``patches``: sum every patch-matrix entry back onto its pixel."""
    B = cols.shape[0]
    OH, OW = out_hw(H, W, K, S)
    c = cols.reshape(B, IC, K, K, OH, OW)
    dx = np.zeros((B, IC, H, W), dtype=np.float64)
    for kh in range(K):
        for kw in range(K):
            dx[:, :, kh:kh + S * (OH - 1) + 1:S, kw:kw + S * (OW - 1) + 1:S] += c[:, :, kh, kw]
    return dx


def fwd(x, w, S, relu, bias=None):
    """With a bias, the patch matrix gets an extra row of ones and the weight
    matrix an extra column holding the bias, so the bias rides in the matmul."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    B, IC, H, W = x.shape
    OC, _, K, _ = w.shape
    OH, OW = out_hw(H, W, K, S)
    cols = patches(x, K, S)
    wm = w.reshape(OC, -1)
    if bias is not None:
        cols = np.concatenate([cols, np.ones((B, 1, OH * OW))], axis=1)
        wm = np.concatenate([wm, np.asarray(bias, np.float64).reshape(OC, 1)], axis=1)
    pre = np.matmul(wm, cols).reshape(B, OC, OH, OW)
    den = np.matmul(np.abs(wm), np.abs(cols)).reshape(B, OC, OH, OW)
    y = np.where(pre > 0, pre, 0.0) if relu else pre
    return y, den, pre


def grad_in(dy, y, relu):
    dy = np.asarray(dy, np.float64)
    return dy * (np.asarray(y) > 0) if relu else dy


def dgrad(dy, w, y, H, W, S, relu):
    g = grad_in(dy, y, relu)
    w = np.asarray(w, np.float64)
    OC, IC, K, _ = w.shape
    B = g.shape[0]
    gm = g.reshape(B, OC, -1)
    wm = w.reshape(OC, -1)
    dx = unpatch(np.matmul(wm.T, gm), IC, H, W, K, S)
    den = unpatch(np.matmul(np.abs(wm).T, np.abs(gm)), IC, H, W, K, S)
    return dx, den


def wgrad(x, dy, y, K, S, relu):
    g = grad_in(dy, y, relu)
    x = np.asarray(x, np.float64)
    B, OC = g.shape[:2]
    IC = x.shape[1]
    cols = patches(x, K, S)
    gm = g.reshape(B, OC, -1)
    dw = np.matmul(gm, cols.transpose(0, 2, 1)).sum(axis=0)
    den = np.matmul(np.abs(gm), np.abs(cols).transpose(0, 2, 1)).sum(axis=0)
    return dw.reshape(OC, IC, K, K), den.reshape(OC, IC, K, K)


def bgrad(dy, y, relu):
    """db[oc] = 1_B^T (G 1_P): both contractions as matmuls with vectors of ones."""
    g = grad_in(dy, y, relu)
    B, OC = g.shape[:2]
    gm = g.reshape(B, OC, -1)
    onesp = np.ones(gm.shape[2])
    onesb = np.ones(B)
    db = np.matmul(onesb, np.matmul(gm, onesp))
    den = np.matmul(onesb, np.matmul(np.abs(gm), onesp))
    return db, den
