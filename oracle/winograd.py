"""Winograd minimal filtering, F(m, r) and F(m x m, r x r), in exact rationals
and fp64 — TEST INFRASTRUCTURE (an oracle for a Winograd convolution path).

Method ("im2col Expansion, FFT Convolution, and Winograd Transforms",
Winograd section; openCNN, Sec. 2-3): an m-output, r-tap correlation over a
window of n = m + r - 1 inputs is computed with n multiplications as

    y = A^T [ (G g) * (B^T d) ]            (* elementwise)

and in two dimensions, per m x m output tile of an n x n input tile,

    Y = A^T [ (G g G^T) * (B^T d B) ] A.

The matrices are not typed in: they come from the Toom-Cook construction on
n - 1 finite interpolation points and the point at infinity.  Toom-Cook
computes the linear convolution c = a (*) g of a length-m and a length-r
sequence as c = C [(V_g g) * (V_a a)], with V_a, V_g the evaluation matrices
(rows p^0, p^1, ... per finite point; the leading coefficient for infinity)
and C the inverse of the n x n evaluation matrix.  Correlation is the
transpose of that map in a (y = T_g^T d where c = T_g a), hence A^T = V_a^T,
G = V_g, B^T = C^T.  A diagonal rescaling moves every fraction of B^T into G,
leaving B^T and A^T integral (as the pages describe: small-integer input and
output transforms, the fractions in the filter transform).

Nothing here is used by the product library.
"""
from __future__ import annotations

from fractions import Fraction
from math import lcm

import numpy as np

INF = None   # the point at infinity


def default_points(m: int, r: int) -> list:
    """0, 1, -1, 2, -2, ... (n - 1 finite points) and infinity."""
    n = m + r - 1
    pts = [Fraction(0)]
    k = 1
    while len(pts) < n - 1:
        pts.append(Fraction(k))
        if len(pts) < n - 1:
            pts.append(Fraction(-k))
        k += 1
    return pts + [INF]


def _eval_matrix(points, cols):
    """Rows: finite point p -> (p^0 .. p^(cols-1)); infinity -> leading coefficient."""
    out = []
    for p in points:
        if p is INF:
            out.append([Fraction(0)] * (cols - 1) + [Fraction(1)])
        else:
            out.append([p ** k for k in range(cols)])
    return out


def _inverse(mat):
    """Exact Gauss-Jordan inverse of a square Fraction matrix."""
    n = len(mat)
    a = [row[:] + [Fraction(int(i == j)) for j in range(n)] for i, row in enumerate(mat)]
    for col in range(n):
        piv = next(i for i in range(col, n) if a[i][col] != 0)
        a[col], a[piv] = a[piv], a[col]
        pv = a[col][col]
        a[col] = [v / pv for v in a[col]]
        for i in range(n):
            if i != col and a[i][col] != 0:
                f = a[i][col]
                a[i] = [vi - f * vc for vi, vc in zip(a[i], a[col])]
    return [row[n:] for row in a]


def transforms(m: int, r: int, points=None):
    """(A^T, G, B^T) for F(m, r) as lists of Fractions: A^T is m x n, G is n x r,
    B^T is n x n, with B^T and A^T integral."""
    n = m + r - 1
    pts = default_points(m, r) if points is None else list(points)
    if len(pts) != n or sum(p is INF for p in pts) != 1:
        raise ValueError("need n - 1 distinct finite points and infinity")
    v_full = _eval_matrix(pts, n)         # evaluation of a degree n-1 polynomial
    c = _inverse(v_full)                  # interpolation
    v_a = _eval_matrix(pts, m)            # n x m
    g = _eval_matrix(pts, r)              # n x r
    at = [[v_a[j][i] for j in range(n)] for i in range(m)]       # m x n
    bt = [[c[j][i] for j in range(n)] for i in range(n)]         # C^T
    # Move each row's denominators of B^T into the matching row of G.
    for j in range(n):
        s = lcm(*[v.denominator for v in bt[j]])
        if s != 1:
            bt[j] = [v * s for v in bt[j]]
            g[j] = [v / s for v in g[j]]
    return at, g, bt


def correlate_1d(d, g, m: int, r: int, points=None):
    """F(m, r) on one window: y[i] = sum_k d[i+k] g[k] for i < m, exact when d
    and g are Fractions or integers."""
    at, gm, bt = transforms(m, r, points)
    n = m + r - 1
    u = [sum(gm[j][k] * g[k] for k in range(r)) for j in range(n)]
    v = [sum(bt[j][i] * d[i] for i in range(n)) for j in range(n)]
    w = [u[j] * v[j] for j in range(n)]
    return [sum(at[i][j] * w[j] for j in range(n)) for i in range(m)]


def _np(mat):
    return np.array([[float(v) for v in row] for row in mat], dtype=np.float64)


def conv2d_winograd(x: np.ndarray, w: np.ndarray, pad: int, m: int = 2) -> np.ndarray:
    """Stride-1 3x3 (any r x r) cross-correlation with zero padding `pad` by
    F(m x m, r x r) tiles, in fp64.  x: [N][Ci][H][W], w: [Co][Ci][r][r].

    Steps per image n and output channel co: for every m x m output tile, the
    n x n input tile d (zero outside the image) of each input channel is
    transformed (B^T d B), multiplied elementwise by the transformed filter
    (G g G^T) of that channel, the products are summed over input channels,
    and the sum is transformed back (A^T . A).  Tiles past the output's edge
    are computed on zero input and cropped."""
    N, Ci, H, W = x.shape
    Co, Ci2, r, r2 = w.shape
    if Ci2 != Ci or r != r2:
        raise ValueError("filter shape")
    Ho, Wo = H + 2 * pad - r + 1, W + 2 * pad - r + 1
    if Ho < 1 or Wo < 1:
        raise ValueError("empty output")
    at, gm, bt = (_np(t) for t in transforms(m, r))
    n = m + r - 1
    th, tw = -(-Ho // m), -(-Wo // m)                     # tiles per column / row
    # Zero-padded input large enough for every tile's n x n window.
    xp = np.zeros((N, Ci, th * m + r - 1, tw * m + r - 1), dtype=np.float64)
    xp[:, :, pad:pad + H, pad:pad + W] = x
    u = np.einsum("ak,oikl,bl->oiab", gm, w.astype(np.float64), gm)        # G g G^T: [Co][Ci][n][n]
    y = np.zeros((N, Co, th * m, tw * m), dtype=np.float64)
    for ty in range(th):
        for tx in range(tw):
            d = xp[:, :, ty * m:ty * m + n, tx * m:tx * m + n]             # [N][Ci][n][n]
            v = np.einsum("ak,zikl,bl->ziab", bt, d, bt)                   # B^T d B
            mprod = np.einsum("oiab,ziab->zoab", u, v)                     # sum over Ci
            y[:, :, ty * m:ty * m + m, tx * m:tx * m + m] = np.einsum("pa,zoab,qb->zopq", at, mprod, at)
    return y[:, :, :Ho, :Wo]
