"""ctypes wrapper around the fp64 C oracle (``conv_ref.c``) — TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU baseline use this.
The product library never imports it, and it imports nothing from the
product.  All arrays are float64 numpy arrays in NCHW / [Co][Ci][Kh][Kw]
order; inputs must already hold the exact values the GPU consumes.

``build()`` compiles ``conv_ref.c`` with gcc (no fast-math, no FMA
contraction, so results do not depend on the host ISA) into
``oracle/_build/liboracle_conv.so``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_conv.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle shared library if it is missing or stale."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                        "-ffp-contract=off", "-fno-fast-math",
                        _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            i64p = ctypes.POINTER(ctypes.c_int64)
            ci = ctypes.c_int
            L.oracle_out_dims.argtypes = [ci] * 6 + [ip, ip]
            L.oracle_conv2d_direct_slice.argtypes = [dp, dp, dp, dp] + [ci] * 13
            L.oracle_conv2d_direct.argtypes = [dp, dp, dp, dp] + [ci] * 9
            L.oracle_conv2d_points.argtypes = [dp, dp, i64p, ctypes.c_int64, dp, dp] + [ci] * 9
            L.oracle_im2col.argtypes = [dp, dp] + [ci] * 7
            L.oracle_gemm_naive.argtypes = [dp, dp, dp, ci, ci, ci]
            L.oracle_gemm_naive.restype = None
            L.oracle_conv2d_im2col.argtypes = [dp, dp, dp, dp] + [ci] * 9
            L.oracle_im2win_transform.argtypes = [dp, dp] + [ci] * 8
            L.oracle_im2win_conv.argtypes = [dp, dp, dp] + [ci] * 9
            L.oracle_add_bias.argtypes = [dp, dp, dp] + [ci] * 4
            for f in ("oracle_out_dims", "oracle_conv2d_direct_slice", "oracle_conv2d_direct",
                      "oracle_conv2d_points", "oracle_im2col", "oracle_conv2d_im2col",
                      "oracle_im2win_transform", "oracle_im2win_conv", "oracle_add_bias"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def out_dims(H, W, Kh, Kw, s, p):
    ho, wo = ctypes.c_int(), ctypes.c_int()
    rc = lib().oracle_out_dims(H, W, Kh, Kw, s, p, ctypes.byref(ho), ctypes.byref(wo))
    if rc != 0:
        raise ValueError("no output window fits")
    return ho.value, wo.value


def conv2d(X, Wt, stride=1, pad=0, with_abs=True):
    """Direct 7-loop.  Returns (Y, S) with S = sum |x*w| (or (Y, None))."""
    X, Wt = _f64(X), _f64(Wt)
    N, Ci, H, W = X.shape
    Co, Ci2, Kh, Kw = Wt.shape
    assert Ci == Ci2
    Ho, Wo = out_dims(H, W, Kh, Kw, stride, pad)
    Y = np.empty((N, Co, Ho, Wo))
    S = np.empty_like(Y) if with_abs else None
    rc = lib().oracle_conv2d_direct(_p(X), _p(Wt), _p(Y), _p(S) if with_abs else None,
                                    N, Ci, H, W, Co, Kh, Kw, stride, pad)
    assert rc == 0
    return Y, S


def conv2d_slice(X, Wt, Y, S, stride, pad, n0, n1, co0, co1):
    """Fill the (n, co) slice of preallocated Y, S (releases the GIL)."""
    N, Ci, H, W = X.shape
    Co, _, Kh, Kw = Wt.shape
    rc = lib().oracle_conv2d_direct_slice(_p(X), _p(Wt), _p(Y), _p(S), N, Ci, H, W, Co,
                                          Kh, Kw, stride, pad, n0, n1, co0, co1)
    assert rc == 0


def conv2d_points(X, Wt, flat_idx, stride=1, pad=0):
    """Outputs at flat NCHW indices.  Returns (y, s) 1-D arrays."""
    X, Wt = _f64(X), _f64(Wt)
    N, Ci, H, W = X.shape
    Co, _, Kh, Kw = Wt.shape
    idx = np.ascontiguousarray(np.asarray(flat_idx, dtype=np.int64))
    y = np.empty(idx.shape[0])
    s = np.empty(idx.shape[0])
    rc = lib().oracle_conv2d_points(_p(X), _p(Wt),
                                    idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                    idx.shape[0], _p(y), _p(s),
                                    N, Ci, H, W, Co, Kh, Kw, stride, pad)
    if rc != 0:
        raise ValueError(f"oracle_conv2d_points failed ({rc})")
    return y, s


def im2col(Xn, Kh, Kw, stride=1, pad=0):
    Xn = _f64(Xn)
    Ci, H, W = Xn.shape
    Ho, Wo = out_dims(H, W, Kh, Kw, stride, pad)
    cols = np.empty((Ci * Kh * Kw, Ho * Wo))
    assert lib().oracle_im2col(_p(Xn), _p(cols), Ci, H, W, Kh, Kw, stride, pad) == 0
    return cols


def gemm(A, B):
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    C = np.empty((M, N))
    lib().oracle_gemm_naive(_p(A), _p(B), _p(C), M, N, K)
    return C


def conv2d_im2col(X, Wt, stride=1, pad=0):
    X, Wt = _f64(X), _f64(Wt)
    N, Ci, H, W = X.shape
    Co, _, Kh, Kw = Wt.shape
    Ho, Wo = out_dims(H, W, Kh, Kw, stride, pad)
    Y = np.empty((N, Co, Ho, Wo))
    cols = np.empty(Ci * Kh * Kw * Ho * Wo)
    assert lib().oracle_conv2d_im2col(_p(X), _p(Wt), _p(Y), _p(cols),
                                      N, Ci, H, W, Co, Kh, Kw, stride, pad) == 0
    return Y


def im2win_transform(X, Kh, Kw, stride=1, pad=0):
    """Eq. (2) strips: shape (N, Ci, Ho, (W+2p)*Kh)."""
    X = _f64(X)
    N, Ci, H, W = X.shape
    Ho, Wo = out_dims(H, W, Kh, Kw, stride, pad)
    Xw = np.empty((N, Ci, Ho, (W + 2 * pad) * Kh))
    assert lib().oracle_im2win_transform(_p(X), _p(Xw), N, Ci, H, W, Kh, Kw, stride, pad) == 0
    return Xw


def im2win_conv(Xw, Wt, H, W, stride=1, pad=0):
    """Eq. (3) on strips made by :func:`im2win_transform`."""
    Xw, Wt = _f64(Xw), _f64(Wt)
    N, Ci = Xw.shape[:2]
    Co, _, Kh, Kw = Wt.shape
    Ho, Wo = out_dims(H, W, Kh, Kw, stride, pad)
    Y = np.empty((N, Co, Ho, Wo))
    assert lib().oracle_im2win_conv(_p(Xw), _p(Wt), _p(Y),
                                    N, Ci, H, W, Co, Kh, Kw, stride, pad) == 0
    return Y


def add_bias(Y, S, b):
    """In place: Y[n, co] += b[co] and S[n, co] += |b[co]| ("Unifying
    Convolutions and GEMM", Sec. 6 listing, `Y_col += bias`).  Y and S are
    C-contiguous float64 NCHW arrays (S may be None)."""
    b = _f64(b).ravel()
    N, Co, Ho, Wo = Y.shape
    assert b.shape[0] == Co and Y.flags.c_contiguous and Y.dtype == np.float64
    if S is not None:
        assert S.shape == Y.shape and S.flags.c_contiguous and S.dtype == np.float64
    assert lib().oracle_add_bias(_p(Y), _p(S) if S is not None else None, _p(b), N, Co, Ho, Wo) == 0
    return Y, S


def parity_error(y_test, y_ref, s_ref):
    """max |y_test - y_ref| / S over outputs with S > 0, and the count of
    outputs with S == 0 where y_test is not exactly zero."""
    y_test = np.asarray(y_test, dtype=np.float64).ravel()
    y_ref = np.asarray(y_ref, dtype=np.float64).ravel()
    s_ref = np.asarray(s_ref, dtype=np.float64).ravel()
    pos = s_ref > 0
    err = 0.0
    if pos.any():
        err = float(np.max(np.abs(y_test[pos] - y_ref[pos]) / s_ref[pos]))
    bad_zero = int(np.count_nonzero(y_test[~pos] != 0.0))
    if not np.all(np.isfinite(y_test)):
        err = float("inf")
    return err, bad_zero
