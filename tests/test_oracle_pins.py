"""Pins for the fp64 oracle: each check ties it to something other than itself.

- values printed on the pages (worked examples, Table I shapes) and cases
  worked by hand from the definitions (tests/golden/);
- brute force in plain Python on tiny inputs;
- library routines for special cases and for the whole operator
  (scipy.signal.correlate2d per channel pair; float64 torch conv2d/unfold);
- closed forms (delta kernel, all-ones counts, 1x1 kernel, dense layer);
- invariants (linearity, batch independence, translation);
- exact small-integer arithmetic.
A mutation test at the end plants plausible mistakes in a copy of the oracle
and checks that these pins catch every one.
"""
import os
import random

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng_case(rng: random.Random):
    N = rng.randint(1, 2)
    Ci = rng.randint(1, 4)
    Co = rng.randint(1, 4)
    Kh = rng.randint(1, 5)
    Kw = rng.randint(1, 5)
    s = rng.randint(1, 3)
    p = rng.randint(0, max(Kh, Kw) - 1)
    H = rng.randint(max(1, Kh - 2 * p), 9)
    W = rng.randint(max(1, Kw - 2 * p), 9)
    return N, Ci, H, W, Co, Kh, Kw, s, p


def _brute(X, Wt, s, p):
    """Plain Python 7-loop with explicit bounds checks."""
    N, Ci, H, W = X.shape
    Co, _, Kh, Kw = Wt.shape
    Ho = (H + 2 * p - Kh) // s + 1
    Wo = (W + 2 * p - Kw) // s + 1
    Y = [[[[0.0] * Wo for _ in range(Ho)] for _ in range(Co)] for _ in range(N)]
    for n in range(N):
        for co in range(Co):
            for ho in range(Ho):
                for wo in range(Wo):
                    acc = 0.0
                    for ci in range(Ci):
                        for kh in range(Kh):
                            for kw in range(Kw):
                                y, x = ho * s + kh - p, wo * s + kw - p
                                if 0 <= y < H and 0 <= x < W:
                                    acc += float(X[n, ci, y, x]) * float(Wt[co, ci, kh, kw])
                    Y[n][co][ho][wo] = acc
    return np.array(Y)


def _scipy_conv(X, Wt, s, p):
    """Sum over input channels of scipy's 2-D cross-correlation of the
    zero-padded plane with the filter, 'valid' mode, then subsample by s."""
    from scipy.signal import correlate2d
    N, Ci, H, W = X.shape
    Co, _, Kh, Kw = Wt.shape
    Xp = np.pad(X, ((0, 0), (0, 0), (p, p), (p, p)))
    Ho = (H + 2 * p - Kh) // s + 1
    Wo = (W + 2 * p - Kw) // s + 1
    Y = np.zeros((N, Co, Ho, Wo))
    for n in range(N):
        for co in range(Co):
            acc = 0
            for ci in range(Ci):
                acc = acc + correlate2d(Xp[n, ci], Wt[co, ci], mode="valid")
            Y[n, co] = acc[::s, ::s][:Ho, :Wo]
    return Y


def _torch_conv(X, Wt, s, p):
    import torch
    import torch.nn.functional as F
    return F.conv2d(torch.from_numpy(X), torch.from_numpy(Wt), stride=s, padding=p).numpy()


# --------------------------------------------------------------- worked examples

def test_winograd_page_worked_example(oracle):
    with open(os.path.join(GOLDEN, "winograd_f23_worked_example.txt")) as f:
        rows = [list(map(float, l.split())) for l in f if l.strip() and not l.startswith("#")]
    d, g, expect = rows
    Y, S = oracle.conv2d(np.array(d).reshape(1, 1, 1, 4), np.array(g).reshape(1, 1, 1, 3))
    assert Y.ravel().tolist() == expect
    assert S.ravel().tolist() == [2 * 1 + 0 + 3, 2 * 2 + 0 + 4]


def test_table1_output_dims(oracle):
    with open(os.path.join(GOLDEN, "im2win_table1_shapes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 12
    for r in rows:
        _, ci, hi, wi, co, hf, wf, s, co2, ho, wo = r[0], *map(int, r[1:])
        assert co == co2
        assert oracle.out_dims(hi, wi, hf, wf, s, 0) == (ho, wo), r[0]


def test_fig1_shapes(oracle):
    # Fig. 1 of the im2win paper: input 1x3x3x3, filter 2x3x2x2, output 1x2x2x2.
    X = np.arange(27, dtype=np.float64).reshape(1, 3, 3, 3)
    Wt = np.ones((2, 3, 2, 2))
    Y, _ = oracle.conv2d(X, Wt)
    assert Y.shape == (1, 2, 2, 2)


def test_im2col_shape_from_page(oracle):
    # im2col page: a (3, 32, 32) input with a 3x3 kernel, stride 1, pad 1
    # expands to a (27, 1024) matrix.
    x = np.random.default_rng(0).normal(size=(3, 32, 32))
    assert oracle.im2col(x, 3, 3, 1, 1).shape == (27, 1024)


def _hand_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "im2win_hand_examples.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "case":
                cur = {"name": tok[1], "dims": list(map(int, tok[2:]))}
                cases.append(cur)
            else:
                cur[tok[0]] = np.array(list(map(float, tok[1:])))
    return cases


@pytest.mark.parametrize("case", _hand_cases(), ids=lambda c: c["name"])
def test_hand_worked_im2win(oracle, case):
    N, Ci, H, W, Co, Kh, Kw, s, p = case["dims"]
    X = case["x"].reshape(N, Ci, H, W)
    Wt = case["w"].reshape(Co, Ci, Kh, Kw)
    Xw = oracle.im2win_transform(X, Kh, Kw, s, p)
    assert Xw.ravel().tolist() == case["strip"].tolist()
    Y, _ = oracle.conv2d(X, Wt, s, p)
    assert Y.ravel().tolist() == case["y"].tolist()
    Y2 = oracle.im2win_conv(Xw, Wt, H, W, s, p)
    assert Y2.ravel().tolist() == case["y"].tolist()
    assert oracle.conv2d_im2col(X, Wt, s, p).ravel().tolist() == case["y"].tolist()


# --------------------------------------------------------------- brute force

def test_bruteforce_random_tiny(oracle):
    rng = random.Random(12345)
    nrng = np.random.default_rng(7)
    for _ in range(220):
        N, Ci, H, W, Co, Kh, Kw, s, p = _rng_case(rng)
        X = nrng.normal(size=(N, Ci, H, W))
        Wt = nrng.normal(size=(Co, Ci, Kh, Kw))
        Y, S = oracle.conv2d(X, Wt, s, p)
        B = _brute(X, Wt, s, p)
        assert Y.shape == B.shape
        assert np.max(np.abs(Y - B)) <= 1e-12 * max(1.0, np.max(S))


# --------------------------------------------------------------- library routines

@pytest.mark.parametrize("shape", [
    (2, 3, 11, 13, 4, 3, 3, 1, 1),
    (1, 2, 17, 9, 3, 5, 2, 2, 1),
    (2, 1, 16, 16, 2, 7, 7, 2, 3),
    (1, 4, 10, 12, 5, 1, 1, 1, 0),
    (1, 3, 15, 15, 2, 4, 3, 3, 2),
    (1, 2, 9, 9, 3, 9, 9, 1, 4),
])
def test_vs_scipy_and_torch(oracle, shape):
    N, Ci, H, W, Co, Kh, Kw, s, p = shape
    r = np.random.default_rng(sum(shape))
    X = r.normal(size=(N, Ci, H, W))
    Wt = r.normal(size=(Co, Ci, Kh, Kw))
    Y, S = oracle.conv2d(X, Wt, s, p)
    tol = 1e-12 * max(1.0, float(np.max(S)))
    assert np.max(np.abs(Y - _scipy_conv(X, Wt, s, p))) <= tol
    assert np.max(np.abs(Y - _torch_conv(X, Wt, s, p))) <= tol


def test_im2col_matches_torch_unfold(oracle):
    import torch
    import torch.nn.functional as F
    r = np.random.default_rng(3)
    for (Ci, H, W, Kh, Kw, s, p) in [(3, 10, 12, 3, 3, 1, 1), (2, 9, 7, 2, 4, 2, 1), (1, 8, 8, 5, 5, 3, 2)]:
        x = r.normal(size=(Ci, H, W))
        cols = oracle.im2col(x, Kh, Kw, s, p)
        ref = F.unfold(torch.from_numpy(x)[None], (Kh, Kw), padding=p, stride=s)[0].numpy()
        assert np.array_equal(cols, ref)


def test_gemm_naive_matches_numpy(oracle):
    r = np.random.default_rng(4)
    A, B = r.normal(size=(7, 13)), r.normal(size=(13, 5))
    assert np.max(np.abs(oracle.gemm(A, B) - A @ B)) < 1e-12


def test_im2col_gemm_path_equals_direct(oracle):
    rng = random.Random(99)
    nrng = np.random.default_rng(99)
    for _ in range(40):
        N, Ci, H, W, Co, Kh, Kw, s, p = _rng_case(rng)
        X = nrng.normal(size=(N, Ci, H, W))
        Wt = nrng.normal(size=(Co, Ci, Kh, Kw))
        Y, S = oracle.conv2d(X, Wt, s, p)
        Y2 = oracle.conv2d_im2col(X, Wt, s, p)
        assert np.max(np.abs(Y - Y2)) <= 1e-12 * max(1.0, np.max(S))


def test_im2win_path_equals_direct_nonsquare(oracle):
    rng = random.Random(5)
    nrng = np.random.default_rng(5)
    seen_nonsquare = 0
    for _ in range(60):
        N, Ci, H, W, Co, Kh, Kw, s, p = _rng_case(rng)
        seen_nonsquare += Kh != Kw
        X = nrng.normal(size=(N, Ci, H, W))
        Wt = nrng.normal(size=(Co, Ci, Kh, Kw))
        Y, S = oracle.conv2d(X, Wt, s, p)
        Xw = oracle.im2win_transform(X, Kh, Kw, s, p)
        assert Xw.shape == (N, Ci, Y.shape[2], (W + 2 * p) * Kh)
        Y2 = oracle.im2win_conv(Xw, Wt, H, W, s, p)
        assert np.max(np.abs(Y - Y2)) <= 1e-12 * max(1.0, np.max(S))
    assert seen_nonsquare >= 20


def test_im2win_memory_vs_im2col(oracle):
    # The strip holds Kh elements per padded input column per output row, so
    # it is smaller than the im2col matrix whenever windows overlap
    # horizontally (s < Kw) and no larger when they do not.
    for (H, W, K, s, p) in [(56, 56, 3, 1, 1), (224, 224, 7, 2, 3), (28, 28, 3, 3, 0)]:
        Ho, Wo = oracle.out_dims(H, W, K, K, s, p)
        win = Ho * (W + 2 * p) * K
        col = Ho * Wo * K * K
        if s < K:
            assert win < col
        else:
            assert win >= col


# --------------------------------------------------------------- closed forms

@pytest.mark.parametrize("K,C,H,W", [(1, 3, 5, 7), (3, 4, 8, 6), (5, 2, 9, 9), (7, 1, 11, 10)])
def test_delta_kernel_reproduces_input(oracle, K, C, H, W):
    p = (K - 1) // 2
    X = np.random.default_rng(K).normal(size=(2, C, H, W))
    Wt = np.zeros((C, C, K, K))
    for c in range(C):
        Wt[c, c, p, p] = 1.0
    Y, S = oracle.conv2d(X, Wt, 1, p)
    assert np.array_equal(Y, X)
    assert np.array_equal(S, np.abs(X))


@pytest.mark.parametrize("H,W,Kh,Kw,s,p,C", [(6, 7, 3, 3, 1, 1, 5), (9, 9, 5, 3, 2, 2, 3),
                                             (8, 5, 4, 2, 3, 3, 2), (12, 12, 7, 7, 2, 3, 3)])
def test_all_ones_counts(oracle, H, W, Kh, Kw, s, p, C):
    Y, S = oracle.conv2d(np.ones((1, C, H, W)), np.ones((2, C, Kh, Kw)), s, p)
    Ho, Wo = Y.shape[2:]
    for ho in range(Ho):
        r = len([kh for kh in range(Kh) if 0 <= ho * s + kh - p < H])
        for wo in range(Wo):
            c = len([kw for kw in range(Kw) if 0 <= wo * s + kw - p < W])
            assert Y[0, 0, ho, wo] == C * r * c == Y[0, 1, ho, wo]
    if p == 0 or Kh == 1:
        pass
    # Interior points see the full window.
    interior = [(ho, wo) for ho in range(Ho) for wo in range(Wo)
                if ho * s - p >= 0 and ho * s - p + Kh <= H and wo * s - p >= 0 and wo * s - p + Kw <= W]
    for ho, wo in interior:
        assert Y[0, 0, ho, wo] == C * Kh * Kw
    assert np.array_equal(Y, S)


def test_1x1_kernel_is_per_pixel_matmul(oracle):
    r = np.random.default_rng(11)
    X = r.normal(size=(2, 6, 5, 7))
    Wt = r.normal(size=(4, 6, 1, 1))
    Y, _ = oracle.conv2d(X, Wt)
    M = Wt[:, :, 0, 0]
    for n in range(2):
        for h in range(5):
            for w in range(7):
                assert np.allclose(Y[n, :, h, w], M @ X[n, :, h, w], rtol=0, atol=1e-12)


def test_dense_layer_is_global_kernel_conv(oracle):
    r = np.random.default_rng(12)
    X = r.normal(size=(3, 4, 5, 6))
    Wt = r.normal(size=(7, 4, 5, 6))
    Y, _ = oracle.conv2d(X, Wt)
    assert Y.shape == (3, 7, 1, 1)
    dense = X.reshape(3, -1) @ Wt.reshape(7, -1).T
    assert np.max(np.abs(Y[:, :, 0, 0] - dense)) < 1e-12


# --------------------------------------------------------------- invariants

def test_linearity_and_batch_independence(oracle):
    r = np.random.default_rng(13)
    X1, X2 = r.normal(size=(2, 3, 3, 9, 8))
    W1, W2 = r.normal(size=(2, 4, 3, 3, 2))
    a, b = 1.5, -0.25
    Y = lambda x, w: oracle.conv2d(x, w, 2, 1)[0]
    assert np.allclose(Y(a * X1 + b * X2, W1), a * Y(X1, W1) + b * Y(X2, W1), atol=1e-12)
    assert np.allclose(Y(X1, a * W1 + b * W2), a * Y(X1, W1) + b * Y(X1, W2), atol=1e-12)
    full = Y(X1, W1)
    for n in range(X1.shape[0]):
        assert np.array_equal(Y(X1[n:n + 1], W1)[0], full[n])


def test_translation(oracle):
    r = np.random.default_rng(14)
    s = 2
    X = r.normal(size=(1, 2, 12, 14))
    Wt = r.normal(size=(3, 2, 3, 3))
    Y, _ = oracle.conv2d(X, Wt, s, 0)
    Xs = np.zeros_like(X)
    Xs[..., s:, s:] = X[..., :-s, :-s]
    Ys, _ = oracle.conv2d(Xs, Wt, s, 0)
    assert np.allclose(Ys[..., 1:, 1:], Y[..., :-1, :-1], atol=1e-12)


def test_small_integers_exact(oracle):
    import synth
    d = synth.make_int_inputs(77, 2, 5, 9, 11, 3, 3, 4, "f32")
    Y, S = oracle.conv2d(d["X64"], d["W64"], 2, 1)
    B = _brute(d["X64"], d["W64"], 2, 1)
    assert np.array_equal(Y, B)
    assert np.all(Y == np.round(Y))


def test_abs_sum_matches_signless_run(oracle):
    r = np.random.default_rng(15)
    X = r.normal(size=(1, 3, 7, 7))
    Wt = r.normal(size=(2, 3, 3, 3))
    _, S = oracle.conv2d(X, Wt, 1, 1)
    Yabs, _ = oracle.conv2d(np.abs(X), np.abs(Wt), 1, 1)
    assert np.allclose(S, Yabs, atol=1e-12)


def test_points_match_direct(oracle):
    r = np.random.default_rng(16)
    X = r.normal(size=(2, 3, 10, 9))
    Wt = r.normal(size=(5, 3, 4, 3))
    Y, S = oracle.conv2d(X, Wt, 2, 1)
    idx = r.choice(Y.size, size=40, replace=False)
    idx = np.concatenate([idx, [0, Y.size - 1]])
    y, s = oracle.conv2d_points(X, Wt, idx, 2, 1)
    assert np.array_equal(y, Y.ravel()[idx]) and np.array_equal(s, S.ravel()[idx])
    with pytest.raises(ValueError):
        oracle.conv2d_points(X, Wt, [Y.size], 2, 1)


def test_parity_error_metric(oracle):
    err, bad = oracle.parity_error([1.0, 2.0, 0.0], [1.0, 2.5, 0.0], [1.0, 5.0, 0.0])
    assert err == pytest.approx(0.1) and bad == 0
    err, bad = oracle.parity_error([0.0, 1e-30], [0.0, 0.0], [1.0, 0.0])
    assert bad == 1


# --------------------------------------------------------------- mutation check

_MUTATIONS = [
    ("int64_t y = ho * s + kh - p;", "int64_t y = ho * s + kh + p;"),          # wrong pad sign
    ("int64_t x = wo * s + kw - p;", "int64_t x = wo * s + (Kw - 1 - kw) - p;"),  # flipped kernel
    ("* wc[kh * Kw + kw];", "* wc[kw * Kh + kh];"),                                   # transposed filter
    ("if (x < 0 || x >= W) continue;", "if (x < 0 || x > W) continue;"),       # off-by-one bound
    ("sabs += fabs(t);", "sabs += t;"),                                         # signed abs-sum
    ("return span / s + 1;", "return (span + s - 1) / s + 1;"),                 # ceil output size
    ("for (int64_t ci = 0; ci < Ci; ++ci) {\n        const double *xc",
     "for (int64_t ci = 0; ci + 1 < Ci; ++ci) {\n        const double *xc"),    # dropped channel
    ("double t = xc[y * W + x] * wc[kh * Kw + kw];",
     "double t = xc[x * H + y] * wc[kh * Kw + kw];"),                           # transposed image
]


def _pins_pass(lib_path):
    """Run a subset of the pins against the direct routine of another build."""
    import ctypes
    L = ctypes.CDLL(lib_path)
    dp = ctypes.POINTER(ctypes.c_double)
    L.oracle_conv2d_direct.argtypes = [dp, dp, dp, dp] + [ctypes.c_int] * 9
    L.oracle_conv2d_direct.restype = ctypes.c_int
    L.oracle_out_dims.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_int)] * 2

    def conv(X, Wt, s, p):
        N, Ci, H, W = X.shape
        Co, _, Kh, Kw = Wt.shape
        ho, wo = ctypes.c_int(), ctypes.c_int()
        L.oracle_out_dims(H, W, Kh, Kw, s, p, ctypes.byref(ho), ctypes.byref(wo))
        Y = np.zeros((N, Co, max(ho.value, 1), max(wo.value, 1)))
        S = np.zeros_like(Y)
        X = np.ascontiguousarray(X); Wt = np.ascontiguousarray(Wt)
        L.oracle_conv2d_direct(X.ctypes.data_as(dp), Wt.ctypes.data_as(dp), Y.ctypes.data_as(dp),
                               S.ctypes.data_as(dp), N, Ci, H, W, Co, Kh, Kw, s, p)
        return Y, S

    r = np.random.default_rng(21)
    # Table I, cv4: 224x224 input, 7x7 filter, stride 2 -> 109x109.
    ho, wo = ctypes.c_int(), ctypes.c_int()
    L.oracle_out_dims(224, 224, 7, 7, 2, 0, ctypes.byref(ho), ctypes.byref(wo))
    if (ho.value, wo.value) != (109, 109):
        return False
    for (N, Ci, H, W, Co, Kh, Kw, s, p) in [(2, 3, 9, 10, 2, 3, 2, 2, 1), (1, 2, 8, 7, 2, 3, 3, 1, 1),
                                            (1, 2, 10, 9, 2, 3, 3, 2, 1)]:
        X = r.normal(size=(N, Ci, H, W))
        Wt = r.normal(size=(Co, Ci, Kh, Kw))
        ref = _scipy_conv(X, Wt, s, p)
        Y, S = conv(X, Wt, s, p)
        if Y.shape != ref.shape or np.max(np.abs(Y - ref)) > 1e-9:
            return False
        Yabs, _ = conv(np.abs(X), np.abs(Wt), s, p)
        if not np.allclose(S, Yabs, atol=1e-12):
            return False
    return True


def test_pins_catch_planted_mistakes(tmp_path, oracle):
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle.__file__), "conv_ref.c")).read()
    clean = tmp_path / "clean.c"
    clean.write_text(src)
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", str(clean), "-o", str(tmp_path / "clean.so"), "-lm"],
                   check=True)
    assert _pins_pass(str(tmp_path / "clean.so"))
    for i, (a, b) in enumerate(_MUTATIONS):
        assert a in src, a
        mut = tmp_path / f"m{i}.c"
        mut.write_text(src.replace(a, b, 1))
        so = tmp_path / f"m{i}.so"
        subprocess.run(["gcc", "-O1", "-fPIC", "-shared", str(mut), "-o", str(so), "-lm"], check=True)
        assert not _pins_pass(str(so)), f"mutation {i} not caught: {b}"


# --------------------------------------------------------------- bias ("Unifying Convolutions and GEMM", Sec. 6)

def _bias_closed_form_ok(add_bias):
    """All-ones X and W plus a bias: Y = Ci * r(ho) * c(wo) + b[co] and
    S = Ci * r(ho) * c(wo) + |b[co]| (r, c = filter rows / columns inside the
    image), with distinct signed biases per channel and two images."""
    import ctypes  # noqa: F401
    N, C, H, W, Co, Kh, Kw, s, p = 2, 3, 6, 7, 4, 3, 3, 1, 1
    from oracle import ref
    Y, S = ref.conv2d(np.ones((N, C, H, W)), np.ones((Co, C, Kh, Kw)), s, p)
    b = np.array([0.5, -2.25, 3.0, -0.125])
    add_bias(Y, S, b)
    Ho, Wo = Y.shape[2:]
    for n in range(N):
        for co in range(Co):
            for ho in range(Ho):
                r = len([kh for kh in range(Kh) if 0 <= ho * s + kh - p < H])
                for wo in range(Wo):
                    c = len([kw for kw in range(Kw) if 0 <= wo * s + kw - p < W])
                    if Y[n, co, ho, wo] != C * r * c + b[co] or S[n, co, ho, wo] != C * r * c + abs(b[co]):
                        return False
    return True


def test_bias_all_ones_closed_form(oracle):
    assert _bias_closed_form_ok(oracle.add_bias)


def test_bias_zero_filter_gives_bias(oracle):
    b = np.array([1.5, -4.0, 0.0])
    Y, S = oracle.conv2d(np.ones((2, 2, 5, 5)), np.zeros((3, 2, 3, 3)), 1, 1)
    oracle.add_bias(Y, S, b)
    assert np.array_equal(Y, np.broadcast_to(b[None, :, None, None], Y.shape))
    assert np.array_equal(S, np.abs(Y))


def test_bias_vs_torch(oracle):
    import torch
    import torch.nn.functional as F
    r = np.random.default_rng(31)
    X = r.normal(size=(3, 5, 9, 8))
    Wt = r.normal(size=(6, 5, 3, 2))
    b = r.normal(size=6)
    Y, S = oracle.conv2d(X, Wt, 2, 1)
    oracle.add_bias(Y, S, b)
    ref = F.conv2d(torch.from_numpy(X), torch.from_numpy(Wt), torch.from_numpy(b), stride=2, padding=1).numpy()
    assert np.max(np.abs(Y - ref)) < 1e-12


_BIAS_MUTATIONS = [
    ("y[i] += b[co];", "y[i] += b[n];"),                       # bias indexed by image
    ("y[i] += b[co];", "y[i] -= b[co];"),                      # wrong sign
    ("if (sa) sa[i] += fabs(b[co]);", "if (sa) sa[i] += b[co];"),   # signed |b| in S
    ("for (int64_t co = 0; co < Co; ++co) {\n            double *y",
     "for (int64_t co = 0; co + 1 < Co; ++co) {\n            double *y"),   # last channel skipped
]


def test_bias_pins_catch_planted_mistakes(tmp_path, oracle):
    import ctypes
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle.__file__), "conv_ref.c")).read()
    dp = ctypes.POINTER(ctypes.c_double)
    for i, (a, b) in enumerate(_BIAS_MUTATIONS):
        assert a in src, a
        mut = tmp_path / f"b{i}.c"
        mut.write_text(src.replace(a, b, 1))
        so = tmp_path / f"b{i}.so"
        subprocess.run(["gcc", "-O1", "-fPIC", "-shared", str(mut), "-o", str(so), "-lm"], check=True)
        L = ctypes.CDLL(str(so))
        L.oracle_add_bias.argtypes = [dp, dp, dp] + [ctypes.c_int] * 4
        L.oracle_add_bias.restype = ctypes.c_int

        def add_bias(Y, S, bias, L=L):
            bias = np.ascontiguousarray(bias, dtype=np.float64)
            N, Co, Ho, Wo = Y.shape
            L.oracle_add_bias(Y.ctypes.data_as(dp), S.ctypes.data_as(dp), bias.ctypes.data_as(dp), N, Co, Ho, Wo)

        assert not _bias_closed_form_ok(add_bias), f"bias mutation {i} not caught: {b}"
