"""GPU parity: every algorithm of the library against the fp64 oracle, through
the C ABI, on the seeded inputs of the benchmark workloads.

- reduced batches, whole output compared element by element;
- full-size workloads in the benchmark's launch configuration, compared on a
  sample of outputs (every border row/column of two images plus random ones);
- small-integer inputs, where the result is exact in every dtype, compared
  bit for bit after the single rounding to the output type;
- a shape fuzz (odd sizes, Kh != Kw, stride 1-3, any pad < K, few channels,
  channel counts off the tile grid) and degenerate cases.
Tolerance: max |y - Y| / sum|x*w| <= 1e-4 (fp32) or 1e-2 (fp16/bf16 in,
fp32 accumulate); where sum|x*w| == 0 the output must be exactly 0.
"""
import functools
import random

import numpy as np
import pytest

import synth
from tests.helpers import TOL, oracle_full, parity, run_gpu

pytestmark = pytest.mark.gpu

ALGOS = {"f32": ["im2win_fp32_cc", "implicit_fp32_cc"],
         "f16": ["im2win_tc", "implicit_tc", "padded_tc", "implicit_nchw_tc"],
         "bf16": ["im2win_tc", "implicit_tc", "padded_tc", "implicit_nchw_tc"]}
REDUCED_N = {"tiny": 1, "resnet_stage1": 2, "stem": 1, "vgg": 1, "sweep_k1": 1, "sweep_k3": 1,
             "sweep_k5": 1, "sweep_k7": 1, "sweep_k9": 1, "sweep_k11": 1, "sweep_k3_s2": 2}
REDUCED_N.update({f"cv{i}": 1 for i in range(1, 13)})


def _supported(wl, algo):
    """The documented shape limits: the padded and in-kernel NCHW paths are stride 1 only; the direct
    fp32 path needs 16-byte input rows (W % 4 == 0) and its staged rows in one
    copy box (63*s + Kw + 6 <= 256)."""
    if algo in ("padded_tc", "implicit_nchw_tc") and wl.stride != 1:
        return False
    if algo == "implicit_fp32_cc" and (wl.W % 4 != 0 or 63 * wl.stride + wl.Kw + 6 > 256):
        return False
    return True


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_convolution_gb300 import build
    build.build()


@functools.lru_cache(maxsize=None)
def _reduced(name, dtype):
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl, dtype, N=REDUCED_N[name])
    Y, S = oracle_full(d["X64"], d["W64"], wl.stride, wl.pad)
    return d, Y, S


def _cases():
    out = []
    for name, wl in synth.WORKLOADS.items():
        for dt in wl.dtypes:
            for algo in ALGOS[dt]:
                if _supported(wl, algo):
                    out.append((name, dt, algo))
    return out


@pytest.mark.parametrize("name,dtype,algo", _cases())
def test_workload_reduced_batch(name, dtype, algo):
    wl = synth.WORKLOADS[name]
    d, Y, S = _reduced(name, dtype)
    y, used, _ = run_gpu(d["X"], d["W"], wl.stride, wl.pad, dtype, algo)
    assert used == algo
    err, bad0 = parity(y, Y, S)
    assert bad0 == 0 and err <= TOL[dtype], (name, dtype, algo, err)


def _sample_idx(N, Co, Ho, Wo, rng, k=3000):
    """Random outputs plus every border output of images 0 and N-1 for a few channels."""
    idx = set(rng.integers(0, N * Co * Ho * Wo, size=k).tolist())
    for n in {0, N - 1}:
        for co in {0, Co // 2, Co - 1}:
            base = (n * Co + co) * Ho * Wo
            for ho in range(Ho):
                idx.update((base + ho * Wo, base + ho * Wo + Wo - 1))
            for wo in range(Wo):
                idx.update((base + wo, base + (Ho - 1) * Wo + wo))
    return np.array(sorted(idx), dtype=np.int64)


def _full_cases():
    out = []
    for name, wl in synth.WORKLOADS.items():
        if name == "cv4":
            continue            # 822 M input elements at N = 256: covered at reduced batch and by the bench
        for dt in wl.dtypes:
            out.append((name, dt, "auto"))
    out += [("vgg", "f16", "im2win_tc"), ("resnet_stage1", "f16", "im2win_tc"), ("stem", "f16", "implicit_tc"),
            ("stem", "f32", "implicit_fp32_cc"), ("resnet_stage1", "f16", "implicit_tc"), ("vgg", "bf16", "padded_tc"),
            ("sweep_k7", "f16", "padded_tc")]
    return out


@pytest.mark.parametrize("name,dtype,algo", _full_cases())
def test_workload_full_size_sampled(name, dtype, algo):
    from oracle import ref
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl, dtype)
    y, used, ws = run_gpu(d["X"], d["W"], wl.stride, wl.pad, dtype, algo)
    N, Co, Ho, Wo = y.shape
    idx = _sample_idx(N, Co, Ho, Wo, np.random.default_rng(wl.seed))
    Ys, Ss = ref.conv2d_points(d["X64"], d["W64"], idx, wl.stride, wl.pad)
    err, bad0 = parity(y.ravel()[idx], Ys, Ss)
    assert bad0 == 0 and err <= TOL[dtype], (name, dtype, used, err)
    assert np.all(np.isfinite(y)), "unwritten outputs"
    # Workspace stays within the im2win tensor of the pages (N*Ci*Ho*(W+2p)*Kh
    # elements) plus the repacked filter.
    elem = 4 if dtype == "f32" else 2
    ci8 = (wl.Ci + 7) // 8 * 8 if dtype != "f32" else wl.Ci
    cap = wl.N * ci8 * Ho * (wl.W + 2 * wl.pad) * wl.Kh * elem + 4 * wl.Co * wl.Ci * wl.Kh * wl.Kw * 4 + 2 ** 20
    assert ws <= cap


def _exact_expected(Y, dtype):
    """Integer oracle result rounded once to the output dtype."""
    import torch
    t = torch.from_numpy(Y.astype(np.float32))
    if dtype == "f16":
        t = t.half()
    elif dtype == "bf16":
        t = t.bfloat16()
    return t.double().numpy()


INT_SHAPES = [
    # N, Ci, H, W, Co, Kh, Kw, s, p
    (2, 64, 14, 14, 64, 3, 3, 1, 1),
    (1, 3, 30, 30, 64, 7, 7, 2, 3),
    (1, 16, 9, 11, 24, 3, 5, 1, 2),
    (2, 5, 17, 13, 7, 2, 3, 3, 1),
    (1, 128, 8, 8, 128, 1, 1, 1, 0),
    (1, 72, 10, 12, 136, 3, 3, 2, 0),
    (3, 8, 5, 5, 264, 5, 5, 1, 4),
    (1, 1, 1, 1, 1, 1, 1, 1, 0),
]


@pytest.mark.parametrize("shape", INT_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_small_integers_bit_exact(shape, dtype):
    from dense_convolution_gb300 import capi
    N, Ci, H, W, Co, Kh, Kw, s, p = shape
    lo, hi = (-3, 3) if dtype != "bf16" else (-1, 1)
    d = synth.make_int_inputs(sum(shape) * 7 + len(dtype), N, Ci, H, W, Co, Kh, Kw, dtype, lo, hi)
    Y, S = oracle_full(d["X64"], d["W64"], s, p)
    assert np.max(np.abs(Y)) < (2048 if dtype == "f16" else 2 ** 24)
    expect = _exact_expected(Y, dtype)
    ran = 0
    for algo in ALGOS[dtype]:
        try:
            y, _, _ = run_gpu(d["X"], d["W"], s, p, dtype, algo)
        except capi.Conv2dError as e:
            assert e.status == capi.ERR_UNSUPPORTED
            continue
        ran += 1
        mism = np.argwhere(y != expect)
        assert mism.size == 0, (algo, mism[:5].tolist(), y[tuple(mism[0])], expect[tuple(mism[0])])
    assert ran >= 1


def _fuzz_shapes(count, seed):
    rng = random.Random(seed)
    out = []
    while len(out) < count:
        Kh, Kw = rng.randint(1, 7), rng.randint(1, 7)
        s = rng.randint(1, 3)
        p = rng.randint(0, max(Kh, Kw) - 1)
        H = rng.randint(max(1, Kh - 2 * p), 40)
        W = rng.choice([rng.randint(max(1, Kw - 2 * p), 40), 4 * rng.randint(max(1, (Kw - 2 * p + 3) // 4), 10)])
        Ci = rng.choice([1, 3, 5, 8, 13, 16, 24, 40, 64, 96])
        Co = rng.choice([1, 5, 16, 17, 48, 64, 80, 130, 200, 256, 300])
        N = rng.randint(1, 3)
        out.append((N, Ci, H, W, Co, Kh, Kw, s, p))
    return out


@pytest.mark.parametrize("shape", _fuzz_shapes(24, 2024), ids=lambda s: "x".join(map(str, s)))
def test_shape_fuzz(shape):
    from dense_convolution_gb300 import capi
    N, Ci, H, W, Co, Kh, Kw, s, p = shape
    for dtype in ("f32", "f16", "bf16"):
        seed = abs(hash(shape)) % 100000 + len(dtype)
        x = synth.normal(seed, 0, (N, Ci, H, W))
        w = synth.normal(seed, 1, (Co, Ci, Kh, Kw))
        X, X64 = synth.round_to(x, dtype)
        Wt, W64 = synth.round_to(w, dtype)
        Y, S = oracle_full(X64, W64, s, p)
        for algo in ALGOS[dtype]:
            try:
                y, _, _ = run_gpu(X, Wt, s, p, dtype, algo)
            except capi.Conv2dError as e:
                assert e.status == capi.ERR_UNSUPPORTED, (algo, e)
                continue
            err, bad0 = parity(y, Y, S)
            assert bad0 == 0 and err <= TOL[dtype], (shape, dtype, algo, err)


def test_dense_layer_as_global_kernel():
    # Kh = H, Kw = W, p = 0: one output pixel per channel (a dense layer).
    d = synth.make_inputs(synth.WORKLOADS["tiny"].scaled(), "f32")
    for dtype in ("f32", "f16"):
        x = synth.normal(5, 0, (4, 16, 8, 8))
        w = synth.normal(5, 1, (32, 16, 8, 8), 0.05)
        X, X64 = synth.round_to(x, dtype)
        Wt, W64 = synth.round_to(w, dtype)
        Y, S = oracle_full(X64, W64, 1, 0)
        for algo in ALGOS[dtype]:
            y, _, _ = run_gpu(X, Wt, 1, 0, dtype, algo)
            assert y.shape == (4, 32, 1, 1)
            err, bad0 = parity(y, Y, S)
            assert bad0 == 0 and err <= TOL[dtype]
    assert d["X"].shape[0] == 1


def test_nhwc_input_layout():
    wl = synth.WORKLOADS["resnet_stage1"]
    d, Y, S = _reduced("resnet_stage1", "f16")
    y, used, ws = run_gpu(d["X"], d["W"], wl.stride, wl.pad, "f16", "implicit_tc", layout="nhwc")
    assert used == "implicit_tc" and ws == wl.Co * 9 * wl.Ci * 2
    err, bad0 = parity(y, Y, S)
    assert bad0 == 0 and err <= TOL["f16"]


def test_repeated_calls_and_streams():
    import torch
    from dense_convolution_gb300.conv import Conv2d
    wl = synth.WORKLOADS["resnet_stage1"]
    d, Y, S = _reduced("resnet_stage1", "f16")
    op = Conv2d(2, wl.Ci, wl.H, wl.W, wl.Co, 3, 3, 1, 1, "f16", "auto")
    x = torch.from_numpy(d["X"]).cuda()
    w = torch.from_numpy(d["W"]).cuda()
    st = torch.cuda.Stream()
    ws = op.alloc_workspace()
    outs = []
    with torch.cuda.stream(st):
        for _ in range(3):
            outs.append(op(x, w, workspace=ws))
    st.synchronize()
    for o in outs:
        err, _ = parity(o.double().cpu().numpy(), Y, S)
        assert err <= TOL["f16"]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# Padded-source edge cases with one channel tile (resident filter): channel
# counts below the tile width, Kw = 2 with 128-wide tiles, odd widths (scalar
# stores), Kh = 1, padding wider than the filter's reach, several images.
PADDED_EDGE_SHAPES = [
    # N, Ci, H, W, Co, Kh, Kw, s, p
    (3, 64, 23, 21, 64, 3, 3, 1, 1),
    (2, 32, 16, 16, 128, 2, 2, 1, 1),
    (1, 24, 40, 36, 40, 3, 3, 1, 0),
    (1, 8, 9, 9, 64, 1, 3, 1, 1),
    (4, 72, 12, 12, 17, 3, 3, 1, 2),
]


@pytest.mark.parametrize("shape", PADDED_EDGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_padded_single_channel_tile(shape, dtype):
    N, Ci, H, W, Co, Kh, Kw, s, p = shape
    seed = sum(shape) * 13 + len(dtype)
    X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), dtype)
    Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, Kh, Kw)), dtype)
    Y, S = oracle_full(X64, W64, s, p)
    y, used, _ = run_gpu(X, Wt, s, p, dtype, "padded_tc")
    err, bad0 = parity(y, Y, S)
    assert bad0 == 0 and err <= TOL[dtype], (shape, dtype, err)


# 1x1 layers run as one GEMM per image on the NCHW tensors (no workspace):
# channel counts off the 64-wide K chunk, pixel counts off the 128-pixel tile
# (a tail shorter than one 64-pixel box, tails that end mid-vector), output
# channels off the 128-channel tile and several channel tiles.
GEMM1X1_SHAPES = [
    # N, Ci, H, W, Co
    (2, 128, 16, 16, 128),
    (3, 72, 10, 12, 17),
    (1, 8, 2, 4, 130),
    (2, 200, 7, 8, 300),
    (4, 64, 56, 56, 64),
    (1, 16, 5, 40, 256),
]


@pytest.mark.parametrize("shape", GEMM1X1_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gemm_1x1(shape, dtype):
    from dense_convolution_gb300 import capi
    N, Ci, H, W, Co = shape
    seed = sum(shape) * 17 + len(dtype)
    X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), dtype)
    Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, 1, 1)), dtype)
    Y, S = oracle_full(X64, W64, 1, 0)
    y, used, ws = run_gpu(X, Wt, 1, 0, dtype, "implicit_tc")
    assert used == "implicit_tc" and ws == 0
    err, bad0 = parity(y, Y, S)
    assert bad0 == 0 and err <= TOL[dtype], (shape, dtype, err)
    d = capi.conv2d_desc_create(N, Ci, H, W, Co, 1, 1, 1, 0, dtype, "implicit_tc")
    try:
        assert capi.conv2d_launches_per_call(d) == 1
    finally:
        capi.conv2d_desc_destroy(d)


@pytest.mark.parametrize("name,dtype,algo", [("resnet_stage1", "f16", "auto"), ("sweep_k1", "f16", "auto"),
                                              ("tiny", "f32", "auto"), ("stem", "bf16", "im2win_tc")])
@pytest.mark.parametrize("pinned", [True, False])
def test_fwd_host_matches_device_call(name, dtype, algo, pinned):
    """conv2d_fwd_host (copy in, call, copy out on one stream) gives the same
    bits as conv2d_fwd on device operands, from page-locked or pageable host
    memory."""
    import torch
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    wl = synth.WORKLOADS[name]
    n = REDUCED_N[name]
    d = synth.make_inputs(wl, dtype, N=n)
    op = Conv2d(n, wl.Ci, wl.H, wl.W, wl.Co, wl.Kh, wl.Kw, wl.stride, wl.pad, dtype, algo)
    xh = (torch.from_numpy(d["X"]) if dtype != "bf16" else d["X"]).contiguous()
    wh = (torch.from_numpy(d["W"]) if dtype != "bf16" else d["W"]).contiguous()
    if pinned:
        xh, wh = xh.pin_memory(), wh.pin_memory()
    ref = op(xh.cuda(), wh.cuda()).cpu()
    xd, wd = torch.empty_like(xh, device="cuda"), torch.empty_like(wh, device="cuda")
    yd = op.alloc_output()
    yh = torch.full(tuple(yd.shape), float("nan"), dtype=yd.dtype)
    if pinned:
        yh = yh.pin_memory()
    ws = op.alloc_workspace()
    st = torch.cuda.current_stream()
    capi.conv2d_fwd_host(op.desc, xh.data_ptr(), wh.data_ptr(), yh.data_ptr(), xd.data_ptr(), wd.data_ptr(),
                         yd.data_ptr(), ws.data_ptr(), op.workspace_bytes, st.cuda_stream)
    st.synchronize()
    assert capi.conv2d_device_status(0) == 0
    assert torch.equal(yh.view(torch.int16) if yh.element_size() == 2 else yh.view(torch.int32),
                       ref.view(torch.int16) if ref.element_size() == 2 else ref.view(torch.int32))
