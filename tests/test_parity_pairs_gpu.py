"""GPU parity on the paths the large layers take, compared over the WHOLE output.

The tensor-core kernel takes tiles in pairs (two MMA issuers, two epilogue
groups) only when a call has at least two tiles per SM; smaller calls run
single tiles.  These cases are sized past 2 x 152 tiles so that the pair
path, the streamed (non-resident) filter, one accumulator per issuer
(256- and 176-wide channel tiles) and the 1x1 GEMM with pairs all run, and every
output element is compared with the fp64 oracle (outputs pre-filled with
NaN, workspace guard bytes checked).  Tolerance as in the other parity tests:
max |y - Y| / sum|x*w| <= 1e-2 for 16-bit inputs with fp32 accumulation.
"""
import numpy as np
import pytest

import synth
from tests.helpers import TOL, oracle_full, parity, run_gpu

pytestmark = pytest.mark.gpu

SMS = 152


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_convolution_gb300 import build
    build.build()


def _tiles(N, Ho, Wo, Co, bn):
    return -(-(N * Ho * Wo) // 128) * -(-Co // bn)


# N, Ci, H, W, Co, K, s, p, algos
PAIR_SHAPES = [
    # 256-wide channel tiles, two of them: streamed filter, one accumulator per issuer.
    (1, 8, 160, 160, 264, 3, 1, 1, ("implicit_tc", "padded_tc", "im2win_tc")),
    # 128-wide channel tile: resident filter with pairs.
    (1, 16, 224, 224, 128, 3, 1, 1, ("implicit_tc", "padded_tc", "im2win_tc")),
    # 64-wide channel tile, pairs, stride 2 on the implicit and window paths.
    (3, 24, 256, 256, 64, 3, 2, 1, ("implicit_tc", "im2win_tc")),
]


@pytest.mark.parametrize("tile_n", [0, 256, 176])
@pytest.mark.parametrize("shape", PAIR_SHAPES, ids=lambda s: "x".join(map(str, s[:8])))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_pairs_whole_output(shape, dtype, tile_n):
    N, Ci, H, W, Co, K, s, p, algos = shape
    if tile_n and Co <= 128:
        pytest.skip("one channel-tile width below 256 channels")
    Ho, Wo = (H + 2 * p - K) // s + 1, (W + 2 * p - K) // s + 1
    bn = tile_n or (64 if Co <= 64 else 128)
    assert _tiles(N, Ho, Wo, Co, bn) >= 2 * SMS
    seed = sum(shape[:8]) * 31 + len(dtype)
    X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), dtype)
    Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, K, K), (2.0 / (Ci * K * K)) ** 0.5), dtype)
    Y, S = oracle_full(X64, W64, s, p)
    for algo in algos:
        y, used, _ = run_gpu(X, Wt, s, p, dtype, algo, tuning={"tile_n": tile_n} if tile_n else None)
        assert used == algo
        assert np.all(np.isfinite(y)), (algo, "unwritten outputs")
        err, bad0 = parity(y, Y, S)
        assert bad0 == 0 and err <= TOL[dtype], (shape, dtype, algo, err)


@pytest.mark.parametrize("name,n,dtype", [("vgg", 26, "f16"), ("vgg", 26, "bf16"), ("sweep_k3", 10, "f16"),
                                           ("sweep_k1", 16, "f16"), ("sweep_k5", 10, "f16")])
def test_workload_whole_output_with_pairs(name, n, dtype):
    """Benchmark layers at a batch large enough for pairs, automatic algorithm."""
    wl = synth.WORKLOADS[name]
    Ho, Wo = wl.out_hw()
    bn = 64 if wl.Co <= 64 else (128 if wl.Co <= 128 else 176)
    assert _tiles(n, Ho, Wo, wl.Co, bn) >= 2 * SMS
    d = synth.make_inputs(wl, dtype, N=n)
    Y, S = oracle_full(d["X64"], d["W64"], wl.stride, wl.pad)
    y, used, _ = run_gpu(d["X"], d["W"], wl.stride, wl.pad, dtype, "auto")
    assert np.all(np.isfinite(y)), "unwritten outputs"
    err, bad0 = parity(y, Y, S)
    assert bad0 == 0 and err <= TOL[dtype], (name, dtype, used, err)


def _exact_expected(Y, dtype):
    import torch
    t = torch.from_numpy(Y.astype(np.float32))
    t = t.half() if dtype == "f16" else t.bfloat16()
    return t.double().numpy()


@pytest.mark.parametrize("tile_n", [256, 176, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_pairs_small_integers_bit_exact(dtype, tile_n):
    """Small integers make every order of summation exact: the pair path must
    match the oracle bit for bit after the one rounding to the output type."""
    from dense_convolution_gb300 import capi
    N, Ci, H, W, Co, K, s, p = 2, 8, 128, 128, 264, 3, 1, 1
    assert _tiles(N, H, W, Co, 256) >= 2 * SMS
    lo, hi = (-3, 3) if dtype == "f16" else (-1, 1)
    d = synth.make_int_inputs(4242 + len(dtype), N, Ci, H, W, Co, K, K, dtype, lo, hi)
    Y, _ = oracle_full(d["X64"], d["W64"], s, p)
    assert np.max(np.abs(Y)) < 2048
    expect = _exact_expected(Y, dtype)
    for algo in ("implicit_tc", "padded_tc", "im2win_tc"):
        y, _, _ = run_gpu(d["X"], d["W"], s, p, dtype, algo, tuning={"tile_n": tile_n})
        mism = np.argwhere(y != expect)
        assert mism.size == 0, (algo, mism[:5].tolist())
    assert capi.conv2d_device_status(0) == 0


def test_cv4_batch32_sampled():
    """The im2win paper's cv4 (64 x 224 x 224 -> 64, 7x7, stride 2, floor
    output size 109) at batch 32 on sampled outputs."""
    from oracle import ref
    from tests.test_parity_gpu import _sample_idx
    wl = synth.WORKLOADS["cv4"]
    d = synth.make_inputs(wl, "f16", N=32)
    y, used, _ = run_gpu(d["X"], d["W"], wl.stride, wl.pad, "f16", "auto")
    N, Co, Ho, Wo = y.shape
    assert (Ho, Wo) == (109, 109)
    idx = _sample_idx(N, Co, Ho, Wo, np.random.default_rng(wl.seed))
    Ys, Ss = ref.conv2d_points(d["X64"], d["W64"], idx, wl.stride, wl.pad)
    err, bad0 = parity(y.ravel()[idx], Ys, Ss)
    assert bad0 == 0 and err <= TOL["f16"], (used, err)
    assert np.all(np.isfinite(y))
