"""The split tail (opt-in, CONV2D_TUNE_SPLIT): when the tile groups of a call do not divide evenly over the
SMs, the filter-tap stages of the last partial wave are spread over all CTAs;
each group's first CTA adds the other CTAs' fp32 partial sums (published with
a per-call epoch flag) before its epilogue.  Only the summation order changes:

- whole outputs against the fp64 oracle at the 16-bit contract (NaN-poisoned,
  workspace guard bytes), including a layer whose tail groups are each split
  over about twenty CTAs;
- small integers, where every order gives the same sums, bit for bit;
- the split and the unsplit call within tolerance of each other, and two
  calls in a row (the flags of the first must not satisfy the second).
"""
import numpy as np
import pytest
import torch

import synth
from tests.helpers import TOL, oracle_full, parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_convolution_gb300 import build
    build.build()


def _split_bytes(shape, dtype, algo):
    from dense_convolution_gb300 import capi
    d = capi.conv2d_desc_create(*shape, dtype, algo)
    try:
        a = capi.conv2d_workspace_size(d)
        capi.conv2d_desc_set_tuning(d, "split", 1)
        return capi.conv2d_workspace_size(d) - a
    finally:
        capi.conv2d_desc_destroy(d)


CASES = [
    # (N, Ci, H, W, Co, K, s, p), dtype, algo
    ((26, 512, 28, 28, 512, 3, 1, 1), "f16", "implicit_tc"),     # 8 tail groups, each over ~19 CTAs
    ((40, 512, 28, 28, 512, 3, 1, 1), "bf16", "implicit_tc"),
    ((16, 128, 64, 64, 128, 3, 1, 1), "f16", "padded_tc"),       # the K3 sweep layer, halo mode
    ((16, 128, 64, 64, 128, 7, 1, 3), "f16", "implicit_tc"),     # the K7 sweep layer
    ((16, 64, 56, 56, 64, 3, 1, 1), "f16", "padded_tc"),         # 64-wide channel tiles, resident filter
    ((10, 128, 64, 64, 128, 3, 1, 1), "f16", "padded_tc"),       # under one stage per CTA: empty shares
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[2] + "-" + "x".join(map(str, c[0])))
def test_split_tail_whole_output(case):
    (N, Ci, H, W, Co, K, s, p), dtype, algo = case
    shape = (N, Ci, H, W, Co, K, K, s, p)
    if _split_bytes(shape, dtype, algo) == 0:
        pytest.skip("the tile groups divide evenly on this GPU: no split")
    seed = N * 31 + Ci + K
    X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), dtype)
    Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, K, K), (2.0 / (Ci * K * K)) ** 0.5), dtype)
    Y, S = oracle_full(X64, W64, s, p)
    y, used, _ = run_gpu(X, Wt, s, p, dtype, algo, tuning={"split": 1})
    assert np.all(np.isfinite(y))
    err, bad0 = parity(y, Y, S)
    assert bad0 == 0 and err <= TOL[dtype], (case, err)


def test_split_tail_small_integers_bit_exact():
    shape = (26, 512, 28, 28, 512, 3, 3, 1, 1)
    if _split_bytes(shape, "f16", "implicit_tc") == 0:
        pytest.skip("no split on this GPU")
    N, Ci, H, W, Co, Kh, Kw, s, p = shape
    d = synth.make_int_inputs(777, N, Ci, H, W, Co, Kh, Kw, "f16", -1, 1)
    Y, _ = oracle_full(d["X64"], d["W64"], s, p)
    assert np.max(np.abs(Y)) < 2048
    expect = torch.from_numpy(Y.astype(np.float32)).half().double().numpy()
    y, _, _ = run_gpu(d["X"], d["W"], s, p, "f16", "implicit_tc", tuning={"split": 1})
    mism = np.argwhere(y != expect)
    assert mism.size == 0, mism[:5].tolist()


def test_split_matches_unsplit_and_repeats():
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    wl = synth.WORKLOADS["vgg"]
    d = synth.make_inputs(wl, "f16", N=26)
    x, w = torch.from_numpy(d["X"]).cuda(), torch.from_numpy(d["W"]).cuda()
    split = Conv2d(26, 512, 28, 28, 512, 3, 3, 1, 1, "f16", "implicit_tc", tuning={"split": 1})
    plain = Conv2d(26, 512, 28, 28, 512, 3, 3, 1, 1, "f16", "implicit_tc")
    ws = split.alloc_workspace()
    ys = []
    for _ in range(2):                  # same workspace: the first call's flags hold the older epoch
        y = split.alloc_output()
        y.fill_(float("nan"))
        split(x, w, y, ws)
        ys.append(y)
    ref = plain(x, w)
    torch.cuda.synchronize()
    assert capi.conv2d_device_status(0) == 0
    assert torch.equal(ys[0], ys[1])
    _, S = oracle_full(d["X64"][:2], d["W64"], 1, 1)          # scale of the first two images
    a = ys[0][:2].double().cpu().numpy()
    b = ref[:2].double().cpu().numpy()
    err, bad0 = parity(a, b, S)
    assert bad0 == 0 and err <= TOL["f16"]
