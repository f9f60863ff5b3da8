"""The 16-bit operand copies in front of the tensor-core contraction: the
zero-padded channels-last grid (padded_tc) and the NHWC copy (implicit_tc on
NCHW input).  Each shape picks a copy variant: 8 or 4 image columns per lane
load (W, or H*W for the NHWC copy, a multiple of 8 or of 4), the byte-wise
fallback (neither), channel counts that leave a partial 64-channel chunk or a
single 8-channel vector, zero and wide padding, and rows split over several
segments.  Whole outputs against the oracle, NaN-poisoned output and a
workspace guard; small integers bit for bit.
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


CASES = [
    # (N, Ci, H, W, Co, K, s, p), algo
    ((2, 200, 16, 24, 32, 3, 1, 1), "padded_tc"),    # W % 8 == 0; chunks of 64, 64, 64 and 8 channels
    ((2, 72, 12, 28, 40, 3, 1, 1), "padded_tc"),     # W % 8 == 4: four columns per load
    ((2, 16, 11, 13, 24, 3, 1, 2), "padded_tc"),     # odd W: byte-wise copy
    ((1, 64, 16, 32, 64, 3, 1, 0), "padded_tc"),     # no padding
    ((2, 3, 20, 24, 16, 5, 1, 2), "padded_tc"),      # three channels: one 8-channel vector per pixel
    ((1, 16, 8, 520, 16, 3, 1, 1), "padded_tc"),     # a row in five segments
    ((2, 24, 14, 12, 32, 3, 1, 1), "implicit_tc"),   # H*W % 8 == 0
    ((2, 40, 10, 10, 32, 3, 1, 1), "implicit_tc"),   # H*W % 8 == 4
    ((1, 16, 9, 9, 16, 3, 1, 1), "implicit_tc"),     # odd H*W: byte-wise copy
    ((1, 8, 64, 64, 16, 3, 2, 1), "implicit_tc"),    # 4096-pixel plane in 32 segments
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c[1] + "-" + "x".join(map(str, c[0])))
def test_copy_variants_whole_output(case, dtype):
    (N, Ci, H, W, Co, K, s, p), algo = case
    seed = 7000 + N * 97 + Ci * 5 + W
    X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), dtype)
    Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, K, K), (2.0 / (Ci * K * K)) ** 0.5), dtype)
    Y, S = oracle_full(X64, W64, s, p)
    y, used, _ = run_gpu(X, Wt, s, p, dtype, algo)
    assert used == algo
    assert np.all(np.isfinite(y))
    err, bad0 = parity(y, Y, S)
    assert bad0 == 0 and err <= TOL[dtype], (case, err)


@pytest.mark.parametrize("case", [CASES[0], CASES[1], CASES[5], CASES[7], CASES[9]],
                         ids=lambda c: c[1] + "-" + "x".join(map(str, c[0])))
def test_copy_variants_small_integers_bit_exact(case):
    (N, Ci, H, W, Co, K, s, p), algo = case
    d = synth.make_int_inputs(8100 + Ci + W, N, Ci, H, W, Co, K, K, "f16", -2, 2)
    Y, _ = oracle_full(d["X64"], d["W64"], s, p)
    assert np.max(np.abs(Y)) < 2048
    expect = torch.from_numpy(Y.astype(np.float32)).half().double().numpy()
    y, used, _ = run_gpu(d["X"], d["W"], s, p, "f16", algo)
    assert used == algo
    mism = np.argwhere(y != expect)
    assert mism.size == 0, mism[:5].tolist()
