"""Pipeline knobs (conv2d_desc_set_tuning) change only how copies overlap and
in which order output tiles are visited, never a sum: every setting must give
the same bits as the default, on every algorithm, and stay within tolerance
of the oracle.  Cases reach tile pairs, a streamed and a resident filter, the
1x1 GEMM, the in-kernel NCHW path and the CUDA-core kernel.
"""

import numpy as np
import pytest
import torch

import synth
from tests.helpers import TOL, oracle_full, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_convolution_gb300 import build
    build.build()


CASES = [
    # (N, Ci, H, W, Co, K, s, p), dtype, algo
    ((1, 8, 160, 160, 264, 3, 1, 1), "f16", "implicit_tc"),      # pairs, two 256-wide channel tiles
    ((3, 64, 56, 56, 64, 3, 1, 1), "f16", "padded_tc"),          # pairs, resident filter
    ((2, 24, 64, 64, 64, 3, 2, 1), "bf16", "im2win_tc"),         # stride 2 window path
    ((16, 128, 32, 32, 128, 1, 1, 0), "f16", "implicit_tc"),     # 1x1 GEMM
    ((2, 64, 28, 28, 128, 3, 1, 1), "f16", "implicit_nchw_tc"),  # in-kernel NCHW halo
    ((2, 16, 30, 30, 40, 3, 1, 1), "f32", "im2win_fp32_cc"),     # CUDA cores
    ((2, 16, 30, 32, 40, 5, 1, 2), "f32", "implicit_fp32_cc"),
    ((8, 3, 64, 64, 64, 3, 1, 0), "f16", "im2win_tc"),           # three-channel window, pairs, 64-wide tiles
    ((4, 32, 40, 40, 96, 5, 1, 2), "bf16", "implicit_tc"),       # 128-wide tiles (single tiles with 3 groups)
    ((8, 64, 56, 56, 64, 3, 1, 1), "f16", "padded_tc"),          # many pairs per CTA
]

# (The opt-in split tail changes the summation order of the split tiles; it
# has its own tests.)
SETTINGS = [{"stages": 1}, {"stages": 2}, {"sync_copies": 1}, {"raster": 1}, {"raster": 2}, {"no_resident": 1},
            {"stages": 1, "raster": 2, "sync_copies": 1}, {"epi_groups": 2}, {"epi_groups": 3},
            {"epi_groups": 3, "stages": 1}, {"tile_n": 128}, {"tile_n": 256}, {"tile_n": 64}]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[2] + "-" + "x".join(map(str, c[0])))
def test_knobs_keep_the_bits(case):
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    (N, Ci, H, W, Co, K, s, p), dtype, algo = case
    seed = N * 1000 + Ci + Co + K
    X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), dtype)
    Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, K, K), (2.0 / (Ci * K * K)) ** 0.5), dtype)
    x = (torch.from_numpy(X) if not isinstance(X, torch.Tensor) else X).cuda()
    w = (torch.from_numpy(Wt) if not isinstance(Wt, torch.Tensor) else Wt).cuda()
    ref = Conv2d(N, Ci, H, W, Co, K, K, s, p, dtype, algo)(x, w)
    torch.cuda.synchronize()
    Y, S = oracle_full(X64, W64, s, p)
    err, bad0 = parity(ref.double().cpu().numpy(), Y, S)
    assert bad0 == 0 and err <= TOL[dtype]
    for tune in SETTINGS:
        op = Conv2d(N, Ci, H, W, Co, K, K, s, p, dtype, algo, tuning=tune)
        y = op.alloc_output()
        y.fill_(float("nan"))
        op(x, w, y)
        torch.cuda.synchronize()
        assert capi.conv2d_device_status(0) == 0
        view = torch.int16 if y.element_size() == 2 else torch.int32
        assert torch.equal(y.view(view), ref.view(view)), (algo, tune)
