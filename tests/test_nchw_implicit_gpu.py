"""GPU parity of the implicit GEMM on NCHW input at stride 1, where the
contraction kernel builds its operand tiles from X itself (the implicit
expansion of "im2col Expansion, FFT Convolution, and Winograd Transforms",
im2col section: indices computed in the load path, no expansion buffer).

The workspace must be the repacked filter alone and a call two launches.
Shapes cover every vector width of the in-kernel loads (W divisible by 8, 4,
2 or odd), valid and wide padding (junk rows of the virtual grid), Kh != Kw,
filters too tall for one halo (several filter-row groups), channel counts off
the 64-wide chunk and off the output tile, and batches large enough for tile
pairs.  Whole outputs are compared with the fp64 oracle (NaN-poisoned y,
workspace guard bytes), and small integers bit for bit.
"""
import numpy as np
import pytest

import synth
from tests.helpers import TOL, oracle_full, parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_convolution_gb300 import build
    build.build()


def _packed_bytes(Ci, Co, Kh, Kw):
    ci8 = (Ci + 7) // 8 * 8
    return Co * Kh * Kw * ((ci8 + 63) // 64 * 64) * 2


SHAPES = [
    # N, Ci, H, W, Co, Kh, Kw, p
    (2, 64, 14, 16, 64, 3, 3, 1),      # W % 8 == 0
    (2, 64, 14, 28, 64, 3, 3, 1),      # W % 4 == 0 (the VGG width)
    (1, 24, 9, 18, 40, 3, 3, 1),       # W % 2 == 0, channels off the chunk
    (1, 13, 11, 13, 17, 3, 5, 2),      # odd W (scalar loads), Kh != Kw
    (2, 72, 10, 12, 136, 3, 3, 0),     # valid convolution: junk rows and columns; two chunks
    (1, 16, 12, 16, 24, 3, 3, 3),      # padding wider than the filter's reach
    (1, 8, 20, 64, 16, 11, 11, 5),     # tall filter on a wide map: several filter-row groups per chunk
    (1, 130, 8, 8, 300, 5, 5, 2),      # three chunks, two 256-wide channel tiles
    (1, 1, 7, 7, 1, 1, 1, 1),          # 1x1 filter with padding (not the in-place GEMM)
    (3, 64, 56, 56, 64, 3, 3, 1),      # ResNet stage 1 shape, tile pairs
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_nchw_implicit_whole_output(shape, dtype):
    from dense_convolution_gb300 import capi
    N, Ci, H, W, Co, Kh, Kw, p = shape
    seed = sum(shape) * 53 + len(dtype)
    X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), dtype)
    Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, Kh, Kw), (2.0 / (Ci * Kh * Kw)) ** 0.5), dtype)
    Y, S = oracle_full(X64, W64, 1, p)
    y, used, ws = run_gpu(X, Wt, 1, p, dtype, "implicit_nchw_tc")
    assert used == "implicit_nchw_tc" and ws == _packed_bytes(Ci, Co, Kh, Kw)
    err, bad0 = parity(y, Y, S)
    assert bad0 == 0 and err <= TOL[dtype], (shape, dtype, err)
    d = capi.conv2d_desc_create(N, Ci, H, W, Co, Kh, Kw, 1, p, dtype, "implicit_nchw_tc")
    try:
        assert capi.conv2d_launches_per_call(d) == 2
    finally:
        capi.conv2d_desc_destroy(d)


@pytest.mark.parametrize("shape", [(2, 8, 128, 128, 264, 3, 3, 1), (1, 24, 9, 18, 40, 3, 3, 1),
                                   (1, 13, 11, 13, 17, 3, 5, 2), (2, 72, 10, 12, 136, 3, 3, 0)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_nchw_implicit_small_integers_bit_exact(shape, dtype):
    import torch
    N, Ci, H, W, Co, Kh, Kw, p = shape
    lo, hi = (-3, 3) if dtype == "f16" else (-1, 1)
    d = synth.make_int_inputs(sum(shape) * 11 + len(dtype), N, Ci, H, W, Co, Kh, Kw, dtype, lo, hi)
    Y, _ = oracle_full(d["X64"], d["W64"], 1, p)
    assert np.max(np.abs(Y)) < 2048
    t = torch.from_numpy(Y.astype(np.float32))
    expect = (t.half() if dtype == "f16" else t.bfloat16()).double().numpy()
    y, _, _ = run_gpu(d["X"], d["W"], 1, p, dtype, "implicit_nchw_tc")
    mism = np.argwhere(y != expect)
    assert mism.size == 0, mism[:5].tolist()
