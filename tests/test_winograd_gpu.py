"""GPU parity of the Winograd F(2x2, 3x3) fp32 path (openCNN, Sec. 2-3) against
the direct fp64 oracle: the fp32 contract max |y - Y| / sum|x*w| <= 1e-4 on
whole outputs (NaN-poisoned), on the benchmark's 3x3 stride-1 layers at
reduced batch, odd sizes (partial 2x2 tiles and tile blocks), padding 0..2,
channel counts off the 8-channel stage and the 64-channel block, bias; and
bit for bit on small integers, where every transformed value is a small
dyadic rational and every sum exact in fp32.
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


@pytest.mark.parametrize("name,n", [("resnet_stage1", 2), ("vgg", 1), ("sweep_k3", 1), ("tiny", 1), ("cv10", 1),
                                    ("cv12", 2)])
def test_winograd_workloads(name, n):
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl, "f32", N=n)
    Y, S = oracle_full(d["X64"], d["W64"], wl.stride, wl.pad)
    y, used, ws = run_gpu(d["X"], d["W"], wl.stride, wl.pad, "f32", "winograd_fp32_cc")
    assert used == "winograd_fp32_cc"
    err, bad0 = parity(y, Y, S)
    assert bad0 == 0 and err <= TOL["f32"], (name, err)


SHAPES = [  # N, Ci, H, W, Co, p
    (1, 1, 1, 1, 1, 1), (2, 3, 5, 7, 5, 1), (1, 13, 17, 19, 70, 1), (1, 8, 10, 10, 64, 0), (2, 20, 9, 33, 130, 2),
    (1, 64, 15, 15, 64, 1), (3, 5, 4, 4, 3, 0),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_winograd_shapes(shape):
    N, Ci, H, W, Co, p = shape
    seed = sum(shape) * 7
    X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), "f32")
    Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, 3, 3), (2.0 / (Ci * 9)) ** 0.5), "f32")
    Y, S = oracle_full(X64, W64, 1, p)
    y, _, _ = run_gpu(X, Wt, 1, p, "f32", "winograd_fp32_cc")
    err, bad0 = parity(y, Y, S)
    assert bad0 == 0 and err <= TOL["f32"], (shape, err)


def test_winograd_bias():
    from dense_convolution_gb300.conv import Conv2d
    from oracle import ref
    X, X64 = synth.round_to(synth.normal(3, 0, (2, 24, 20, 18)), "f32")
    Wt, W64 = synth.round_to(synth.normal(3, 1, (96, 24, 3, 3), 0.1), "f32")
    B, B64 = synth.round_to(synth.normal(3, 2, (96,)), "f32")
    Y, S = oracle_full(X64, W64, 1, 1)
    ref.add_bias(Y, S, B64)
    op = Conv2d(2, 24, 20, 18, 96, 3, 3, 1, 1, "f32", "winograd_fp32_cc")
    y = op(torch.from_numpy(X).cuda(), torch.from_numpy(Wt).cuda(), bias=torch.from_numpy(B).cuda())
    err, bad0 = parity(y.double().cpu().numpy(), Y, S)
    assert bad0 == 0 and err <= TOL["f32"], err


@pytest.mark.parametrize("shape", [(2, 16, 14, 14, 64, 1), (1, 9, 7, 11, 70, 2), (1, 64, 28, 28, 128, 1)],
                         ids=lambda s: "x".join(map(str, s)))
def test_winograd_small_integers_bit_exact(shape):
    N, Ci, H, W, Co, p = shape
    d = synth.make_int_inputs(sum(shape) * 3, N, Ci, H, W, Co, 3, 3, "f32", -3, 3)
    Y, _ = oracle_full(d["X64"], d["W64"], 1, p)
    y, _, _ = run_gpu(d["X"], d["W"], 1, p, "f32", "winograd_fp32_cc")
    mism = np.argwhere(y != Y)
    assert mism.size == 0, mism[:5].tolist()
