"""GPU parity of the bias epilogue and of fp32 output for 16-bit inputs.

Bias: one value per output channel added after the sum, the `Y_col += bias`
of the PyTorch listing in "Unifying Convolutions and GEMM", Sec. 6; the
oracle adds b[co] to Y and |b[co]| to sum|x*w| (oracle_add_bias).  fp32
output: the fp32 accumulator stored without the rounding to 16 bits.

Every algorithm runs through the C ABI on NaN-poisoned outputs: whole
outputs against the oracle at the contract tolerance (1e-2 for 16-bit inputs,
1e-4 for fp32; fp32 outputs of 16-bit inputs are also held to 1e-3, since
nothing rounds them to 16 bits), and small integers with integer biases,
where every result is exact, bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from tests.helpers import TOL, oracle_full, parity

pytestmark = pytest.mark.gpu

ALGOS = {"f32": ["im2win_fp32_cc", "implicit_fp32_cc"], "f16": ["im2win_tc", "implicit_tc", "padded_tc"],
         "bf16": ["im2win_tc", "implicit_tc", "padded_tc"]}
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_convolution_gb300 import build
    build.build()


def _run(X, Wt, b, s, p, dtype, algo, out_dtype):
    """One call with bias b (storage dtype) and output type out_dtype; returns y as float64."""
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    N, Ci, H, W = X.shape
    Co, _, Kh, Kw = Wt.shape
    op = Conv2d(N, Ci, H, W, Co, Kh, Kw, s, p, dtype, algo, out_dtype=out_dtype)
    x = (torch.from_numpy(X) if not isinstance(X, torch.Tensor) else X).cuda()
    w = (torch.from_numpy(Wt) if not isinstance(Wt, torch.Tensor) else Wt).cuda()
    bd = (torch.from_numpy(b) if not isinstance(b, torch.Tensor) else b).cuda() if b is not None else None
    y = op.alloc_output()
    assert y.dtype == TORCH[out_dtype]
    y.fill_(float("nan"))
    op(x, w, y, bias=bd)
    torch.cuda.synchronize()
    assert capi.conv2d_device_status(0) == 0
    return y.double().cpu().numpy(), op.algo


SHAPES = [
    # N, Ci, H, W, Co, Kh, Kw, s, p
    (2, 64, 14, 14, 64, 3, 3, 1, 1),        # single tiles, vector stores
    (2, 5, 17, 13, 7, 2, 3, 3, 1),          # odd sizes: scalar stores, few channels
    (1, 16, 9, 11, 300, 3, 5, 1, 2),        # two 256-wide channel tiles, Kh != Kw
    (1, 8, 160, 160, 264, 3, 3, 1, 1),      # tile pairs, streamed filter
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype,out_dtype", [("f16", "f16"), ("f16", "f32"), ("bf16", "bf16"), ("bf16", "f32"),
                                             ("f32", "f32")])
def test_bias_and_output_type(shape, dtype, out_dtype):
    from dense_convolution_gb300 import capi
    from oracle import ref
    N, Ci, H, W, Co, Kh, Kw, s, p = shape
    seed = sum(shape) * 41 + len(dtype) + 3 * len(out_dtype)
    X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), dtype)
    Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, Kh, Kw), (2.0 / (Ci * Kh * Kw)) ** 0.5), dtype)
    B, B64 = synth.round_to(synth.normal(seed, 2, (Co,)), dtype)
    Y, S = oracle_full(X64, W64, s, p)
    ref.add_bias(Y, S, B64)
    ran = 0
    for algo in ALGOS[dtype]:
        try:
            y, used = _run(X, Wt, B, s, p, dtype, algo, out_dtype)
        except capi.Conv2dError as e:
            assert e.status == capi.ERR_UNSUPPORTED
            continue
        ran += 1
        err, bad0 = parity(y, Y, S)
        tol = 1e-3 if (out_dtype == "f32" and dtype != "f32") else TOL[dtype]
        assert bad0 == 0 and err <= tol, (shape, dtype, out_dtype, algo, err)
    assert ran >= 1


GEMM_SHAPES = [(2, 200, 7, 8, 300), (3, 72, 10, 12, 17), (16, 128, 64, 64, 128)]


@pytest.mark.parametrize("shape", GEMM_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype,out_dtype", [("f16", "f32"), ("bf16", "bf16"), ("f16", "f16")])
def test_bias_and_output_type_1x1(shape, dtype, out_dtype):
    """The in-place 1x1 GEMM (TMA-store epilogue), including a batch with tile pairs."""
    from oracle import ref
    N, Ci, H, W, Co = shape
    seed = sum(shape) * 43 + len(dtype) + 3 * len(out_dtype)
    X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), dtype)
    Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, 1, 1), (2.0 / Ci) ** 0.5), dtype)
    B, B64 = synth.round_to(synth.normal(seed, 2, (Co,)), dtype)
    Y, S = oracle_full(X64, W64, 1, 0)
    ref.add_bias(Y, S, B64)
    y, used = _run(X, Wt, B, 1, 0, dtype, "implicit_tc", out_dtype)
    err, bad0 = parity(y, Y, S)
    tol = 1e-3 if out_dtype == "f32" else TOL[dtype]
    assert bad0 == 0 and err <= tol, (shape, dtype, out_dtype, err)


@pytest.mark.parametrize("shape", [(2, 8, 128, 128, 264, 3, 3, 1, 1), (1, 16, 9, 11, 24, 3, 5, 1, 2),
                                   (2, 64, 16, 16, 130, 1, 1, 1, 0)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype,out_dtype", [("f16", "f16"), ("f16", "f32"), ("bf16", "f32"), ("f32", "f32")])
def test_bias_small_integers_bit_exact(shape, dtype, out_dtype):
    """Integer inputs and biases: every result is an exact integer, so each
    algorithm must equal the oracle bit for bit (after the one rounding to a
    16-bit output type)."""
    from dense_convolution_gb300 import capi
    from oracle import ref
    N, Ci, H, W, Co, Kh, Kw, s, p = shape
    lo, hi = (-3, 3) if dtype != "bf16" else (-1, 1)
    d = synth.make_int_inputs(sum(shape) * 5 + len(dtype) + len(out_dtype), N, Ci, H, W, Co, Kh, Kw, dtype, lo, hi)
    B, B64 = synth.round_to(synth.small_ints(sum(shape), 2, (Co,), -8, 8), dtype)
    Y, S = oracle_full(d["X64"], d["W64"], s, p)
    ref.add_bias(Y, S, B64)
    assert np.max(np.abs(Y)) < 2048
    t = torch.from_numpy(Y.astype(np.float32))
    expect = (t.to(TORCH[out_dtype]) if out_dtype != "f32" else t).double().numpy()
    algos = ALGOS[dtype] if not (Kh == 1 and Kw == 1) else (["implicit_tc"] if dtype != "f32" else ALGOS["f32"])
    ran = 0
    for algo in algos:
        try:
            y, _ = _run(d["X"], d["W"], B, s, p, dtype, algo, out_dtype)
        except capi.Conv2dError as e:
            assert e.status == capi.ERR_UNSUPPORTED
            continue
        ran += 1
        mism = np.argwhere(y != expect)
        assert mism.size == 0, (algo, mism[:5].tolist())
    assert ran >= 1


def test_bias_cleared_between_calls():
    """A call without bias after one with bias gives the plain sum (the
    descriptor's bias pointer is replaced on every call of the tensor layer)."""
    from dense_convolution_gb300.conv import Conv2d
    X, _ = synth.round_to(synth.normal(7, 0, (1, 16, 12, 12)), "f16")
    Wt, _ = synth.round_to(synth.normal(7, 1, (32, 16, 3, 3), 0.1), "f16")
    B, _ = synth.round_to(synth.normal(7, 2, (32,)), "f16")
    op = Conv2d(1, 16, 12, 12, 32, 3, 3, 1, 1, "f16", "auto")
    x, w, b = torch.from_numpy(X).cuda(), torch.from_numpy(Wt).cuda(), torch.from_numpy(B).cuda()
    y0 = op(x, w)
    y1 = op(x, w, bias=b)
    y2 = op(x, w)
    torch.cuda.synchronize()
    assert torch.equal(y0, y2) and not torch.equal(y0, y1)
