"""Options in combination: input layout (NCHW, or NHWC on the implicit
tensor-core path), per-channel bias, fp32 output for 16-bit inputs, a
pre-packed filter and the number of epilogue warp groups, drawn as seeded
combinations over every algorithm and a few shapes (single tiles and pairs,
Kh = Kw = 5, stride 2).  Each call runs on a NaN-poisoned output and is held
to the oracle (with the bias added by oracle_add_bias) at the contract
tolerance: 1e-4 for fp32 inputs, 1e-2 for 16-bit outputs, 1e-3 for fp32
outputs of 16-bit inputs.
"""
import itertools
import random

import numpy as np
import pytest
import torch

import synth
from tests.helpers import oracle_full, parity

pytestmark = pytest.mark.gpu

SHAPES = [
    # N, Ci, H, W, Co, K, s, p
    (2, 64, 20, 24, 96, 3, 1, 1),
    (3, 16, 17, 20, 64, 5, 1, 2),
    (2, 32, 15, 15, 128, 3, 2, 1),
    (8, 64, 56, 56, 64, 3, 1, 1),      # tile pairs
]
ALGOS = {"f16": ["implicit_tc", "padded_tc", "im2win_tc", "implicit_nchw_tc"],
         "bf16": ["implicit_tc", "padded_tc", "im2win_tc", "implicit_nchw_tc"],
         "f32": ["im2win_fp32_cc", "implicit_fp32_cc", "winograd_fp32_cc"]}


def _valid(shape, dtype, algo):
    N, Ci, H, W, Co, K, s, p = shape
    if algo in ("padded_tc", "implicit_nchw_tc") and s != 1:
        return False
    if algo == "winograd_fp32_cc" and (K != 3 or s != 1):
        return False
    if algo == "implicit_fp32_cc" and W % 4 != 0:
        return False
    return True


def _combos():
    rng = random.Random(20261202)
    out = []
    for dtype, algos in ALGOS.items():
        for si, shape in enumerate(SHAPES):
            for algo in algos:
                if not _valid(shape, dtype, algo):
                    continue
                layouts = ["nchw", "nhwc"] if algo == "implicit_tc" and shape[1] % 8 == 0 else ["nchw"]
                outs = [dtype, "f32"] if dtype != "f32" else ["f32"]
                epis = [0, 3] if algo in ("implicit_tc", "padded_tc", "im2win_tc") else [0]
                allc = list(itertools.product(layouts, [False, True], outs, [False, True], epis))
                for c in rng.sample(allc, min(4, len(allc))):
                    out.append((dtype, si, algo) + c)
    return out


CASES = _combos()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_convolution_gb300 import build
    build.build()


_REF = {}


def _reference(dtype, si):
    if (dtype, si) not in _REF:
        N, Ci, H, W, Co, K, s, p = SHAPES[si]
        seed = 9900 + 10 * si + len(dtype)
        X, X64 = synth.round_to(synth.normal(seed, 0, (N, Ci, H, W)), dtype)
        Wt, W64 = synth.round_to(synth.normal(seed, 1, (Co, Ci, K, K), (2.0 / (Ci * K * K)) ** 0.5), dtype)
        b, b64 = synth.round_to(synth.normal(seed, 2, (Co,), 0.5), dtype)
        Y, S = oracle_full(X64, W64, s, p)
        _REF[(dtype, si)] = (X, Wt, b, b64, Y, S)
    return _REF[(dtype, si)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(str(v) for v in c))
def test_option_combination(case):
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    from oracle import ref
    dtype, si, algo, layout, with_bias, out_dtype, prepacked, epi = case
    N, Ci, H, W, Co, K, s, p = SHAPES[si]
    X, Wt, b, b64, Y, S = _reference(dtype, si)
    tuning = {"epi_groups": epi} if epi else None
    op = Conv2d(N, Ci, H, W, Co, K, K, s, p, dtype, algo, layout, out_dtype=out_dtype, tuning=tuning)
    assert op.algo == algo
    as_t = lambda a: (torch.from_numpy(a) if not isinstance(a, torch.Tensor) else a).cuda()
    x = as_t(X)
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous()
    w = as_t(Wt)
    if prepacked:
        w = op.pack_filter(w)
        op.set_prepacked(True)
    bias = as_t(b) if with_bias else None
    y = op.alloc_output()
    y.fill_(float("nan"))
    op(x, w, y, bias=bias)
    torch.cuda.synchronize()
    assert capi.conv2d_device_status(0) == 0
    got = y.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    Yr, Sr = Y.copy(), S.copy()
    if with_bias:
        ref.add_bias(Yr, Sr, b64)
    err, bad0 = parity(got, Yr, Sr)
    tol = 1e-4 if dtype == "f32" else (1e-3 if out_dtype == "f32" else 1e-2)
    assert bad0 == 0 and err <= tol, (case, err)
