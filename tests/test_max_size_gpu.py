"""The largest input the tensor-core paths accept: N*Ci*H*W just under 2^31
elements (4.3 GB of fp16 X, as much Y and an operand copy of the same size),
so that every element index and byte offset of the copies, the TMA
coordinates and the epilogue's stores run at the top of their ranges.  X is
small integers made on the device (a hash of the element index), W small
integers, so every output is exact: windows cut from X at the first rows and
columns, in the middle and at the last rows and columns go through the
oracle, and the GPU output there must match bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from tests.helpers import oracle_full

pytestmark = pytest.mark.gpu

N, CI, HW, CO, K = 1, 64, 5792, 64, 3          # 64 * 5792^2 = 2,147,024,896 < 2^31 elements


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 24 * 2 ** 30:
        pytest.skip("needs about 16 GB of free device memory")
    from dense_convolution_gb300 import build
    build.build()


def _device_x():
    """X[i] = (hash(i) mod 3) - 1 for the flat NCHW index i, in fp16."""
    n = N * CI * HW * HW
    x = torch.empty(n, dtype=torch.float16, device="cuda")
    step = 1 << 27
    for a in range(0, n, step):
        i = torch.arange(a, min(n, a + step), dtype=torch.int64, device="cuda")
        x[a:a + i.numel()] = (((i * 2654435761) >> 13) % 3 - 1).to(torch.float16)
    return x.view(N, CI, HW, HW)


@pytest.mark.parametrize("algo", ["implicit_tc", "padded_tc"])
def test_largest_input_exact_windows(algo):
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    x = _device_x()
    d = synth.make_int_inputs(9300, 1, CI, 1, 1, CO, K, K, "f16", -2, 2)
    w = torch.from_numpy(d["W"]).cuda()
    op = Conv2d(N, CI, HW, HW, CO, K, K, 1, 1, "f16", algo)
    assert op.algo == algo
    y = op.alloc_output()
    y.fill_(float("nan"))
    ws = op.alloc_workspace()
    op(x, w, y, ws)
    torch.cuda.synchronize()
    assert capi.conv2d_device_status(0) == 0
    del ws
    # (crop origin, output rows/cols of the crop that see only real neighbours or real padding)
    for r0, c0 in ((0, 0), (HW // 2 - 17, HW // 3 - 17), (HW - 34, HW - 34)):
        xc = x[:, :, r0:r0 + 34, c0:c0 + 34].double().cpu().numpy()
        Yc, _ = oracle_full(xc, d["W64"], 1, 1)
        assert np.max(np.abs(Yc)) < 2048
        ra = 0 if r0 == 0 else 1
        rb = 34 if r0 + 34 == HW else 33
        ca = 0 if c0 == 0 else 1
        cb = 34 if c0 + 34 == HW else 33
        expect = torch.from_numpy(Yc[:, :, ra:rb, ca:cb].astype(np.float32)).half().double().numpy()
        got = y[:, :, r0 + ra:r0 + rb, c0 + ca:c0 + cb].double().cpu().numpy()
        mism = np.argwhere(got != expect)
        assert mism.size == 0, (algo, r0, c0, mism[:5].tolist())
