"""conv2d_fwd_static_workspace: the entry point for callers that cannot
allocate device memory (their host application owns all of it, or a
cudaMalloc's synchronisation is not affordable).  Its scratch is the
library's built-in device array, so the caller passes only x, w and y.

Checked here through the C ABI: two calls in a row give the same result as
conv2d_fwd with a caller-allocated workspace (within the parity tolerance of
the other tests), and a descriptor that needs more scratch than the array
holds is refused before anything is launched.  This file is collected last
so that a run stopping at the first failure has run every other test first.
"""
import numpy as np
import pytest

import synth
from tests.helpers import TOL, oracle_full, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_convolution_gb300 import build
    build.build()


@pytest.mark.parametrize("name,dtype,algo", [("resnet_stage1", "f16", "auto"), ("tiny", "f32", "auto"),
                                              ("stem", "bf16", "im2win_tc"), ("vgg", "bf16", "auto")])
def test_static_workspace_matches_fwd(name, dtype, algo):
    import torch
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    wl = synth.WORKLOADS[name]
    n = 1 if name in ("stem", "vgg", "tiny") else 2
    d = synth.make_inputs(wl, dtype, N=n)
    op = Conv2d(n, wl.Ci, wl.H, wl.W, wl.Co, wl.Kh, wl.Kw, wl.stride, wl.pad, dtype, algo)
    assert 0 < op.workspace_bytes <= capi.STATIC_WORKSPACE_BYTES
    x = (torch.from_numpy(d["X"]) if dtype != "bf16" else d["X"]).cuda()
    w = (torch.from_numpy(d["W"]) if dtype != "bf16" else d["W"]).cuda()
    ref_y = op(x, w)                                   # caller-allocated workspace
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(2):                                 # two calls in a row share the array
        y = op.alloc_output()
        y.fill_(float("nan"))
        capi.conv2d_fwd_static_workspace(op.desc, x.data_ptr(), w.data_ptr(), y.data_ptr(), stream)
        outs.append(y)
    torch.cuda.synchronize()
    assert capi.conv2d_device_status(stream) == 0
    _, S = oracle_full(d["X64"], d["W64"], wl.stride, wl.pad)
    r = ref_y.double().cpu().numpy()
    for y in outs:
        yv = y.double().cpu().numpy()
        assert np.all(np.isfinite(yv))
        err, bad0 = parity(yv, r, S)
        assert bad0 == 0 and err <= TOL[dtype], err


def test_static_workspace_refuses_oversized_problem():
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    # Stem layer at batch 64, im2win window tensor: about 79 MB of scratch.
    op = Conv2d(64, 3, 224, 224, 64, 7, 7, 2, 3, "f16", "im2win_tc")
    assert op.workspace_bytes > capi.STATIC_WORKSPACE_BYTES
    with pytest.raises(capi.Conv2dError) as e:
        capi.conv2d_fwd_static_workspace(op.desc, 1 << 20, 1 << 20, 1 << 20, 0)
    assert e.value.status == capi.ERR_WORKSPACE_TOO_SMALL
