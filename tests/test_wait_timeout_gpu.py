"""The bounded-wait path of the kernels, exercised on the GPU without any wait
that never ends.

Every pipeline wait of the library's kernels gives up after a limit (2 s by
default): the kernel then lets the copies and MMAs it already issued finish,
exits, and sets the device status bit that conv2d_device_status reports as
CONV2D_ERR_DEVICE_TIMEOUT.  Here the limit is lowered to 1 ns so that
ordinary waits (for a copy to land, for the tensor core to finish a tile)
give up; nothing is held back and nothing is skipped.  The test checks that
the status comes back as a timeout, that the context stays usable, and that
the next call with the default limit gives the same bits as before.
"""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_convolution_gb300 import build
    build.build()


@pytest.mark.parametrize("name,n,dtype,algo", [("vgg", 8, "f16", "implicit_tc"),
                                                ("resnet_stage1", 4, "f16", "padded_tc"),
                                                ("resnet_stage1", 2, "f32", "im2win_fp32_cc"),
                                                ("sweep_k1", 16, "f16", "implicit_tc")])
def test_wait_limit_expires_and_recovers(name, n, dtype, algo):
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl, dtype, N=n)
    op = Conv2d(n, wl.Ci, wl.H, wl.W, wl.Co, wl.Kh, wl.Kw, wl.stride, wl.pad, dtype, algo)
    x = (torch.from_numpy(d["X"]) if dtype != "bf16" else d["X"]).cuda()
    w = (torch.from_numpy(d["W"]) if dtype != "bf16" else d["W"]).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    assert capi.conv2d_device_status(stream) == 0
    ref_y = op(x, w)
    torch.cuda.synchronize()
    assert capi.conv2d_device_status(stream) == 0
    timed_out = False
    try:
        capi.conv2d_set_wait_limit(1, stream)
        for _ in range(3):              # a wait that is never contended cannot expire; retry a few calls
            op(x, w)
            torch.cuda.synchronize()
            code = capi.conv2d_device_status(stream)
            if code:
                assert code & 1, code
                timed_out = True
                break
    finally:
        capi.conv2d_set_wait_limit(0, stream)
    assert timed_out, "no wait gave up under a 1 ns limit"
    # The context is still usable and the default limit is back.
    y = op(x, w)
    torch.cuda.synchronize()
    assert capi.conv2d_device_status(stream) == 0
    assert torch.equal(y.view(torch.int16) if y.element_size() == 2 else y.view(torch.int32),
                       ref_y.view(torch.int16) if ref_y.element_size() == 2 else ref_y.view(torch.int32))
