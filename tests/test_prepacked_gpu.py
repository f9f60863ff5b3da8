"""Pre-packed filters: conv2d_pack_filter once, then conv2d_fwd with the
packed filter (no repack launch, smaller workspace).  The kernels see the same
operands, so every algorithm must give the same bits as the ordinary call, on
two calls in a row, and the same through conv2d_fwd_host.
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


CASES = [("resnet_stage1", 2, "f16", "padded_tc"), ("resnet_stage1", 2, "bf16", "implicit_tc"),
         ("resnet_stage1", 2, "f16", "implicit_nchw_tc"), ("stem", 1, "f16", "im2win_tc"),
         ("sweep_k1", 4, "f16", "implicit_tc"), ("vgg", 2, "f16", "implicit_tc"),
         ("tiny", 1, "f32", "im2win_fp32_cc"), ("tiny", 1, "f32", "implicit_fp32_cc"),
         ("resnet_stage1", 1, "f32", "winograd_fp32_cc")]


@pytest.mark.parametrize("name,n,dtype,algo", CASES)
def test_prepacked_matches_ordinary_call(name, n, dtype, algo):
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl, dtype, N=n)
    x = (torch.from_numpy(d["X"]) if dtype != "bf16" else d["X"]).cuda()
    w = (torch.from_numpy(d["W"]) if dtype != "bf16" else d["W"]).cuda()
    op = Conv2d(n, wl.Ci, wl.H, wl.W, wl.Co, wl.Kh, wl.Kw, wl.stride, wl.pad, dtype, algo)
    ref = op(x, w)
    n_launch = capi.conv2d_launches_per_call(op.desc)
    wp = op.pack_filter(w)
    op.set_prepacked(True)
    assert capi.conv2d_launches_per_call(op.desc) == (1 if n_launch == 1 else n_launch - 1)
    view = torch.int16 if ref.element_size() == 2 else torch.int32
    for _ in range(2):
        y = op.alloc_output()
        y.fill_(float("nan"))
        op(x, wp, y)
        torch.cuda.synchronize()
        assert capi.conv2d_device_status(0) == 0
        assert torch.equal(y.view(view), ref.view(view)), (name, algo)
    # Host-buffer call with the packed filter copied in.
    xh, wh = x.cpu().pin_memory(), wp.cpu().pin_memory()
    yh = torch.empty(ref.shape, dtype=ref.dtype).pin_memory()
    xd, wd, yd = torch.empty_like(x), torch.empty_like(wp), op.alloc_output()
    ws = op.alloc_workspace()
    st = torch.cuda.current_stream()
    capi.conv2d_fwd_host(op.desc, xh.data_ptr(), wh.data_ptr(), yh.data_ptr(), xd.data_ptr(), wd.data_ptr(),
                         yd.data_ptr(), ws.data_ptr() if op.workspace_bytes else 0, op.workspace_bytes, st.cuda_stream)
    st.synchronize()
    assert torch.equal(yh.view(view), ref.cpu().view(view))
