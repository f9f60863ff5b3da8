"""Shared helpers for the GPU parity tests: run the library through its C ABI
on seeded inputs and compare with the oracle."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

TOL = {"f32": 1e-4, "f16": 1e-2, "bf16": 1e-2}   # max |y - Y| / sum|x*w|


def oracle_full(X64, W64, s, p, threads=None):
    """Whole output from the oracle, split over output-channel slices on host
    threads (the C routine releases the GIL)."""
    from oracle import ref
    N, Ci, H, W = X64.shape
    Co, _, Kh, Kw = W64.shape
    Ho, Wo = ref.out_dims(H, W, Kh, Kw, s, p)
    Y = np.empty((N, Co, Ho, Wo))
    S = np.empty_like(Y)
    X64 = np.ascontiguousarray(X64)
    W64 = np.ascontiguousarray(W64)
    threads = threads or min(32, os.cpu_count() or 1)
    step = max(1, (Co + threads - 1) // threads)
    jobs = [(n, co, min(Co, co + step)) for n in range(N) for co in range(0, Co, step)]
    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda j: ref.conv2d_slice(X64, W64, Y, S, s, p, j[0], j[0] + 1, j[1], j[2]), jobs))
    return Y, S


def to_device(arr, dtype):
    import torch
    if isinstance(arr, torch.Tensor):
        return arr.contiguous().cuda()
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def run_gpu(X, W, s, p, dtype, algo="auto", layout="nchw", poison=True, guard=True, tuning=None):
    """Run one convolution through the C ABI.  Returns (y float64 numpy,
    algo used, workspace bytes).  The output is pre-filled with NaN and the
    workspace is followed by a guard region that must stay untouched."""
    import torch
    from dense_convolution_gb300 import capi
    from dense_convolution_gb300.conv import Conv2d
    xd, wd = to_device(X, dtype), to_device(W, dtype)
    if layout == "nhwc":
        xd = xd.permute(0, 2, 3, 1).contiguous()
    N, Ci, H, Wd = X.shape
    Co, _, Kh, Kw = W.shape
    op = Conv2d(N, Ci, H, Wd, Co, Kh, Kw, s, p, dtype, algo, layout, tuning=tuning)
    y = op.alloc_output()
    if poison:
        y.fill_(float("nan"))
    g = 4096 if guard else 0
    ws = torch.empty(op.workspace_bytes + g, dtype=torch.uint8, device="cuda")
    if g:
        ws[op.workspace_bytes:].fill_(0xA5)
    op(xd, wd, y, ws[:max(op.workspace_bytes, 1)] if op.workspace_bytes else None)
    torch.cuda.synchronize()
    assert capi.conv2d_device_status(0) == 0
    if g:
        assert bool((ws[op.workspace_bytes:] == 0xA5).all()), "workspace guard overwritten"
    return y.double().cpu().numpy(), op.algo, op.workspace_bytes


def parity(y, Y, S):
    from oracle import ref
    return ref.parity_error(y, Y, S)
