"""PyTorch-tensor convenience layer over the C ABI.

PyTorch provides device memory (output and workspace tensors) and the current
stream; every arithmetic step runs in the library's kernels.  Shapes are
checked here only so that a wrong tensor fails with a Python error instead of
a bad pointer.
"""
from __future__ import annotations

import torch

from . import capi

_TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
_NAME = {v: k for k, v in _TORCH_DTYPE.items()}


class Conv2d:
    """One problem shape: descriptor, output shape and workspace size."""

    def __init__(self, N, Cin, H, W, Cout, Kh, Kw, stride=1, pad=0, dtype="f32", algo="auto", layout="nchw",
                 out_dtype=None, tuning=None):
        self.shape = (N, Cin, H, W, Cout, Kh, Kw, stride, pad)
        self.dtype = dtype
        self.out_dtype = out_dtype or dtype
        self.layout = layout
        self.desc = capi.conv2d_desc_create(N, Cin, H, W, Cout, Kh, Kw, stride, pad, dtype, algo)
        if layout != "nchw":
            capi.conv2d_desc_set_input_layout(self.desc, layout)
        if self.out_dtype != dtype:
            capi.conv2d_desc_set_output_dtype(self.desc, self.out_dtype)
        for knob, value in (tuning or {}).items():
            capi.conv2d_desc_set_tuning(self.desc, knob, value)
        self.Ho, self.Wo = capi.conv2d_out_dims(self.desc)
        self.workspace_bytes = capi.conv2d_workspace_size(self.desc)
        self.algo = capi.conv2d_get_algo(self.desc)

    def pack_filter(self, w: torch.Tensor, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
        """The filter in the kernels' order (a byte tensor), for set_prepacked calls."""
        N, Ci, H, W, Co, Kh, Kw = self.shape[:7]
        if tuple(w.shape) != (Co, Ci, Kh, Kw) or not w.is_contiguous() or w.dtype != _TORCH_DTYPE[self.dtype]:
            raise ValueError(f"w must be a contiguous {self.dtype} tensor of shape {(Co, Ci, Kh, Kw)}")
        wp = torch.empty(capi.conv2d_packed_filter_bytes(self.desc), dtype=torch.uint8, device=w.device)
        st = (stream or torch.cuda.current_stream(w.device)).cuda_stream
        capi.conv2d_pack_filter(self.desc, w.data_ptr(), wp.data_ptr(), st)
        return wp

    def set_prepacked(self, on: bool = True):
        """From now on __call__ takes the output of pack_filter as w (no repack per call)."""
        capi.conv2d_desc_set_filter_prepacked(self.desc, on)
        self.prepacked = on
        self.workspace_bytes = capi.conv2d_workspace_size(self.desc)

    def __del__(self):
        d = getattr(self, "desc", None)
        if d:
            try:
                capi.conv2d_desc_destroy(d)
            except Exception:
                pass
            self.desc = None

    @property
    def out_shape(self):
        N, _, _, _, Co = self.shape[:5]
        return (N, Co, self.Ho, self.Wo)

    def alloc_workspace(self, device="cuda"):
        n = max(self.workspace_bytes, 1)
        return torch.empty(n, dtype=torch.uint8, device=device)

    def alloc_output(self, device="cuda"):
        return torch.empty(self.out_shape, dtype=_TORCH_DTYPE[self.out_dtype], device=device)

    def __call__(self, x: torch.Tensor, w: torch.Tensor, y: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None,
                 bias: torch.Tensor | None = None) -> torch.Tensor:
        N, Ci, H, W, Co, Kh, Kw = self.shape[:7]
        want_x = (N, Ci, H, W) if self.layout == "nchw" else (N, H, W, Ci)
        if tuple(x.shape) != want_x or not x.is_contiguous() or x.dtype != _TORCH_DTYPE[self.dtype]:
            raise ValueError(f"x must be a contiguous {self.dtype} tensor of shape {want_x}")
        if getattr(self, "prepacked", False):
            if w.dtype != torch.uint8 or w.numel() != capi.conv2d_packed_filter_bytes(self.desc):
                raise ValueError("w must be the byte tensor pack_filter returned for this descriptor")
        elif tuple(w.shape) != (Co, Ci, Kh, Kw) or not w.is_contiguous() or w.dtype != x.dtype:
            raise ValueError(f"w must be a contiguous {self.dtype} tensor of shape {(Co, Ci, Kh, Kw)}")
        if bias is not None and (tuple(bias.shape) != (Co,) or not bias.is_contiguous() or bias.dtype != x.dtype):
            raise ValueError(f"bias must be a contiguous {self.dtype} tensor of shape {(Co,)}")
        capi.conv2d_desc_set_bias(self.desc, bias.data_ptr() if bias is not None else 0)
        if y is None:
            y = self.alloc_output(x.device)
        if workspace is None and self.workspace_bytes:
            workspace = self.alloc_workspace(x.device)
        st = (stream or torch.cuda.current_stream(x.device)).cuda_stream
        capi.conv2d_fwd(self.desc, x.data_ptr(), w.data_ptr(), y.data_ptr(),
                        workspace.data_ptr() if workspace is not None else 0,
                        workspace.numel() if workspace is not None else 0, st)
        return y


def conv2d(x: torch.Tensor, w: torch.Tensor, stride: int = 1, pad: int = 0, algo: str = "auto") -> torch.Tensor:
    """Y = conv2d(X, W) for NCHW x and [Co][Ci][Kh][Kw] w on the current stream."""
    N, Ci, H, W = x.shape
    Co, _, Kh, Kw = w.shape
    op = Conv2d(N, Ci, H, W, Co, Kh, Kw, stride, pad, _NAME[x.dtype], algo)
    return op(x, w)
