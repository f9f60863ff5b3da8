"""ctypes binding of ``include/conv2d.h`` — argument marshalling only.

Every function here has the name of the C entry point it wraps and raises
``Conv2dError`` on a non-OK status.  Pointers are plain integers (device
addresses, e.g. ``tensor.data_ptr()``); streams are integer handles (e.g.
``torch.cuda.current_stream().cuda_stream``).  Loading fails loudly when the
shared library has not been built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libconv2d_gb300.so")

OK, ERR_BAD_PARAM, ERR_UNSUPPORTED, ERR_NULL_PTR, ERR_MISALIGNED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, \
    ERR_DEVICE_TIMEOUT = range(8)
DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
ALGOS = {"auto": 0, "im2win_fp32_cc": 1, "im2win_tc": 2, "implicit_tc": 3, "implicit_fp32_cc": 4, "padded_tc": 5,
         "implicit_nchw_tc": 6, "winograd_fp32_cc": 7}
ALGO_NAMES = {v: k for k, v in ALGOS.items()}
LAYOUTS = {"nchw": 0, "nhwc": 1}
TUNING = {"stages": 0, "sync_copies": 1, "raster": 2, "no_resident": 3, "split": 4, "epi_groups": 5, "tile_n": 6}

EXPORTED = ("conv2d_desc_create", "conv2d_desc_set_input_layout", "conv2d_desc_set_output_dtype",
            "conv2d_desc_set_bias", "conv2d_desc_set_tuning", "conv2d_packed_filter_bytes", "conv2d_pack_filter",
            "conv2d_desc_set_filter_prepacked", "conv2d_desc_destroy", "conv2d_out_dims",
            "conv2d_workspace_size", "conv2d_get_algo", "conv2d_fwd", "conv2d_fwd_profiled", "conv2d_fwd_host",
            "conv2d_launches_per_call", "conv2d_fwd_static_workspace", "conv2d_static_workspace_bytes",
            "conv2d_set_wait_limit", "conv2d_device_status", "conv2d_status_string")


class Conv2dError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {conv2d_status_string(status)} (status {status})")


_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    L = ctypes.CDLL(path)
    c_int, c_size, vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    L.conv2d_desc_create.argtypes = [ctypes.POINTER(vp)] + [c_int] * 11
    L.conv2d_desc_set_input_layout.argtypes = [vp, c_int]
    L.conv2d_desc_set_output_dtype.argtypes = [vp, c_int]
    L.conv2d_desc_set_bias.argtypes = [vp, vp]
    L.conv2d_desc_set_tuning.argtypes = [vp, c_int, c_int]
    L.conv2d_packed_filter_bytes.argtypes = [vp, ctypes.POINTER(c_size)]
    L.conv2d_pack_filter.argtypes = [vp, vp, vp, vp]
    L.conv2d_desc_set_filter_prepacked.argtypes = [vp, c_int]
    L.conv2d_desc_destroy.argtypes = [vp]
    L.conv2d_out_dims.argtypes = [vp, ctypes.POINTER(c_int), ctypes.POINTER(c_int)]
    L.conv2d_workspace_size.argtypes = [vp, ctypes.POINTER(c_size)]
    L.conv2d_get_algo.argtypes = [vp, ctypes.POINTER(c_int)]
    L.conv2d_fwd.argtypes = [vp, vp, vp, vp, vp, c_size, vp]
    L.conv2d_fwd_profiled.argtypes = [vp, vp, vp, vp, vp, c_size, vp, vp, vp]
    L.conv2d_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, c_size, vp]
    L.conv2d_launches_per_call.argtypes = [vp, ctypes.POINTER(c_int)]
    L.conv2d_fwd_static_workspace.argtypes = [vp, vp, vp, vp, vp]
    L.conv2d_static_workspace_bytes.argtypes = [ctypes.POINTER(c_size)]
    L.conv2d_set_wait_limit.argtypes = [ctypes.c_uint64, vp]
    L.conv2d_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.conv2d_status_string.argtypes = [c_int]
    L.conv2d_status_string.restype = ctypes.c_char_p
    for f in EXPORTED[:-1]:
        getattr(L, f).restype = c_int
    _lib = L
    return L


def _check(status: int, where: str):
    if status != OK:
        raise Conv2dError(status, where)


def conv2d_status_string(status: int) -> str:
    return load().conv2d_status_string(int(status)).decode()


def conv2d_desc_create(N, Cin, H, W, Cout, Kh, Kw, stride, pad, dtype="f32", algo="auto") -> int:
    d = ctypes.c_void_p()
    dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    al = ALGOS[algo] if isinstance(algo, str) else int(algo)
    _check(load().conv2d_desc_create(ctypes.byref(d), N, Cin, H, W, Cout, Kh, Kw, stride, pad, dt, al),
           "conv2d_desc_create")
    return d.value


def conv2d_desc_set_input_layout(desc: int, layout="nchw"):
    lo = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    _check(load().conv2d_desc_set_input_layout(desc, lo), "conv2d_desc_set_input_layout")


def conv2d_desc_set_output_dtype(desc: int, out="f32"):
    dt = DTYPES[out] if isinstance(out, str) else int(out)
    _check(load().conv2d_desc_set_output_dtype(desc, dt), "conv2d_desc_set_output_dtype")


def conv2d_desc_set_bias(desc: int, bias: int):
    """Device address of Cout bias values of the input dtype (0 = no bias)."""
    _check(load().conv2d_desc_set_bias(desc, bias or None), "conv2d_desc_set_bias")


def conv2d_desc_set_tuning(desc: int, knob, value: int):
    """Pipeline knob for ablations: "stages", "sync_copies", "raster", "no_resident", "split"."""
    k = TUNING[knob] if isinstance(knob, str) else int(knob)
    _check(load().conv2d_desc_set_tuning(desc, k, int(value)), "conv2d_desc_set_tuning")


def conv2d_packed_filter_bytes(desc: int) -> int:
    b = ctypes.c_size_t()
    _check(load().conv2d_packed_filter_bytes(desc, ctypes.byref(b)), "conv2d_packed_filter_bytes")
    return b.value


def conv2d_pack_filter(desc: int, w: int, w_packed: int, stream: int = 0):
    _check(load().conv2d_pack_filter(desc, w, w_packed, stream or None), "conv2d_pack_filter")


def conv2d_desc_set_filter_prepacked(desc: int, prepacked: bool = True):
    _check(load().conv2d_desc_set_filter_prepacked(desc, 1 if prepacked else 0), "conv2d_desc_set_filter_prepacked")


def conv2d_desc_destroy(desc: int):
    _check(load().conv2d_desc_destroy(desc), "conv2d_desc_destroy")


def conv2d_out_dims(desc: int):
    ho, wo = ctypes.c_int(), ctypes.c_int()
    _check(load().conv2d_out_dims(desc, ctypes.byref(ho), ctypes.byref(wo)), "conv2d_out_dims")
    return ho.value, wo.value


def conv2d_workspace_size(desc: int) -> int:
    b = ctypes.c_size_t()
    _check(load().conv2d_workspace_size(desc, ctypes.byref(b)), "conv2d_workspace_size")
    return b.value


def conv2d_get_algo(desc: int) -> str:
    a = ctypes.c_int()
    _check(load().conv2d_get_algo(desc, ctypes.byref(a)), "conv2d_get_algo")
    return ALGO_NAMES[a.value]


def conv2d_fwd(desc: int, x: int, w: int, y: int, workspace: int, workspace_bytes: int, stream: int = 0):
    _check(load().conv2d_fwd(desc, x, w, y, workspace or None, workspace_bytes, stream or None), "conv2d_fwd")


def conv2d_fwd_profiled(desc: int, x: int, w: int, y: int, workspace: int, workspace_bytes: int, stream: int,
                        ev_start: int, ev_end: int):
    _check(load().conv2d_fwd_profiled(desc, x, w, y, workspace or None, workspace_bytes, stream or None,
                                      ev_start or None, ev_end or None), "conv2d_fwd_profiled")


def conv2d_fwd_host(desc: int, x_host: int, w_host: int, y_host: int, x_dev: int, w_dev: int, y_dev: int,
                    workspace: int, workspace_bytes: int, stream: int = 0):
    """conv2d_fwd on host operands: copy in, call, copy out, all on `stream`."""
    _check(load().conv2d_fwd_host(desc, x_host, w_host, y_host, x_dev, w_dev, y_dev, workspace or None,
                                  workspace_bytes, stream or None), "conv2d_fwd_host")


def conv2d_launches_per_call(desc: int) -> int:
    n = ctypes.c_int()
    _check(load().conv2d_launches_per_call(desc, ctypes.byref(n)), "conv2d_launches_per_call")
    return n.value


def conv2d_fwd_static_workspace(desc: int, x: int, w: int, y: int, stream: int = 0):
    """conv2d_fwd without a workspace argument, for callers that cannot
    allocate device memory: scratch comes from the library's built-in
    device array of conv2d_static_workspace_bytes() bytes (shared by all
    calls; overlapping calls race)."""
    _check(load().conv2d_fwd_static_workspace(desc, x, w, y, stream or None), "conv2d_fwd_static_workspace")


def conv2d_static_workspace_bytes() -> int:
    b = ctypes.c_size_t()
    _check(load().conv2d_static_workspace_bytes(ctypes.byref(b)), "conv2d_static_workspace_bytes")
    return b.value


def __getattr__(name):
    # STATIC_WORKSPACE_BYTES is read from the library, so it cannot drift from the C side.
    if name == "STATIC_WORKSPACE_BYTES":
        return conv2d_static_workspace_bytes()
    raise AttributeError(name)


def conv2d_set_wait_limit(ns: int, stream: int = 0):
    """Limit of each kernel pipeline wait in ns (0 = the default 2 s); tests only."""
    _check(load().conv2d_set_wait_limit(int(ns), stream or None), "conv2d_set_wait_limit")


def conv2d_device_status(stream: int = 0) -> int:
    code = ctypes.c_uint32()
    st = load().conv2d_device_status(stream or None, ctypes.byref(code))
    if st not in (OK, ERR_DEVICE_TIMEOUT):
        _check(st, "conv2d_device_status")
    return code.value
