"""Seeded synthetic inputs and the workload table.

This module is shared by the tests, the smoke check and the benchmark.  It
holds no convolution arithmetic: it only draws numbers and rounds them to the
storage dtype, so the CUDA path and the oracle see identical bits.

Generator: counter-based splitmix64 (Steele, Lea, Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) gives 64 random bits per
element; the top 53 bits make a uniform double in [0,1); normals come from the
Box-Muller transform.  Element i of stream t under seed k is a pure function
of (k, t, i), so any sub-range can be regenerated.

Dtype rounding: values are drawn in float64, rounded once to float32, then,
for 16-bit runs, rounded float32 -> float16 / bfloat16 with round-to-nearest-
even (numpy's float16 cast, torch's bfloat16 cast).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _bits(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    key = _mix(np.array([(seed * 0x100000001B3 + stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + i * _G)


def uniform01(seed: int, stream: int, count: int) -> np.ndarray:
    """Uniform doubles in [0, 1)."""
    return (_bits(seed, stream, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform(seed, stream, shape, lo, hi) -> np.ndarray:
    n = int(np.prod(shape))
    return (lo + (hi - lo) * uniform01(seed, stream, n)).reshape(shape)


def normal(seed, stream, shape, std=1.0) -> np.ndarray:
    n = int(np.prod(shape))
    m = (n + 1) // 2
    u = uniform01(seed, stream, 2 * m)
    u1 = 1.0 - u[0::2]          # (0, 1]: log is finite
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m)
    z[0::2] = r * np.cos(2.0 * math.pi * u2)
    z[1::2] = r * np.sin(2.0 * math.pi * u2)
    return (std * z[:n]).reshape(shape)


def small_ints(seed, stream, shape, lo=-3, hi=3) -> np.ndarray:
    """Integers in [lo, hi]: every product and partial sum of a convolution on
    such values is an exact small integer in fp32 and fits fp16/bf16 inputs."""
    n = int(np.prod(shape))
    span = hi - lo + 1
    v = (_bits(seed, stream, n) % np.uint64(span)).astype(np.int64) + lo
    return v.astype(np.float64).reshape(shape)


DTYPES = ("f32", "f16", "bf16")


def round_to(values64: np.ndarray, dtype: str):
    """Round float64 values to the storage dtype.

    Returns (storage, exact64): ``storage`` is a numpy float32/float16 array or
    a torch bfloat16 tensor; ``exact64`` holds the same values widened to
    float64 (what the oracle reads)."""
    v32 = np.ascontiguousarray(values64, dtype=np.float32)
    if dtype == "f32":
        return v32, v32.astype(np.float64)
    if dtype == "f16":
        v16 = v32.astype(np.float16)
        return v16, v16.astype(np.float64)
    if dtype == "bf16":
        import torch
        t = torch.from_numpy(v32).to(torch.bfloat16)
        return t, t.to(torch.float64).numpy()
    raise ValueError(dtype)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    Ci: int
    H: int
    W: int
    Co: int
    Kh: int
    Kw: int
    stride: int
    pad: int
    dtypes: tuple
    x_dist: str          # "u-1_1", "u0_1", "n"
    w_dist: str          # "u-1_1", "kaiming", "n_sweep"
    seed: int

    def out_hw(self):
        ho = (self.H + 2 * self.pad - self.Kh) // self.stride + 1
        wo = (self.W + 2 * self.pad - self.Kw) // self.stride + 1
        return ho, wo

    def flops(self) -> int:
        ho, wo = self.out_hw()
        return 2 * self.N * self.Co * ho * wo * self.Ci * self.Kh * self.Kw

    def scaled(self, N=None, name=None) -> "Workload":
        return dataclasses.replace(self, N=N if N is not None else self.N,
                                   name=name or self.name)


def _sweep(K, stride=1):
    seed = 1004 * 100 + K + (50 if stride == 2 else 0)
    nm = f"sweep_k{K}" + ("_s2" if stride == 2 else "")
    return Workload(nm, 16, 128, 64, 64, 128, K, K, stride, K // 2 if stride == 1 else 1,
                    ("f32", "f16"), "n", "n_sweep", seed)


# The five benchmark layers: shapes, dtypes and value distributions.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 16, 32, 32, 16, 3, 3, 1, 1, ("f32",), "u-1_1", "u-1_1", 1000),
    "resnet_stage1": Workload("resnet_stage1", 32, 64, 56, 56, 64, 3, 3, 1, 1,
                              ("f16", "f32"), "n", "kaiming", 1001),
    "stem": Workload("stem", 32, 3, 224, 224, 64, 7, 7, 2, 3, ("f16", "f32"), "u0_1", "kaiming", 1002),
    "vgg": Workload("vgg", 64, 512, 28, 28, 512, 3, 3, 1, 1, ("bf16", "f16"), "n", "kaiming", 1003),
}
for _k in (1, 3, 5, 7, 9, 11):
    WORKLOADS[f"sweep_k{_k}"] = _sweep(_k)
WORKLOADS["sweep_k3_s2"] = _sweep(3, 2)

# The twelve layers of "Enabling Memory-efficient Im2win Convolution ...",
# Table I (input Ci x Hi x Wi, filter Co x Hf x Wf with stride, no padding:
# the table's output sizes are those of p = 0), at the batch of its Sec. IV-C
# (Ni = 256).  The paper gives no value distributions: N(0, 1) inputs and
# Kaiming-normal filters, as for the other layers.
_CV = [  # Ci, H, W, Co, K, s
    (3, 227, 227, 96, 11, 4), (3, 231, 231, 96, 11, 4), (3, 227, 227, 64, 7, 2), (64, 224, 224, 64, 7, 2),
    (96, 24, 24, 256, 5, 1), (256, 12, 12, 512, 3, 1), (3, 224, 224, 64, 3, 1), (64, 112, 112, 128, 3, 1),
    (64, 56, 56, 64, 3, 1), (128, 28, 28, 128, 3, 1), (256, 14, 14, 256, 3, 1), (512, 7, 7, 512, 3, 1),
]
for _i, (_ci, _h, _w, _co, _k, _s) in enumerate(_CV, start=1):
    WORKLOADS[f"cv{_i}"] = Workload(f"cv{_i}", 256, _ci, _h, _w, _co, _k, _k, _s, 0, ("f32", "f16"), "n", "kaiming",
                                    1100 + _i)


def make_inputs(wl: Workload, dtype: str, N: int | None = None):
    """Draw X and W for a workload.  ``N`` may shrink the batch (the first N
    samples of the full batch are identical to the full draw's).

    Returns dict with X, W (storage arrays/tensors) and X64, W64 (float64)."""
    n = wl.N if N is None else N
    xs = (n, wl.Ci, wl.H, wl.W)
    ws = (wl.Co, wl.Ci, wl.Kh, wl.Kw)
    if wl.x_dist == "u-1_1":
        x = uniform(wl.seed, 0, xs, -1.0, 1.0)
    elif wl.x_dist == "u0_1":
        x = uniform(wl.seed, 0, xs, 0.0, 1.0)
    else:
        x = normal(wl.seed, 0, xs)
    fan_in = wl.Ci * wl.Kh * wl.Kw
    if wl.w_dist == "u-1_1":
        w = uniform(wl.seed, 1, ws, -1.0, 1.0)
    elif wl.w_dist == "kaiming":
        w = normal(wl.seed, 1, ws, math.sqrt(2.0 / fan_in))
    else:
        w = normal(wl.seed, 1, ws, math.sqrt(1.0 / fan_in))
    X, X64 = round_to(x, dtype)
    W, W64 = round_to(w, dtype)
    return {"X": X, "W": W, "X64": X64, "W64": W64}


def make_int_inputs(seed, N, Ci, H, W, Co, Kh, Kw, dtype, lo=-3, hi=3):
    """Small-integer X and W (exact in every dtype)."""
    X, X64 = round_to(small_ints(seed, 0, (N, Ci, H, W), lo, hi), dtype)
    Wt, W64 = round_to(small_ints(seed, 1, (Co, Ci, Kh, Kw), lo, hi), dtype)
    return {"X": X, "W": Wt, "X64": X64, "W64": W64}
