"""Seeded synthetic gradients and the workload definitions.

This module is the only thing the oracle side and the CUDA side share: it makes
inputs.  It holds none of the all-reduce's arithmetic.

Generator (counter based, so any element can be drawn on its own):
  * ``mix`` is the SplitMix64 output function (Steele, Lea & Flood, "Fast
    splittable pseudorandom number generators", OOPSLA 2014); output n >= 1 of
    SplitMix64 seeded with s is ``mix(s + n * GAMMA)`` (mod 2^64).
  * ``key(seed, rank)``   = output ``rank + 1`` of SplitMix64 seeded with ``seed``.
  * ``word(seed, rank, n)`` = output ``n + 1`` of SplitMix64 seeded with ``key``.
  * Element i of a rank uses words 3i, 3i+1, 3i+2.
  * "normal": the twelve 16-bit lanes k_j of those words give the classic
    sum-of-twelve-uniforms approximation of N(0, 1):
    z = sum_j (k_j + 1/2) / 2^16 - 6 = (sum_j k_j - 393210) / 2^16 (exact in
    binary64), bounded to |z| <= 6.  The value is fl64(z * sigma), rounded to
    binary32, then (fp16 workloads) rounded to binary16.
  * "int1000": integer uniform in [-1000, 1000]: (word(3i) >> 11) mod 2001 - 1000.
Only integer operations and single IEEE roundings are used, so the host (numpy)
and device (``fill.cu``) versions produce identical bits; a test checks that.

Workloads: the five all-reduce problems of the web pages' models (ResNet-50 and
ResNet-101 gradients from "索尼发布新的方法...224秒内成功训练了ResNet-50" and
"[论文解读] PowerAI DDL"; the 300M-parameter language model's 1.2 GB gradient
from the Baidu ring-allreduce write-up's opening example).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def key(seed: int, rank: int) -> np.uint64:
    with np.errstate(over="ignore"):
        return _mix(np.array([seed], dtype=np.uint64) + np.uint64(rank + 1) * GAMMA)[0]


def words(seed: int, rank: int, n: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        n = np.asarray(n, dtype=np.uint64)
        return _mix(key(seed, rank) + (n + np.uint64(1)) * GAMMA)


def draw(seed: int, rank: int, idx, dist: str, sigma: float = 1.0, dtype: str = "f32") -> np.ndarray:
    """Values of ``rank`` at element indices ``idx``: float32 array, or uint16
    binary16 bit patterns for dtype 'f16'."""
    idx = np.asarray(idx, dtype=np.uint64)
    three = np.uint64(3)
    if dist == "int1000":
        w = words(seed, rank, idx * three)
        v = ((w >> np.uint64(11)) % np.uint64(2001)).astype(np.int64) - 1000
        x = v.astype(np.float32)
    elif dist == "normal":
        s = np.zeros(idx.shape, dtype=np.int64)
        for q in range(3):
            w = words(seed, rank, idx * three + np.uint64(q))
            for lane in range(4):
                s += ((w >> np.uint64(16 * lane)) & np.uint64(0xFFFF)).astype(np.int64)
        z = (s - 393210).astype(np.float64) / 65536.0
        x = (z * np.float64(sigma)).astype(np.float32)
    else:
        raise ValueError(dist)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    return x


def draw_rank(seed: int, rank: int, N: int, dist: str, sigma: float = 1.0, dtype: str = "f32",
              start: int = 0) -> np.ndarray:
    return draw(seed, rank, np.arange(start, start + N, dtype=np.uint64), dist, sigma, dtype)


# --------------------------------------------------------------------------
# ResNet parameter tensors in forward order, from the architecture rule
# (He et al. 2016, bottleneck ResNets as in torchvision): stem 7x7 conv + BN;
# four stages of bottleneck blocks (1x1 reduce, 3x3, 1x1 expand x4, each with
# BN weight and bias); a 1x1 projection conv + BN on each stage's first block;
# fc 2048 -> 1000 with bias.
# --------------------------------------------------------------------------

def resnet_param_sizes(blocks=(3, 4, 6, 3), num_classes: int = 1000):
    sizes = [64 * 3 * 7 * 7, 64, 64]
    cin = 64
    for stage, nb in enumerate(blocks):
        width = 64 * (2 ** stage)
        cout = width * 4
        for b in range(nb):
            sizes += [width * cin, width, width]
            sizes += [width * width * 9, width, width]
            sizes += [cout * width, cout, cout]
            if b == 0:
                sizes += [cout * cin, cout, cout]
            cin = cout
    sizes += [num_classes * cin, num_classes]
    return sizes


RESNET50 = resnet_param_sizes((3, 4, 6, 3))
RESNET101 = resnet_param_sizes((3, 4, 23, 3))


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    P: int
    N: int
    dtype: str            # "f32" or "f16"
    topo: str             # "ring" | "multiring" | "torus" | "torus_nd"
    k: int = 1
    X: int = 0
    Y: int = 0
    bucket_bytes: int = 0
    layers: tuple | None = None
    dims: tuple | None = None   # n-D torus sizes (topo "torus_nd")
    scale: float = 1.0
    dist: str = "normal"
    sigma: float = 1.0
    seed: int = 0

    @property
    def esize(self) -> int:
        return 2 if self.dtype == "f16" else 4

    @property
    def min_bytes(self) -> int:
        """Read every rank element once and write it once."""
        return 2 * self.P * self.N * self.esize

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def rank_values(self, rank: int, idx=None) -> np.ndarray:
        if idx is None:
            idx = np.arange(self.N, dtype=np.uint64)
        return draw(self.seed, rank, idx, self.dist, self.sigma, self.dtype)


_SEED0 = 20171
WORKLOADS = {
    # ring, P=4, 65,536 fp32 integers in [-1000, 1000], scale 1
    "ring4_int": Workload("ring4_int", P=4, N=65536, dtype="f32", topo="ring", scale=1.0,
                          dist="int1000", seed=_SEED0 + 1),
    # 4x4 torus, ResNet-50 gradient (25,557,032 fp32), N(0, 1e-3), scale 1/16
    "torus4x4_resnet50": Workload("torus4x4_resnet50", P=16, N=sum(RESNET50), dtype="f32", topo="torus",
                                  X=4, Y=4, scale=1.0 / 16, sigma=1e-3, seed=_SEED0 + 2),
    # 8x4 torus, fp16 hops, ResNet-50 layout (161 tensors), N(0, 1e-2), scale 1/32
    "torus8x4_resnet50_f16": Workload("torus8x4_resnet50_f16", P=32, N=sum(RESNET50), dtype="f16",
                                      topo="torus", X=8, Y=4, layers=tuple(RESNET50), scale=1.0 / 32,
                                      sigma=1e-2, seed=_SEED0 + 3),
    # multi-ring P=64, k=4, ResNet-101 gradient (44,549,160 fp32), 25 MiB
    # reverse-layer buckets, N(0, 1e-3), scale 1/64
    "multiring64_resnet101": Workload("multiring64_resnet101", P=64, N=sum(RESNET101), dtype="f32",
                                      topo="multiring", k=4, bucket_bytes=25 * 2 ** 20,
                                      layers=tuple(RESNET101), scale=1.0 / 64, sigma=1e-3,
                                      seed=_SEED0 + 4),
    # n-D torus 4x4x4 (P=64) on the ResNet-101 gradient in 25 MiB buckets
    "torus4x4x4_resnet101": Workload("torus4x4x4_resnet101", P=64, N=sum(RESNET101), dtype="f32",
                                     topo="torus_nd", dims=(4, 4, 4), bucket_bytes=25 * 2 ** 20,
                                     layers=tuple(RESNET101), scale=1.0 / 64, sigma=1e-3, seed=_SEED0 + 6),
    # n-D torus 4x4x2 (P=32) with fp16 hops on the ResNet-50 layout: the 8x4
    # fp16 torus's bytes on three dimensions
    "torus4x4x2_resnet50_f16": Workload("torus4x4x2_resnet50_f16", P=32, N=sum(RESNET50), dtype="f16",
                                        topo="torus_nd", dims=(4, 4, 2), layers=tuple(RESNET50),
                                        scale=1.0 / 32, sigma=1e-2, seed=_SEED0 + 7),
    # P=16, 300M fp32 (1.2 GB per rank, the language model's gradient), N(0, 1e-4)
    "ring16_lm300m": Workload("ring16_lm300m", P=16, N=300_000_000, dtype="f32", topo="ring",
                              scale=1.0 / 16, sigma=1e-4, seed=_SEED0 + 5),
    "multiring16_lm300m": Workload("multiring16_lm300m", P=16, N=300_000_000, dtype="f32",
                                   topo="multiring", k=2, scale=1.0 / 16, sigma=1e-4, seed=_SEED0 + 5),
    "torus4x4_lm300m": Workload("torus4x4_lm300m", P=16, N=300_000_000, dtype="f32", topo="torus",
                                X=4, Y=4, scale=1.0 / 16, sigma=1e-4, seed=_SEED0 + 5),
}


# --------------------------------------------------------------------------
# Device fill (fill.cu -> libsynth.so)
# --------------------------------------------------------------------------

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fill.cu")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
             "-Xcompiler", "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB):
                raise ImportError("libsynth.so is not built: run __graft_entry__.build()")
            lib = ctypes.CDLL(_LIB)
            lib.synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                       ctypes.c_void_p]
            lib.synth_fill.restype = ctypes.c_int
            _lib = lib
    return _lib


def fill_device(ptr: int, n: int, seed: int, rank: int, dist: str, sigma: float, dtype: str,
                stream: int = 0, start: int = 0) -> None:
    """Write elements [start, start+n) of ``rank``'s values to device memory."""
    rc = _load().synth_fill(ptr, n, start, seed, rank, {"int1000": 0, "normal": 1}[dist], sigma,
                            {"f32": 0, "f16": 1}[dtype], stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill failed with CUDA error {rc}")
