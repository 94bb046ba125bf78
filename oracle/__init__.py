"""The oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow, single-threaded CPU emulation (C++, ``oracle.cpp``) of the
gradient all-reduce schedules: ring, multi-ring and 2D-torus, each run
send-by-send and add-by-add, plus an independent per-element closed form.
Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.

Parity status per function:
  emulate       pinned (hand traces, exact integer sums, brute force, invariants)
  closed_form   pinned (equals emulate on non-associative inputs; hand traces)
  fold_order    pinned (hand traces of the ring and the 2x2 torus)
  buckets       pinned (hand-computed layer packing, closed form of fixed buckets)
  f32_to_f16    pinned (exhaustive against numpy's and the C compiler's binary16)
  ref64         pinned (integer inputs: exact sums)
  cost          pinned (closed forms; the 400 ms language-model example; a hand-worked
                P=4, k=2 multi-ring on one shared link and on a link per ring)
  sgd           pinned (exact dyadic arithmetic; torch.optim.SGD within one rounding)

Buffers are numpy arrays: float32 for fp32, uint16 bit patterns for fp16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

TOPO = {"ring": 0, "multiring": 1, "torus": 2, "torus_nd": 3}
DTYPE = {"f32": 0, "f16": 1}


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (plain g++, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c++17", "-fPIC",
             "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("P", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("N", ctypes.c_uint64),
        ("topo", ctypes.c_int32),
        ("k", ctypes.c_int32),
        ("X", ctypes.c_int32),
        ("Y", ctypes.c_int32),
        ("bucket_bytes", ctypes.c_uint64),
        ("n_layers", ctypes.c_int64),
        ("layers", ctypes.POINTER(ctypes.c_uint64)),
        ("ndims", ctypes.c_int32),
        ("dims", ctypes.c_int32 * 4),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            u64, i64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32
            cfgp = ctypes.POINTER(_Cfg)
            lib.oracle_emulate.argtypes = [cfgp, P, ctypes.c_float, i64, ctypes.POINTER(u64), ctypes.POINTER(u64)]
            lib.oracle_emulate.restype = ctypes.c_int
            lib.oracle_closed_form.argtypes = [cfgp, P, P, u64, ctypes.c_float, P]
            lib.oracle_closed_form.restype = ctypes.c_int
            lib.oracle_fold_order.argtypes = [cfgp, u64, P, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            lib.oracle_fold_order.restype = ctypes.c_int
            lib.oracle_buckets.argtypes = [cfgp, P, P, i64]
            lib.oracle_buckets.restype = i64
            lib.oracle_ring_strides.argtypes = [i32, i32, P]
            lib.oracle_ring_strides.restype = ctypes.c_int
            lib.oracle_ref64.argtypes = [i32, u64, i32, P, ctypes.c_double, P]
            lib.oracle_ref64.restype = None
            lib.oracle_cost.argtypes = [cfgp, ctypes.c_double, ctypes.c_double, ctypes.c_int32,
                                        ctypes.POINTER(ctypes.c_double)]
            lib.oracle_cost.restype = ctypes.c_int
            lib.oracle_sgd.argtypes = [cfgp, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                       ctypes.c_float]
            lib.oracle_sgd.restype = ctypes.c_int
            lib.oracle_f32_to_f16.argtypes = [P, P, u64]
            lib.oracle_f16_to_f32.argtypes = [P, P, u64]
            lib.oracle_f32_pattern_to_f16.argtypes = [u64, u64, P]
            _lib = lib
    return _lib


class OracleError(ValueError):
    pass


class Config:
    """One all-reduce problem: P rank buffers of N elements, a schedule and buckets."""

    def __init__(self, P: int, N: int, dtype: str = "f32", topo: str = "ring", k: int = 1,
                 X: int = 0, Y: int = 0, bucket_bytes: int = 0, layers=None, dims=None):
        self.P, self.N, self.dtype, self.topo = int(P), int(N), dtype, topo
        self.k, self.X, self.Y, self.bucket_bytes = int(k), int(X), int(Y), int(bucket_bytes)
        self._layers = None if layers is None else np.ascontiguousarray(layers, dtype=np.uint64)
        c = _Cfg()
        c.P, c.dtype, c.N, c.topo = self.P, DTYPE[dtype], self.N, TOPO[topo]
        c.k, c.X, c.Y, c.bucket_bytes = self.k, self.X, self.Y, self.bucket_bytes
        if self._layers is not None and len(self._layers):
            c.n_layers = len(self._layers)
            c.layers = self._layers.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64))
        else:
            c.n_layers = 0
        self.dims = None if dims is None else [int(d) for d in dims]
        if self.dims is not None:
            c.ndims = len(self.dims)
            for i, d in enumerate(self.dims[:4]):
                c.dims[i] = d
        self._c = c

    @property
    def np_dtype(self):
        return np.uint16 if self.dtype == "f16" else np.float32

    def _ref(self):
        return ctypes.byref(self._c)


def _ptrs(bufs):
    arr = (ctypes.c_void_p * len(bufs))(*[b.ctypes.data for b in bufs])
    return arr


def _check(rc):
    if rc < 0:
        raise OracleError(f"oracle rejected the configuration (code {rc})")
    return rc


def emulate(cfg: Config, bufs, scale: float, stop_after: int = -1):
    """Run the schedule in place on ``bufs`` (list of P contiguous arrays).
    Returns (elements moved in total over all messages, communication steps)."""
    lib = _load()
    if bufs is not None:
        assert len(bufs) == cfg.P
        for b in bufs:
            assert b.dtype == cfg.np_dtype and b.flags.c_contiguous and b.size == cfg.N
        p = _ptrs(bufs)
    else:
        p = None
    moved, steps = ctypes.c_uint64(), ctypes.c_uint64()
    _check(lib.oracle_emulate(cfg._ref(), p, ctypes.c_float(scale), stop_after,
                              ctypes.byref(moved), ctypes.byref(steps)))
    return moved.value, steps.value


def traffic(cfg: Config):
    """Elements moved and steps, counted by the emulation without data."""
    return emulate(cfg, None, 1.0)


def cost(cfg: Config, alpha: float, beta: float, links: int = 1) -> float:
    """alpha-beta seconds of the schedule on P real workers with `links`
    network links each: per step alpha plus beta times the bytes of the
    busiest link (ring j of a step on link j mod links), steps in sequence."""
    lib = _load()
    t = ctypes.c_double()
    _check(lib.oracle_cost(cfg._ref(), alpha, beta, int(links), ctypes.byref(t)))
    return t.value


def sgd(cfg: Config, grads, params, moms, scale: float, lr: float, mu: float, wd: float) -> None:
    """All-reduce ``grads`` (step emulation), then momentum SGD on every
    rank's fp32 ``params`` and ``moms`` (None when mu == 0), all in place."""
    lib = _load()
    for a in list(params) + list(moms or []):
        assert a.dtype == np.float32 and a.flags.c_contiguous and a.size == cfg.N
    mp = _ptrs(moms) if moms is not None else None
    _check(lib.oracle_sgd(cfg._ref(), _ptrs(grads), _ptrs(params), mp, ctypes.c_float(scale),
                          ctypes.c_float(lr), ctypes.c_float(mu), ctypes.c_float(wd)))


def closed_form(cfg: Config, x_rows: np.ndarray, idx: np.ndarray, scale: float) -> np.ndarray:
    """x_rows[s, r] = rank r's stored value at element idx[s]; returns the
    stored result at each sampled element."""
    lib = _load()
    x_rows = np.ascontiguousarray(x_rows, dtype=cfg.np_dtype)
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    assert x_rows.shape == (idx.size, cfg.P)
    out = np.empty(idx.size, dtype=cfg.np_dtype)
    _check(lib.oracle_closed_form(cfg._ref(), x_rows.ctypes.data, idx.ctypes.data, idx.size,
                                  ctypes.c_float(scale), out.ctypes.data))
    return out


def closed_form_full(cfg: Config, bufs, scale: float) -> np.ndarray:
    """Closed form at every element of small buffers."""
    x = np.stack(bufs, axis=1)
    return closed_form(cfg, x, np.arange(cfg.N, dtype=np.uint64), scale)


def fold_order(cfg: Config, i: int):
    lib = _load()
    order = np.empty(cfg.P, dtype=np.int32)
    inner, groups = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.oracle_fold_order(cfg._ref(), i, order.ctypes.data, ctypes.byref(inner), ctypes.byref(groups)))
    return order, inner.value, groups.value


def buckets(cfg: Config):
    lib = _load()
    nb = _check(lib.oracle_buckets(cfg._ref(), None, None, 0))
    b = np.empty(nb, dtype=np.uint64)
    e = np.empty(nb, dtype=np.uint64)
    lib.oracle_buckets(cfg._ref(), b.ctypes.data, e.ctypes.data, nb)
    return list(zip(b.tolist(), e.tolist()))


def ring_strides(P: int, k: int):
    lib = _load()
    out = np.empty(k, dtype=np.int32)
    _check(lib.oracle_ring_strides(P, k, out.ctypes.data))
    return out.tolist()


def ref64(bufs, scale: float, dtype: str = "f32") -> np.ndarray:
    lib = _load()
    P, N = len(bufs), bufs[0].size
    out = np.empty(N, dtype=np.float64)
    lib.oracle_ref64(P, N, DTYPE[dtype], _ptrs(bufs), float(scale), out.ctypes.data)
    return out


def f32_to_f16(x: np.ndarray) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.size, dtype=np.uint16)
    lib.oracle_f32_to_f16(x.ctypes.data, out.ctypes.data, x.size)
    return out.reshape(x.shape)


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    lib = _load()
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.size, dtype=np.float32)
    lib.oracle_f16_to_f32(h.ctypes.data, out.ctypes.data, h.size)
    return out.reshape(h.shape)


def f32_patterns_to_f16(lo: int, hi: int) -> np.ndarray:
    lib = _load()
    out = np.empty(hi - lo, dtype=np.uint16)
    lib.oracle_f32_pattern_to_f16(lo, hi, out.ctypes.data)
    return out
