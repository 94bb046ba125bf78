"""ctypes binding of libddl (include/ddl.h): the same entry points, same names.

Argument marshalling only: every step of the all-reduce runs in the library's
CUDA kernels.  There is no fallback -- if libddl.so is missing, importing this
module raises.  PyTorch is optional plumbing: ``Plan.allreduce`` accepts torch
CUDA tensors (their ``data_ptr`` and the current stream) as well as raw device
pointers.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# DDL_LIBRARY may name another build of the same library (e.g. one compiled
# with different kernel tuning macros); the default is the in-tree build.
LIB_PATH = os.environ.get("DDL_LIBRARY") or os.path.join(_HERE, "libddl.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run gradient_all_reduce_ddl_gb300.build.build() "
                      "(or __graft_entry__.build()) first")

_lib = ctypes.CDLL(LIB_PATH)

# ddl_status_t
DDL_OK, DDL_ERR_INVALID_ARG, DDL_ERR_UNSUPPORTED, DDL_ERR_OOM, DDL_ERR_CUDA, DDL_ERR_DEVICE_CHECK = range(6)
# ddl_dtype_t
DDL_FP32, DDL_FP16 = 0, 1
# ddl_topo_kind_t
DDL_RING, DDL_MULTIRING, DDL_TORUS = 0, 1, 2
# ddl_mode_t
DDL_MODE_FUSED, DDL_MODE_STEPWISE, DDL_MODE_RANKORDER = 0, 1, 2
# ddl_kernel_t
DDL_KERNEL_AUTO, DDL_KERNEL_LDG, DDL_KERNEL_BULK_LOAD, DDL_KERNEL_CHUNKED = 0, 1, 3, 5

EXPORTS = [
    "ddl_plan_create", "ddl_plan_set_layers", "ddl_plan_set_mode", "ddl_plan_set_kernel", "ddl_allreduce",
    "ddl_allreduce_bucket", "ddl_allreduce_host", "ddl_overlap_begin", "ddl_bucket_ready", "ddl_overlap_end",
    "ddl_plan_num_buckets", "ddl_plan_bucket_range", "ddl_plan_traffic", "ddl_plan_fold_order",
    "ddl_plan_launches", "ddl_plan_kernel_name", "ddl_plan_check", "ddl_status_string", "ddl_plan_destroy",
    "ddl_allreduce_noalloc", "ddl_plan_cost", "ddl_plan_set_torus_dims", "ddl_allreduce_sgd", "ddl_selftest_wait_timeout",
    "ddl_allreduce_slab", "ddl_noalloc_check",
]


class ddl_topology_t(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("k", ctypes.c_int32), ("X", ctypes.c_int32), ("Y", ctypes.c_int32)]


_vp, _i, _sz, _u64, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64, ctypes.c_float
_P = ctypes.POINTER


def _sig(name, res, *args):
    fn = getattr(_lib, name)
    fn.restype = res
    fn.argtypes = list(args)
    return fn


_sig("ddl_plan_create", _i, _i, _sz, _i, ddl_topology_t, _sz, _P(_vp))
_sig("ddl_plan_set_layers", _i, _vp, _i, _P(_sz))
_sig("ddl_plan_set_mode", _i, _vp, _i)
_sig("ddl_plan_set_torus_dims", _i, _vp, _i, _P(_i))
_sig("ddl_plan_set_kernel", _i, _vp, _i)
_sig("ddl_allreduce", _i, _vp, _P(_vp), _f, _vp)
_sig("ddl_allreduce_bucket", _i, _vp, _i, _P(_vp), _f, _vp)
_sig("ddl_allreduce_slab", _i, _vp, _vp, _sz, _f, _vp)
_sig("ddl_allreduce_sgd", _i, _vp, _P(_vp), _P(_vp), _P(_vp), _f, _f, _f, _f, _i, _vp)
_sig("ddl_allreduce_host", _i, _vp, _P(_vp), _P(_vp), _f, _vp)
_sig("ddl_overlap_begin", _i, _vp, _P(_vp), _f, _vp)
_sig("ddl_bucket_ready", _i, _vp, _i, _vp)
_sig("ddl_overlap_end", _i, _vp, _vp)
_sig("ddl_plan_num_buckets", _i, _vp, _P(_i))
_sig("ddl_plan_bucket_range", _i, _vp, _i, _P(_sz), _P(_sz))
_sig("ddl_plan_traffic", _i, _vp, _P(_u64), _P(_u64))
_sig("ddl_plan_cost", _i, _vp, ctypes.c_double, ctypes.c_double, _i, _P(ctypes.c_double))
_sig("ddl_plan_fold_order", _i, _vp, _sz, _P(ctypes.c_int32), _P(ctypes.c_int32), _P(ctypes.c_int32))
_sig("ddl_plan_launches", _i, _vp, _P(_u64))
_sig("ddl_plan_kernel_name", _i, _vp, _P(ctypes.c_char_p))
_sig("ddl_plan_check", _i, _vp)
_sig("ddl_selftest_wait_timeout", _i, _vp, ctypes.c_uint32, _vp)
_sig("ddl_status_string", ctypes.c_char_p, _i)
_sig("ddl_plan_destroy", _i, _vp)
_sig("ddl_allreduce_noalloc", _i, _i, _sz, _i, ddl_topology_t, _sz, _i, _P(_sz), _P(_vp), _f, _vp)
_sig("ddl_noalloc_check", _i, _vp)


class DDLError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {ddl_status_string(status)}")


def _ok(status: int, where: str) -> None:
    if status != DDL_OK:
        raise DDLError(status, where)


def ddl_status_string(status: int) -> str:
    return _lib.ddl_status_string(status).decode()


def _ptr_array(ptrs):
    return (ctypes.c_void_p * len(ptrs))(*[int(p) for p in ptrs])


def _dev_ptrs(bufs):
    return [b.data_ptr() if hasattr(b, "data_ptr") else int(b) for b in bufs]


def _stream_handle(stream):
    if stream is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:  # noqa: BLE001 - no torch / no GPU: the legacy default stream
            return 0
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# -- thin wrappers with the C names ------------------------------------------

def ddl_plan_create(P, N, dtype, topology, bucket_bytes=0):
    """topology: ddl_topology_t, or a dict(kind=..., k=..., X=..., Y=...)."""
    if isinstance(topology, dict):
        topology = ddl_topology_t(topology.get("kind", DDL_RING), topology.get("k", 1), topology.get("X", 0),
                                  topology.get("Y", 0))
    h = ctypes.c_void_p()
    _ok(_lib.ddl_plan_create(P, N, dtype, topology, bucket_bytes, ctypes.byref(h)), "ddl_plan_create")
    return h


def ddl_plan_set_layers(plan, numel_fwd_order):
    arr = (ctypes.c_size_t * len(numel_fwd_order))(*[int(v) for v in numel_fwd_order])
    _ok(_lib.ddl_plan_set_layers(plan, len(numel_fwd_order), arr), "ddl_plan_set_layers")


def ddl_plan_set_torus_dims(plan, dims):
    arr = (ctypes.c_int * len(dims))(*[int(d) for d in dims])
    _ok(_lib.ddl_plan_set_torus_dims(plan, len(dims), arr), "ddl_plan_set_torus_dims")


def ddl_plan_set_mode(plan, mode):
    _ok(_lib.ddl_plan_set_mode(plan, mode), "ddl_plan_set_mode")


def ddl_plan_set_kernel(plan, kernel):
    _ok(_lib.ddl_plan_set_kernel(plan, kernel), "ddl_plan_set_kernel")


def ddl_allreduce(plan, rank_bufs, scale, stream=None):
    _ok(_lib.ddl_allreduce(plan, _ptr_array(_dev_ptrs(rank_bufs)), scale, _stream_handle(stream)),
        "ddl_allreduce")


def ddl_allreduce_sgd(plan, grad_bufs, param_bufs, mom_bufs, scale, lr, momentum=0.0, weight_decay=0.0,
                      keep_grads=True, stream=None):
    moms = None if mom_bufs is None else _ptr_array(_dev_ptrs(mom_bufs))
    _ok(_lib.ddl_allreduce_sgd(plan, _ptr_array(_dev_ptrs(grad_bufs)), _ptr_array(_dev_ptrs(param_bufs)), moms,
                               scale, lr, momentum, weight_decay, 1 if keep_grads else 0, _stream_handle(stream)),
        "ddl_allreduce_sgd")


def ddl_allreduce_slab(plan, base, rank_stride_bytes, scale, stream=None):
    """base: device pointer (or tensor) of the slab; rank r at base + r * stride."""
    ptr = base.data_ptr() if hasattr(base, "data_ptr") else int(base)
    _ok(_lib.ddl_allreduce_slab(plan, ptr, rank_stride_bytes, scale, _stream_handle(stream)), "ddl_allreduce_slab")


def ddl_allreduce_bucket(plan, bucket, rank_bufs, scale, stream=None):
    _ok(_lib.ddl_allreduce_bucket(plan, bucket, _ptr_array(_dev_ptrs(rank_bufs)), scale,
                                  _stream_handle(stream)), "ddl_allreduce_bucket")


def ddl_allreduce_host(plan, host_bufs, dev_bufs, scale, stream=None):
    """dev_bufs None: the fused pass works on the host buffers in place."""
    dev = None if dev_bufs is None else _ptr_array(_dev_ptrs(dev_bufs))
    _ok(_lib.ddl_allreduce_host(plan, _ptr_array(_dev_ptrs(host_bufs)), dev, scale, _stream_handle(stream)),
        "ddl_allreduce_host")


def ddl_overlap_begin(plan, rank_bufs, scale, stream=None):
    _ok(_lib.ddl_overlap_begin(plan, _ptr_array(_dev_ptrs(rank_bufs)), scale, _stream_handle(stream)),
        "ddl_overlap_begin")


def ddl_bucket_ready(plan, bucket, stream=None):
    _ok(_lib.ddl_bucket_ready(plan, bucket, _stream_handle(stream)), "ddl_bucket_ready")


def ddl_overlap_end(plan, stream=None):
    _ok(_lib.ddl_overlap_end(plan, _stream_handle(stream)), "ddl_overlap_end")


def ddl_plan_num_buckets(plan):
    n = ctypes.c_int()
    _ok(_lib.ddl_plan_num_buckets(plan, ctypes.byref(n)), "ddl_plan_num_buckets")
    return n.value


def ddl_plan_bucket_range(plan, bucket):
    b, e = ctypes.c_size_t(), ctypes.c_size_t()
    _ok(_lib.ddl_plan_bucket_range(plan, bucket, ctypes.byref(b), ctypes.byref(e)), "ddl_plan_bucket_range")
    return b.value, e.value


def ddl_plan_traffic(plan):
    m, s = ctypes.c_uint64(), ctypes.c_uint64()
    _ok(_lib.ddl_plan_traffic(plan, ctypes.byref(m), ctypes.byref(s)), "ddl_plan_traffic")
    return m.value, s.value


def ddl_plan_cost(plan, alpha_s, beta_s_per_byte, links_per_worker=1):
    t = ctypes.c_double()
    _ok(_lib.ddl_plan_cost(plan, alpha_s, beta_s_per_byte, links_per_worker, ctypes.byref(t)), "ddl_plan_cost")
    return t.value


def ddl_plan_fold_order(plan, i, P):
    order = (ctypes.c_int32 * P)()
    inner, groups = ctypes.c_int32(), ctypes.c_int32()
    _ok(_lib.ddl_plan_fold_order(plan, i, order, ctypes.byref(inner), ctypes.byref(groups)), "ddl_plan_fold_order")
    return list(order), inner.value, groups.value


def ddl_plan_kernel_name(plan):
    """The kernel ddl_allreduce launches for the plan with 16-byte-aligned buffers."""
    name = ctypes.c_char_p()
    _ok(_lib.ddl_plan_kernel_name(plan, ctypes.byref(name)), "ddl_plan_kernel_name")
    return name.value.decode()


def ddl_plan_launches(plan):
    n = ctypes.c_uint64()
    _ok(_lib.ddl_plan_launches(plan, ctypes.byref(n)), "ddl_plan_launches")
    return n.value


def ddl_plan_check(plan):
    return _lib.ddl_plan_check(plan)


def ddl_selftest_wait_timeout(plan, limit_us, stream=None):
    _ok(_lib.ddl_selftest_wait_timeout(plan, limit_us, _stream_handle(stream)), "ddl_selftest_wait_timeout")


def ddl_plan_destroy(plan):
    _ok(_lib.ddl_plan_destroy(plan), "ddl_plan_destroy")


def ddl_allreduce_noalloc(P, N, dtype, topology, bucket_bytes, layers, rank_bufs, scale, stream=None):
    """Allocation-free all-reduce (no plan): tables in the library's static
    device array.  dtype: DDL_FP32/DDL_FP16; topology: ddl_topology_t or dict;
    layers: None or the tensor sizes in forward order."""
    if isinstance(topology, dict):
        topology = ddl_topology_t(topology.get("kind", DDL_RING), topology.get("k", 1), topology.get("X", 0),
                                  topology.get("Y", 0))
    layers = list(layers or [])
    arr = (ctypes.c_size_t * max(1, len(layers)))(*[int(v) for v in layers])
    _ok(_lib.ddl_allreduce_noalloc(P, N, dtype, topology, bucket_bytes, len(layers), arr,
                                   _ptr_array(_dev_ptrs(rank_bufs)), scale, _stream_handle(stream)),
        "ddl_allreduce_noalloc")


def ddl_noalloc_check(stream=None):
    """Status of the last allocation-free call's kernel on the current device
    (waits for `stream`); DDL_ERR_DEVICE_CHECK raises."""
    _ok(_lib.ddl_noalloc_check(_stream_handle(stream)), "ddl_noalloc_check")


# -- convenience object --------------------------------------------------------

# the per-call path of Plan.allreduce: the same entry point without argtypes,
# given ready-made ctypes arguments (no conversion on each call)
_ddl_allreduce = ctypes.CDLL(LIB_PATH).ddl_allreduce
_ddl_allreduce.restype = ctypes.c_int
_ddl_allreduce_sgd = ctypes.CDLL(LIB_PATH).ddl_allreduce_sgd
_ddl_allreduce_sgd.restype = ctypes.c_int
_NO_STREAM = object()  # no stream object seen yet (None means the current stream, looked up each call)

TOPOLOGIES = {"ring": DDL_RING, "multiring": DDL_MULTIRING, "torus": DDL_TORUS, "torus_nd": DDL_RING}
DTYPES = {"f32": DDL_FP32, "f16": DDL_FP16}
MODES = {"fused": DDL_MODE_FUSED, "stepwise": DDL_MODE_STEPWISE, "rankorder": DDL_MODE_RANKORDER}
KERNELS = {"auto": DDL_KERNEL_AUTO, "ldg": DDL_KERNEL_LDG, "bulkload": DDL_KERNEL_BULK_LOAD,
           "chunked": DDL_KERNEL_CHUNKED}


class Plan:
    """An all-reduce plan for P rank buffers of N elements (owns a ddl_plan_t)."""

    def __init__(self, P, N, dtype="f32", topo="ring", k=1, X=0, Y=0, bucket_bytes=0, layers=None,
                 mode="fused", kernel="auto", dims=None):
        self.P, self.N, self.dtype = int(P), int(N), dtype
        self._last_ptrs, self._last_arr = None, None
        self._last_stream, self._last_handle = _NO_STREAM, None
        self._sgd_key, self._sgd_arrs = None, None
        self._sgd_hyper, self._sgd_c = None, None
        self._scale, self._c_scale = None, None
        topo_t = ddl_topology_t(TOPOLOGIES[topo], int(k), int(X), int(Y))
        self.handle = ddl_plan_create(self.P, self.N, DTYPES[dtype], topo_t, int(bucket_bytes))
        self._c_handle = self.handle  # a ctypes.c_void_p
        try:
            if layers is not None:
                ddl_plan_set_layers(self.handle, list(layers))
            if topo == "torus_nd":
                ddl_plan_set_torus_dims(self.handle, list(dims))
            if mode != "fused":
                ddl_plan_set_mode(self.handle, MODES[mode])
            if kernel != "auto":
                ddl_plan_set_kernel(self.handle, KERNELS[kernel])
        except Exception:
            ddl_plan_destroy(self.handle)
            self.handle = None
            self._c_handle = ctypes.c_void_p(None)
            raise

    @classmethod
    def for_workload(cls, w, **kw):
        return cls(w.P, w.N, w.dtype, w.topo, k=w.k, X=w.X, Y=w.Y, bucket_bytes=w.bucket_bytes,
                   layers=w.layers, dims=getattr(w, "dims", None), **kw)

    def _stream_c(self, stream):
        # the stream handle, kept for the stream object last seen (None: the
        # current stream, looked up on every call)
        if stream is None or stream is not self._last_stream:
            self._last_stream, self._last_handle = stream, ctypes.c_void_p(_stream_handle(stream))
            if stream is None:
                self._last_stream = _NO_STREAM
        return self._last_handle

    def _rank_array(self, rank_bufs, stream):
        # the per-call path of small all-reduces: the ctypes pointer array is
        # rebuilt only when the buffers change
        try:
            ptrs = [b.data_ptr() for b in rank_bufs]
        except AttributeError:
            ptrs = _dev_ptrs(rank_bufs)
        if ptrs != self._last_ptrs:
            self._last_ptrs, self._last_arr = ptrs, _ptr_array(ptrs)
        return self._last_arr, self._stream_c(stream)

    def allreduce(self, rank_bufs, scale, stream=None):
        arr, handle = self._rank_array(rank_bufs, stream)
        if scale != self._scale:
            self._scale, self._c_scale = scale, ctypes.c_float(scale)
        status = _ddl_allreduce(self._c_handle, arr, self._c_scale, handle)
        if status:
            raise DDLError(status, "ddl_allreduce")

    def allreduce_sgd(self, grad_bufs, param_bufs, mom_bufs, scale, lr, momentum=0.0, weight_decay=0.0,
                      keep_grads=True, stream=None):
        # as in allreduce: the three pointer arrays are rebuilt only when a
        # buffer changes (the pointers are compared on every call)
        try:
            key = ([b.data_ptr() for b in grad_bufs], [b.data_ptr() for b in param_bufs],
                   None if mom_bufs is None else [b.data_ptr() for b in mom_bufs])
        except AttributeError:
            key = (_dev_ptrs(grad_bufs), _dev_ptrs(param_bufs), None if mom_bufs is None else _dev_ptrs(mom_bufs))
        if key != self._sgd_key:
            self._sgd_key = key
            self._sgd_arrs = (_ptr_array(key[0]), _ptr_array(key[1]), None if key[2] is None else _ptr_array(key[2]))
        g, pa, m = self._sgd_arrs
        hyper = (scale, lr, momentum, weight_decay, bool(keep_grads))
        if hyper != self._sgd_hyper:  # the scalars as ctypes values, rebuilt when one changes
            self._sgd_hyper = hyper
            self._sgd_c = tuple(ctypes.c_float(v) for v in hyper[:4]) + (ctypes.c_int(1 if keep_grads else 0),)
        status = _ddl_allreduce_sgd(self._c_handle, g, pa, m, *self._sgd_c, self._stream_c(stream))
        if status:
            raise DDLError(status, "ddl_allreduce_sgd")

    def allreduce_slab(self, base, rank_stride_bytes, scale, stream=None):
        ddl_allreduce_slab(self.handle, base, rank_stride_bytes, scale, stream)

    def allreduce_bucket(self, bucket, rank_bufs, scale, stream=None):
        arr, handle = self._rank_array(rank_bufs, stream)
        _ok(_lib.ddl_allreduce_bucket(self.handle, bucket, arr, scale, handle.value), "ddl_allreduce_bucket")

    def allreduce_host(self, host_bufs, dev_bufs, scale, stream=None):
        ddl_allreduce_host(self.handle, host_bufs, dev_bufs, scale, stream)

    def overlap_begin(self, rank_bufs, scale, stream=None):
        ddl_overlap_begin(self.handle, rank_bufs, scale, stream)

    def bucket_ready(self, bucket, stream=None):
        ddl_bucket_ready(self.handle, bucket, stream)

    def overlap_end(self, stream=None):
        ddl_overlap_end(self.handle, stream)

    def set_mode(self, mode):
        ddl_plan_set_mode(self.handle, MODES[mode])

    def set_kernel(self, kernel):
        ddl_plan_set_kernel(self.handle, KERNELS[kernel])

    @property
    def num_buckets(self):
        return ddl_plan_num_buckets(self.handle)

    def bucket_range(self, b):
        return ddl_plan_bucket_range(self.handle, b)

    def buckets(self):
        return [self.bucket_range(b) for b in range(self.num_buckets)]

    def traffic(self):
        return ddl_plan_traffic(self.handle)

    def fold_order(self, i):
        return ddl_plan_fold_order(self.handle, i, self.P)

    @property
    def kernel_name(self):
        """The kernel ddl_allreduce launches (16-byte-aligned buffers)."""
        return ddl_plan_kernel_name(self.handle)

    def cost(self, alpha_s, beta_s_per_byte, links=1):
        """alpha-beta model of this schedule on P real workers with `links`
        network links each (seconds)."""
        return ddl_plan_cost(self.handle, alpha_s, beta_s_per_byte, links)

    @property
    def launches(self):
        return ddl_plan_launches(self.handle)

    def check(self):
        _ok(ddl_plan_check(self.handle), "ddl_plan_check")

    def close(self):
        if self.handle is not None:
            ddl_plan_destroy(self.handle)
            self.handle = None
            self._c_handle = ctypes.c_void_p(None)  # a later call gets DDL_ERR_INVALID_ARG

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
