"""The C-ABI library on the host: it loads, exports every declared symbol, and
its host-only calls (plan tables, traffic, errors) agree with the oracle.
No GPU work is done here."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ddl():
    from gradient_all_reduce_ddl_gb300.build import build
    build()
    from gradient_all_reduce_ddl_gb300 import ddl as mod
    return mod


def _declared():
    src = open(os.path.join(ROOT, "include", "ddl.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ddl_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(ddl):
    names = _declared()
    assert len(names) >= 18
    lib = ctypes.CDLL(ddl.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(ddl.EXPORTS) == names


def test_status_strings(ddl):
    for s in range(6):
        assert ddl.ddl_status_string(s).startswith("DDL_")
    assert "unknown" in ddl.ddl_status_string(99)


def _pair(P, N, dtype="f32", topo="ring", k=1, X=0, Y=0, bucket_bytes=0, layers=None, mode="fused", dims=None):
    from gradient_all_reduce_ddl_gb300 import ddl
    plan = ddl.Plan(P, N, dtype, topo, k=k, X=X, Y=Y, bucket_bytes=bucket_bytes, layers=layers, mode=mode,
                    dims=dims)
    cfg = oracle.Config(P, N, dtype, topo, k=k, X=X, Y=Y, bucket_bytes=bucket_bytes, layers=layers, dims=dims)
    return plan, cfg


CASES = [
    dict(P=1, N=5),
    dict(P=3, N=7),
    dict(P=5, N=103, bucket_bytes=64),
    dict(P=7, N=6),
    dict(P=16, N=1000, topo="multiring", k=2),
    dict(P=9, N=301, topo="multiring", k=5, bucket_bytes=400),
    dict(P=4, N=8, topo="torus", X=2, Y=2),
    dict(P=16, N=999, topo="torus", X=4, Y=4, bucket_bytes=1000),
    dict(P=12, N=500, topo="torus", X=3, Y=4),
    dict(P=6, N=50, topo="torus", X=6, Y=1, dtype="f16", bucket_bytes=30),
    dict(P=6, N=50, topo="torus", X=1, Y=6, layers=[10, 20, 15, 5], bucket_bytes=40),
    dict(P=8, N=77, topo="torus_nd", dims=[2, 2, 2]),
    dict(P=64, N=1001, topo="torus_nd", dims=[4, 4, 4], bucket_bytes=1200),
    dict(P=24, N=333, topo="torus_nd", dims=[2, 3, 2, 2], dtype="f16"),
    dict(P=12, N=120, topo="torus_nd", dims=[3, 1, 4, 1]),
]


@pytest.mark.parametrize("case", CASES)
def test_tables_match_oracle(ddl, case):
    """Buckets, traffic, steps and the fold order of every element, from the
    library's own tables, equal the oracle's."""
    plan, cfg = _pair(**case)
    with plan:
        assert plan.buckets() == oracle.buckets(cfg)
        assert plan.traffic() == oracle.traffic(cfg)
        for i in range(cfg.N):
            o_ord, o_in, o_gr = oracle.fold_order(cfg, i)
            l_ord, l_in, l_gr = plan.fold_order(i)
            assert (l_ord, l_in, l_gr) == (o_ord.tolist(), o_in, o_gr), i


@pytest.mark.parametrize("case", CASES)
def test_cost_model_matches_oracle(ddl, case):
    plan, cfg = _pair(**case)
    with plan:
        for a, b in [(0.0, 1e-9), (2e-6, 0.0), (3e-6, 1.6e-10)]:
            for links in (1, 2, 3, 8):
                assert plan.cost(a, b, links) == pytest.approx(oracle.cost(cfg, a, b, links), rel=1e-12,
                                                               abs=1e-18), links
        with pytest.raises(ddl.DDLError):
            plan.cost(-1.0, 0.0)
        with pytest.raises(ddl.DDLError):
            plan.cost(1.0, 0.0, 0)


@pytest.mark.parametrize("name", ["torus4x4_resnet50", "torus8x4_resnet50_f16", "multiring64_resnet101",
                                  "ring16_lm300m", "torus4x4_lm300m", "torus4x4x4_resnet101",
                                  "torus4x4x2_resnet50_f16"])
def test_workload_tables_match_oracle(ddl, name):
    w = synth.WORKLOADS[name]
    with ddl.Plan.for_workload(w) as plan:
        cfg = oracle.Config(w.P, w.N, w.dtype, w.topo, k=w.k, X=w.X, Y=w.Y, bucket_bytes=w.bucket_bytes,
                            layers=w.layers, dims=w.dims)
        assert plan.buckets() == oracle.buckets(cfg)
        moved, steps = plan.traffic()
        assert moved == 2 * (w.P - 1) * w.N
        assert (moved, steps) == oracle.traffic(cfg)
        rng = np.random.default_rng(0)
        for i in rng.integers(0, w.N, 300).tolist() + [0, w.N - 1]:
            o_ord, o_in, o_gr = oracle.fold_order(cfg, i)
            assert plan.fold_order(i) == (o_ord.tolist(), o_in, o_gr)


@pytest.mark.parametrize("case", [CASES[2], CASES[5], CASES[7], CASES[9]])
@pytest.mark.parametrize("kernel", ["bulkload", "chunked"])
def test_staged_kernel_tables_match_oracle(ddl, case, kernel):
    """Selecting a staged kernel rebuilds the work items at its tile size (the
    rank-chunked pass keeps the register pass's); the fold orders stay the
    oracle's."""
    plan, cfg = _pair(**case)
    with plan:
        plan.set_kernel(kernel)
        assert plan.buckets() == oracle.buckets(cfg)
        for i in range(cfg.N):
            o_ord, o_in, o_gr = oracle.fold_order(cfg, i)
            assert plan.fold_order(i) == (o_ord.tolist(), o_in, o_gr), i


def test_nd_torus_dims_validation(ddl):
    E = ddl.DDLError
    with ddl.Plan(8, 100) as p:
        for dims in ([3, 3], [0, 8], [2, 2, 2, 1, 1], []):
            with pytest.raises(E):
                ddl.ddl_plan_set_torus_dims(p.handle, dims)
        ddl.ddl_plan_set_torus_dims(p.handle, [2, 4, 1])     # trailing 1 dropped
        assert p.traffic() == oracle.traffic(oracle.Config(8, 100, topo="torus", X=2, Y=4))


def test_rankorder_and_stepwise_tables(ddl):
    plan, cfg = _pair(P=5, N=50, topo="torus", X=5, Y=1, mode="rankorder")
    with plan:
        assert plan.fold_order(13) == ([0, 1, 2, 3, 4], 5, 1)
        assert plan.traffic() == oracle.traffic(cfg)
    plan, cfg = _pair(P=5, N=50, mode="stepwise")
    with plan:
        with pytest.raises(ddl.DDLError):
            plan.fold_order(0)
        assert plan.traffic() == oracle.traffic(cfg)


def test_invalid_arguments(ddl):
    E = ddl.DDLError
    bad = [
        dict(P=0, N=10), dict(P=4, N=0), dict(P=6, N=10, topo="torus", X=4, Y=2),
        dict(P=4, N=10, topo="multiring", k=0), dict(P=4, N=10, layers=[3, 3]),
        dict(P=4, N=10, bucket_bytes=2), dict(P=4, N=10, layers=[5, 0, 5]),
    ]
    for c in bad:
        with pytest.raises(E) as ei:
            ddl.Plan(**c)
        assert ei.value.status == ddl.DDL_ERR_INVALID_ARG, c
    for c in [dict(P=257, N=10), dict(P=16, N=10, topo="multiring", k=9)]:
        with pytest.raises(E) as ei:
            ddl.Plan(**c)
        assert ei.value.status == ddl.DDL_ERR_UNSUPPORTED, c
    h = ctypes.c_void_p()
    assert ddl._lib.ddl_plan_create(4, 10, 7, ddl.ddl_topology_t(0, 1, 0, 0), 0, ctypes.byref(h)) == \
        ddl.DDL_ERR_INVALID_ARG
    assert ddl._lib.ddl_plan_create(4, 10, 0, ddl.ddl_topology_t(0, 1, 0, 0), 0, None) == ddl.DDL_ERR_INVALID_ARG
    # calls on a null plan
    assert ddl._lib.ddl_plan_set_mode(None, 0) == ddl.DDL_ERR_INVALID_ARG
    assert ddl._lib.ddl_allreduce(None, None, ctypes.c_float(1.0), None) == ddl.DDL_ERR_INVALID_ARG
    assert ddl._lib.ddl_plan_destroy(None) == ddl.DDL_OK
    with ddl.Plan(4, 100) as p:
        # null / duplicate / overlapping rank pointers are refused before any GPU call
        for ptrs in ([0, 4096, 8192, 12288], [4096, 4096, 8192, 12288], [4096, 4200, 8192, 12288]):
            arr = (ctypes.c_void_p * 4)(*ptrs)
            assert ddl._lib.ddl_allreduce(p.handle, arr, ctypes.c_float(1.0), None) == ddl.DDL_ERR_INVALID_ARG
        assert ddl._lib.ddl_allreduce(p.handle, None, ctypes.c_float(1.0), None) == ddl.DDL_ERR_INVALID_ARG
        with pytest.raises(E):
            p.allreduce_bucket(5, [4096 * (i + 1) for i in range(4)], 1.0, stream=0)
        with pytest.raises(E):
            p.bucket_ready(0, stream=0)      # no overlap_begin
        with pytest.raises(E):
            p.overlap_end(stream=0)
        with pytest.raises(E):
            ddl.ddl_plan_set_mode(p.handle, 7)
        with pytest.raises(E):
            ddl.ddl_plan_set_layers(p.handle, [50, 49])
        # a failed set_layers leaves the plan as it was
        assert p.buckets() == [(0, 100)]
        ddl.ddl_plan_set_layers(p.handle, [50, 50])
        assert p.launches == 0


def test_kernel_choice_range(ddl):
    """Every ddl_kernel_t value is accepted on a host-only plan; the unused
    values 2 and 4 (passes removed from the library), the next one and a
    negative one are refused."""
    with ddl.Plan(8, 10_000) as plan:
        for k in (0, 1, 3, 5):
            assert ddl._lib.ddl_plan_set_kernel(plan.handle, k) == ddl.DDL_OK, k
        for k in (2, 4, 6, -1):
            assert ddl._lib.ddl_plan_set_kernel(plan.handle, k) == ddl.DDL_ERR_INVALID_ARG, k


# (plan, the kernel ddl_allreduce launches): large buffers take the register
# pass; small items of P >= 16 ranks the latency pass (one-group instance for a
# single fold group, until its items exceed one wave of CTAs); small items of
# one unrounded group below that the small-item pass; the n-D torus its own
# passes; stepwise mode the step kernel; a staged choice its kernel.
DISPATCH = [
    (dict(P=16, N=3_000_000), "fold_ldg_kernel"),
    (dict(P=16, N=25_557_032, topo="torus", X=4, Y=4), "fold_ldg_kernel"),
    (dict(P=32, N=25_557_032, dtype="f16", topo="torus", X=8, Y=4), "fold_ldg_kernel"),
    (dict(P=4, N=65_536), "fold_small_kernel"),
    (dict(P=8, N=16_384, dtype="f16"), "fold_lat_kernel (one group)"),  # binary16 hops: the latency pass from P = 8
    (dict(P=8, N=16_384, dtype="f16", topo="torus", X=4, Y=2), "fold_lat_kernel"),
    (dict(P=4, N=65_536, dtype="f16"), "fold_ldg_kernel"),            # binary16 hops, P < 8
    (dict(P=8, N=16_384, dtype="f16", mode="rankorder"), "fold_small_kernel"),
    (dict(P=8, N=16_384, topo="torus", X=4, Y=2), "fold_ldg_kernel"),
    (dict(P=16, N=16_384), "fold_lat_kernel (one group)"),
    (dict(P=16, N=16_384, topo="torus", X=4, Y=4), "fold_lat_kernel"),
    (dict(P=32, N=16_384, dtype="f16", topo="torus", X=8, Y=4), "fold_lat_kernel"),
    (dict(P=64, N=16_384, topo="multiring", k=4), "fold_lat_kernel (one group)"),
    (dict(P=64, N=100_000, topo="multiring", k=4), "fold_small_kernel"),  # past one wave of the latency pass
    (dict(P=16, N=65_536), "fold_lat_kernel (one group)"),                # 512-byte items
    (dict(P=16, N=262_144), "fold_small_kernel"),                         # 2 KB items, one group below 32 ranks
    (dict(P=16, N=262_144, topo="torus", X=4, Y=4), "fold_lat_kernel"),  # 2 KB items, four groups
    (dict(P=16, N=524_288, topo="torus", X=4, Y=4), "fold_ldg_kernel"),  # 4 KB items
    (dict(P=32, N=524_288, dtype="f16", topo="torus", X=8, Y=4), "fold_lat_kernel"),
    (dict(P=16, N=524_288, dtype="f16"), "fold_lat_kernel (one group)"),  # binary16 hops, 2 KB items
    (dict(P=16, N=1_048_576, dtype="f16"), "fold_ldg_kernel"),            # binary16 hops, 4 KB items
    (dict(P=64, N=16_384, topo="torus_nd", dims=[4, 4, 4]), "fold_lat_nd_kernel"),
    (dict(P=64, N=2_000_000, topo="torus_nd", dims=[4, 4, 4]), "fold_nd_kernel"),
    (dict(P=32, N=2_000_000, dtype="f16", topo="torus_nd", dims=[4, 4, 2]), "fold_nd_h2_kernel"),
    (dict(P=16, N=16_384, mode="stepwise"), "step_kernel"),
    (dict(P=16, N=16_384, kernel="chunked"), "fold_chunked_kernel"),
    (dict(P=16, N=1_000_000, kernel="bulkload"), "fold_bulk_kernel"),
]


@pytest.mark.parametrize("case,want", DISPATCH, ids=[f"{i}-{w}" for i, (_, w) in enumerate(DISPATCH)])
def test_dispatch_rules(ddl, case, want):
    """ddl_plan_kernel_name reports the pass the library's own dispatch takes
    (the same function the launcher switches on), host-only."""
    with ddl.Plan(**case) as plan:
        assert plan.kernel_name == want


def test_kernel_name_follows_mode_and_kernel_changes(ddl):
    with ddl.Plan(16, 16_384, topo="torus", X=4, Y=4) as plan:
        assert plan.kernel_name == "fold_lat_kernel"
        plan.set_mode("rankorder")
        assert plan.kernel_name == "fold_lat_kernel (one group)"
        plan.set_mode("stepwise")
        assert plan.kernel_name == "step_kernel"
        plan.set_mode("fused")
        plan.set_kernel("chunked")
        assert plan.kernel_name == "fold_chunked_kernel"
    with pytest.raises(ddl.DDLError):
        ddl.ddl_plan_kernel_name(None)


def test_layer_sizes_that_would_wrap_are_refused(ddl):
    """A layer list whose sum wraps around 2^64 to N is not a partition of N."""
    with ddl.Plan(3, 1) as plan:
        with pytest.raises(ddl.DDLError) as ei:
            ddl.ddl_plan_set_layers(plan.handle, [2 ** 64 - 1, 2])
        assert ei.value.status == ddl.DDL_ERR_INVALID_ARG
        assert plan.buckets() == [(0, 1)]


def test_noalloc_refuses_oversized_problems_before_any_gpu_work(ddl):
    """Sizes are checked without forming N * element size (which could wrap),
    and the table count stops at the first table that no longer fits the
    static array: both refusals come back at once, before any CUDA call."""
    import time
    ring = ddl.ddl_topology_t(ddl.DDL_RING, 1, 0, 0)
    fake = [1 << 30, 2 << 30]
    for N in (2 ** 62 + 1, 2 ** 63 + 7):     # N * 4 wraps to a small number
        with pytest.raises(ddl.DDLError) as ei:
            ddl.ddl_allreduce_noalloc(2, N, ddl.DDL_FP32, ring, 0, None, fake, 0.5)
        assert ei.value.status == ddl.DDL_ERR_UNSUPPORTED
    t = time.perf_counter()
    with pytest.raises(ddl.DDLError) as ei:        # 2^40 bytes per rank: ~2^27 tiles, far over 1 MiB of tables
        ddl.ddl_allreduce_noalloc(2, 2 ** 38, ddl.DDL_FP32, ring, 4, None, fake, 0.5)
    assert ei.value.status == ddl.DDL_ERR_UNSUPPORTED
    assert time.perf_counter() - t < 1.0
    torus = ddl.ddl_topology_t(3, 1, 0, 0)      # the n-D kind is not part of the topology struct
    with pytest.raises(ddl.DDLError) as ei:
        ddl.ddl_allreduce_noalloc(2, 100, ddl.DDL_FP32, torus, 0, None, fake, 0.5)
    assert ei.value.status == ddl.DDL_ERR_INVALID_ARG

