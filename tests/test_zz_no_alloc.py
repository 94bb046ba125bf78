"""ddl_allreduce_noalloc, the allocation-free entry point, against ddl_allreduce.

Some callers cannot call cudaMalloc: their device memory all belongs to a
framework's own pool, or their training loop must not take cudaMalloc's
implicit device synchronisation, or their deployment fixes its memory
footprint at start-up.  ddl_allreduce_noalloc serves them: it keeps the fused
kernel's work tables in a static device array inside the library instead of a
plan's device memory.  This test calls it through the C ABI twice in a row (on
different inputs, so the second call runs over the first call's leftover
tables) and checks each result against the plan-based ddl_allreduce on the
same inputs.  Both run the schedule in its own order, so the tolerance is the
one every schedule-order test here uses: bit-for-bit equality.

It also checks the allocation-free results against the oracle's
step-by-step emulation (bit for bit, as for every schedule-order path), on a
binary16 torus with a layer list, on rank buffers that are not 16-byte
aligned, and on a single rank; and that ddl_noalloc_check, which reads the
kernel's error word without allocating, reports no error after good calls.

The file is named to be collected last, and it builds what it needs, so it
passes both on its own in a fresh process and after the other tests.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402


@pytest.fixture(scope="module")
def ddl():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    from gradient_all_reduce_ddl_gb300 import ddl as mod
    return mod


CASES = [
    dict(P=16, N=1_000_003, dtype="f32", topo="torus", X=4, Y=4),
    dict(P=8, N=300_001, dtype="f16", topo="multiring", k=3, bucket_bytes=200_000,
         layers=[100_000, 50_001, 75_000, 75_000]),
    dict(P=5, N=123_457, dtype="f32", topo="ring", bucket_bytes=100_000),
]


def _bufs(P, N, dtype, seed):
    tdt = torch.float16 if dtype == "f16" else torch.float32
    out = []
    for r in range(P):
        t = torch.empty(N, dtype=tdt, device="cuda:0")
        synth.fill_device(t.data_ptr(), N, seed, r, "normal", 1e-2 if dtype == "f16" else 1e-3, dtype,
                          stream=torch.cuda.current_stream().cuda_stream)
        out.append(t)
    return out


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.float16 else t.view(torch.int32)


@pytest.mark.parametrize("case", CASES, ids=["torus4x4-f32", "multiring-f16-layers", "ring-f32-buckets"])
def test_noalloc_matches_plan_on_two_calls_in_a_row(ddl, case):
    P, N, dtype = case["P"], case["N"], case["dtype"]
    topo = ddl.ddl_topology_t(ddl.TOPOLOGIES[case["topo"]], case.get("k", 1), case.get("X", 0), case.get("Y", 0))
    scale = float(np.float32(1.0 / P))
    layers = case.get("layers")
    bucket_bytes = case.get("bucket_bytes", 0)
    for call, seed in enumerate((11, 12)):
        a = _bufs(P, N, dtype, seed)
        b = [t.clone() for t in a]
        torch.cuda.synchronize()
        ddl.ddl_allreduce_noalloc(P, N, ddl.DTYPES[dtype], topo, bucket_bytes, layers, a, scale)
        ddl.ddl_noalloc_check()
        with ddl.Plan(P, N, dtype, case["topo"], k=case.get("k", 1), X=case.get("X", 0), Y=case.get("Y", 0),
                      bucket_bytes=bucket_bytes, layers=layers) as plan:
            plan.allreduce(b, scale)
            torch.cuda.synchronize()
            plan.check()
        for r in range(P):
            assert torch.equal(_bits(a[r]), _bits(b[r])), f"call {call + 1}, rank {r}"
        assert not torch.equal(_bits(a[0]), _bits(_bufs(P, N, dtype, seed)[0]))  # the data did change


def test_noalloc_refuses_tables_beyond_the_static_array(ddl):
    # 300M fp32 elements per rank need ~2.3 MB of work items: over the 1 MiB array
    topo = ddl.ddl_topology_t(ddl.DDL_RING, 1, 0, 0)
    with pytest.raises(ddl.DDLError) as ei:
        ddl.ddl_allreduce_noalloc(2, 300_000_000, ddl.DDL_FP32, topo, 0, None, [1 << 30, 2 << 30], 0.5)
    assert ei.value.status == ddl.DDL_ERR_UNSUPPORTED


ORACLE_CASES = [
    dict(P=4, N=9_999, dtype="f16", topo="torus", X=2, Y=2, bucket_bytes=6_000, layers=[3_000, 999, 4_000, 2_000]),
    dict(P=16, N=60_001, dtype="f16", topo="torus", X=4, Y=4, bucket_bytes=40_000,
         layers=[10_000, 20_001, 5_000, 25_000]),
    dict(P=8, N=30_011, dtype="f32", topo="multiring", k=3, bucket_bytes=50_000),
    dict(P=5, N=20_003, dtype="f32", topo="ring", misalign=1),
    dict(P=6, N=12_345, dtype="f16", topo="torus", X=3, Y=2, misalign=3),
    dict(P=1, N=777, dtype="f32", topo="ring"),
    dict(P=1, N=1_000, dtype="f16", topo="torus", X=1, Y=1),
]


def _host(P, N, dtype, seed):
    sigma = 1e-2 if dtype == "f16" else 1e-3
    return [synth.draw_rank(seed, r, N, "normal", sigma, dtype) for r in range(P)]


def _to_device(h, misalign):
    tdt = torch.float16 if h.dtype == np.uint16 else torch.float32
    raw = torch.from_numpy(h.view(np.int16) if h.dtype == np.uint16 else h).to("cuda:0")
    big = torch.zeros(h.size + misalign, dtype=tdt, device="cuda:0")
    big[misalign:] = raw.view(tdt)
    return big[misalign:]


def _numpy_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.float16 else t.cpu().numpy()


@pytest.mark.parametrize("case", ORACLE_CASES,
                         ids=["torus2x2-f16-layers", "torus4x4-f16-layers", "multiring-f32-buckets",
                              "ring-f32-unaligned", "torus3x2-f16-unaligned", "ring-P1", "torus1x1-f16"])
def test_noalloc_matches_oracle(ddl, case):
    P, N, dtype = case["P"], case["N"], case["dtype"]
    topo = ddl.ddl_topology_t(ddl.TOPOLOGIES[case["topo"]], case.get("k", 1), case.get("X", 0), case.get("Y", 0))
    scale = float(np.float32(1.0 / P))
    layers = case.get("layers")
    bucket_bytes = case.get("bucket_bytes", 0)
    host = _host(P, N, dtype, 31)
    bufs = [_to_device(h, case.get("misalign", 0)) for h in host]
    torch.cuda.synchronize()
    ddl.ddl_allreduce_noalloc(P, N, ddl.DTYPES[dtype], topo, bucket_bytes, layers, bufs, scale)
    ddl.ddl_noalloc_check()
    ref = [h.copy() for h in host]
    cfg = oracle.Config(P, N, dtype, case["topo"], k=case.get("k", 1), X=case.get("X", 0), Y=case.get("Y", 0),
                        bucket_bytes=bucket_bytes, layers=layers)
    oracle.emulate(cfg, ref, scale)
    for r in range(P):
        got = _numpy_bits(bufs[r])
        bad = np.nonzero(got != ref[r])[0]
        assert bad.size == 0, f"rank {r}: {bad.size} elements differ from the oracle, first at {bad[:5]}"
