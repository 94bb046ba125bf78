"""Parity of the CUDA path (through the C ABI) with the oracle.

Schedule-order modes (fused, stepwise) must match the oracle bit for bit;
the rank-order mode must be within 1e-6 (fp32) / 2e-3 (fp16) normwise of the
fp64 sum of the stored inputs.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (device_bufs_from_host, device_bufs_generated, edge_samples, oracle_cfg, rankorder_margins,
                      to_numpy_bits, torch_dtype)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ddl():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    from gradient_all_reduce_ddl_gb300 import ddl as mod
    return mod


DEV = "cuda:0"


def _w(P, N, dtype="f32", topo="ring", k=1, X=0, Y=0, bucket_bytes=0, layers=None, dist="normal", sigma=None,
       scale=None, seed=1, dims=None):
    if sigma is None:
        sigma = 1e-2 if dtype == "f16" else 1e-3
    if scale is None:
        scale = float(np.float32(1.0 / P))
    return synth.Workload(name="t", P=P, N=N, dtype=dtype, topo=topo, k=k, X=X, Y=Y, bucket_bytes=bucket_bytes,
                          layers=None if layers is None else tuple(layers), scale=scale, dist=dist, sigma=sigma,
                          seed=seed, dims=None if dims is None else tuple(dims))


def _host_inputs(w):
    return [w.rank_values(r) for r in range(w.P)]


def _check_exact(ddl, w, mode="fused", kernel="auto", misalign=0):
    host = _host_inputs(w)
    if misalign:
        # rank buffers that start `misalign` elements into a larger tensor
        bufs = []
        for h in host:
            big = torch.zeros(w.N + misalign, dtype=torch_dtype(w.dtype), device=DEV)
            dev = device_bufs_from_host([h], DEV)[0]
            big[misalign:] = dev
            bufs.append(big[misalign:])
    else:
        bufs = device_bufs_from_host(host, DEV)
    with ddl.Plan.for_workload(w, mode=mode, kernel=kernel) as plan:
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        plan.check()
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    for r in range(w.P):
        got = to_numpy_bits(bufs[r])
        if not np.array_equal(got, ref[r]):
            bad = np.nonzero(got != ref[r])[0]
            raise AssertionError(f"rank {r}: {bad.size} elements differ, first at {bad[:8]}: "
                                 f"got {got[bad[:4]]} want {ref[r][bad[:4]]}")


# Small cases: several 8 KB tiles per rank, ragged tails, every schedule.
SMALL = [
    dict(P=4, N=65_536, dist="int1000", scale=1.0),
    dict(P=1, N=5000),
    dict(P=2, N=10_001),
    dict(P=3, N=7),
    dict(P=5, N=40_003),
    dict(P=7, N=30_011, bucket_bytes=20_000),
    dict(P=16, N=70_001, topo="multiring", k=2),
    dict(P=9, N=50_000, topo="multiring", k=5, bucket_bytes=40_000),
    dict(P=64, N=20_011, topo="multiring", k=4, bucket_bytes=30_000),
    dict(P=4, N=8, topo="torus", X=2, Y=2),
    dict(P=16, N=99_999, topo="torus", X=4, Y=4),
    dict(P=12, N=40_000, topo="torus", X=3, Y=4, bucket_bytes=50_000),
    dict(P=32, N=33_333, topo="torus", X=8, Y=4),
    dict(P=6, N=12_345, topo="torus", X=6, Y=1),
    dict(P=6, N=12_345, topo="torus", X=1, Y=6),
    dict(P=200, N=3001, topo="ring"),
    dict(P=16, N=20_000, layers=[1000, 5000, 3, 7000, 6997], bucket_bytes=20_000),
    dict(P=8, N=30_001, topo="torus_nd", dims=[2, 2, 2]),
    dict(P=64, N=20_011, topo="torus_nd", dims=[4, 4, 4], bucket_bytes=30_000),
    dict(P=24, N=17_777, topo="torus_nd", dims=[2, 3, 2, 2]),
    dict(P=12, N=9_001, topo="torus_nd", dims=[3, 1, 4]),
]


@pytest.mark.parametrize("kernel", ["ldg", "bulkload", "chunked"])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_fused_matches_oracle(ddl, case, dtype, kernel):
    if dtype == "f16" and case.get("dist") == "int1000":
        pytest.skip("integer case is fp32")
    _check_exact(ddl, _w(dtype=dtype, **case), kernel=kernel)


@pytest.mark.parametrize("kernel", ["ldg", "bulkload", "chunked"])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("case", [SMALL[4], SMALL[7], SMALL[11], SMALL[16], SMALL[18]])
def test_fused_unaligned_buffers_match_oracle(ddl, case, dtype, kernel):
    """Rank pointers that are not 16-byte aligned take the element-wise path."""
    _check_exact(ddl, _w(dtype=dtype, **case), misalign=1, kernel=kernel)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("case", [SMALL[0], SMALL[1], SMALL[4], SMALL[7], SMALL[10], SMALL[12], SMALL[14],
                                  SMALL[17], SMALL[19]])
def test_stepwise_matches_oracle(ddl, case, dtype):
    if dtype == "f16" and case.get("dist") == "int1000":
        pytest.skip("integer case is fp32")
    _check_exact(ddl, _w(dtype=dtype, **case), mode="stepwise")


@pytest.mark.parametrize("dtype,tol", [("f32", 1e-6), ("f16", 2e-3)])
@pytest.mark.parametrize("case", [dict(P=16, N=100_003), dict(P=32, N=50_000, topo="torus", X=8, Y=4),
                                  dict(P=64, N=30_001, topo="multiring", k=4, bucket_bytes=40_000),
                                  dict(P=256, N=9_001), dict(P=7, N=20_000, dist="int1000", scale=1.0)])
def test_rankorder_within_tolerance(ddl, case, dtype, tol):
    """Rank-order mode: normwise within 1e-6 (fp32) / 2e-3 (fp16) of the
    binary64 sum of the stored inputs, and every element within the error
    bound of a P-term binary32 left fold (plus one binary16 rounding for
    fp16); all ranks identical."""
    w = _w(dtype=dtype, **case)
    host = _host_inputs(w)
    bufs = device_bufs_from_host(host, DEV)
    with ddl.Plan.for_workload(w, mode="rankorder") as plan:
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        plan.check()
    got0 = to_numpy_bits(bufs[0])
    norm, elem = rankorder_margins(host, got0, w.scale, dtype)
    assert norm <= tol, norm
    assert elem <= 1.0, elem
    if case.get("dist") == "int1000" and dtype == "f32":
        # integers: every order gives the exact sum
        assert np.array_equal(got0, np.stack(host).astype(np.int64).sum(axis=0).astype(np.float32))
    for r in range(1, w.P):
        assert np.array_equal(to_numpy_bits(bufs[r]), got0)


SGD_CASES = [
    dict(P=4, N=50_001),
    dict(P=16, N=70_001, topo="multiring", k=2, bucket_bytes=100_000),
    dict(P=16, N=99_999, topo="torus", X=4, Y=4),
    dict(P=32, N=20_000, topo="torus", X=8, Y=4, dtype="f16"),
    dict(P=8, N=30_011, dtype="f16", bucket_bytes=20_000),
    # small items: the staged pass (one group; several groups with binary16
    # hops and cut columns; P < 16), and 2 KB items in the register pass
    dict(P=64, N=9_001, topo="multiring", k=4),
    dict(P=32, N=16_385, topo="torus", X=8, Y=4, dtype="f16"),
    dict(P=8, N=20_001, topo="torus", X=4, Y=2, dtype="f16"),
    dict(P=16, N=200_003, topo="torus", X=4, Y=4),
]


@pytest.mark.parametrize("keep", [True, False])
@pytest.mark.parametrize("mom", [True, False])
@pytest.mark.parametrize("case", SGD_CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_allreduce_sgd_matches_oracle(ddl, case, mom, keep):
    w = _w(seed=41, **case)
    host = _host_inputs(w)
    rng = np.random.default_rng(7)
    p0 = rng.standard_normal(w.N).astype(np.float32)
    v0 = (rng.standard_normal(w.N) * 0.1).astype(np.float32)
    lr, mu, wd = 0.05, (0.9 if mom else 0.0), 1e-4
    g_ref = [h.copy() for h in host]
    p_ref = [p0.copy() for _ in range(w.P)]
    m_ref = [v0.copy() for _ in range(w.P)] if mom else None
    oracle.sgd(oracle_cfg(w), g_ref, p_ref, m_ref, w.scale, lr, mu, wd)
    grads = device_bufs_from_host(host, DEV)
    params = [torch.from_numpy(p0).to(DEV) for _ in range(w.P)]
    moms = [torch.from_numpy(v0).to(DEV) for _ in range(w.P)] if mom else None
    with ddl.Plan.for_workload(w) as plan:
        plan.allreduce_sgd(grads, params, moms, w.scale, lr, mu, wd, keep_grads=keep)
        torch.cuda.synchronize()
        plan.check()
    for r in range(w.P):
        assert np.array_equal(params[r].cpu().numpy(), p_ref[r]), ("params", r)
        if mom:
            assert np.array_equal(moms[r].cpu().numpy(), m_ref[r]), ("moms", r)
        assert np.array_equal(to_numpy_bits(grads[r]), g_ref[r] if keep else host[r]), ("grads", r)


# Small buffers (items of 1-4 KB per rank): P >= 32 takes the latency pass
# (shared-memory staged, the fold's levels folded group by group in
# parallel; 2D and n-D tori) while its tiles fit in 96 KB; smaller
# single-group unrounded folds take the small-item pass; the rest the
# register passes.  N is odd, so items end in cut columns.
SMALL_BUFFERS = [
    dict(P=32, N=40_001, topo="torus", X=8, Y=4),
    dict(P=32, N=9_999, topo="torus", X=4, Y=8),
    dict(P=32, N=20_003, topo="torus", X=1, Y=32),
    dict(P=32, N=20_003, topo="torus", X=32, Y=1),
    dict(P=48, N=30_007, topo="multiring", k=3, bucket_bytes=40_000),
    dict(P=64, N=16_385, topo="multiring", k=4),
    dict(P=64, N=70_001, topo="torus", X=8, Y=8),
    dict(P=96, N=20_001, topo="torus", X=12, Y=8),
    dict(P=40, N=5_001, layers=[1_000, 2_001, 2_000], bucket_bytes=4_000),
    dict(P=8, N=40_001, topo="multiring", k=2),
    dict(P=12, N=30_001, topo="torus", X=4, Y=3),
    dict(P=64, N=20_001, topo="torus_nd", dims=[4, 4, 4]),
    dict(P=32, N=30_003, topo="torus_nd", dims=[4, 4, 2]),
    dict(P=32, N=12_345, topo="torus_nd", dims=[2, 4, 4]),
    dict(P=32, N=9_001, topo="torus_nd", dims=[4, 1, 8]),
    dict(P=32, N=20_001, topo="torus_nd", dims=[8, 4]),
    dict(P=48, N=30_001, topo="torus_nd", dims=[2, 3, 2, 4], bucket_bytes=50_000),
]


@pytest.mark.parametrize("mode", ["fused", "rankorder"])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("case", SMALL_BUFFERS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_small_buffer_passes_match_oracle(ddl, case, dtype, mode):
    w = _w(dtype=dtype, seed=23, **case)
    if mode == "fused":
        _check_exact(ddl, w)
        return
    host = _host_inputs(w)
    bufs = device_bufs_from_host(host, DEV)
    with ddl.Plan.for_workload(w, mode="rankorder") as plan:
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        plan.check()
    got0 = to_numpy_bits(bufs[0])
    # rank order is one binary32 left fold in rank order: the same bits from
    # the element-wise path on unaligned copies of the inputs
    big = []
    for h in host:
        t = torch.zeros(w.N + 1, dtype=torch_dtype(w.dtype), device=DEV)
        t[1:] = device_bufs_from_host([h], DEV)[0]
        big.append(t[1:])
    with ddl.Plan.for_workload(w, mode="rankorder") as plan:
        plan.allreduce(big, w.scale)
        torch.cuda.synchronize()
    assert np.array_equal(got0, to_numpy_bits(big[0]))
    norm, elem = rankorder_margins(host, got0, w.scale, dtype)
    assert norm <= (1e-6 if dtype == "f32" else 2e-3) and elem <= 1.0, (norm, elem)
    for r in range(1, w.P):
        assert np.array_equal(to_numpy_bits(bufs[r]), got0), r


# Buffers between the latency passes and the HBM regime, each landing on the
# pass named (2 and 4 KB work items: the one-column register passes, the
# small-item pass with 4 KB items, the latency pass at its 2 KB limit), several
# with sizes whose chunks end inside 16-byte columns.
MID_SIZE = [
    (dict(P=16, N=524_288, topo="torus", X=4, Y=4), "fold_ldg_kernel"),
    (dict(P=16, N=600_001, topo="torus", X=4, Y=4), "fold_ldg_kernel"),
    (dict(P=8, N=400_003, topo="torus", X=4, Y=2), "fold_ldg_kernel"),
    (dict(P=32, N=1_048_576, dtype="f16", topo="torus", X=8, Y=4), "fold_ldg_kernel"),
    (dict(P=16, N=1_000_003, dtype="f16"), "fold_ldg_kernel"),
    (dict(P=16, N=524_288, dtype="f16"), "fold_lat_kernel (one group)"),
    (dict(P=16, N=262_144, topo="torus", X=4, Y=4), "fold_lat_kernel"),
    (dict(P=16, N=500_001), "fold_small_kernel"),
    (dict(P=64, N=262_144, topo="torus_nd", dims=[4, 4, 4]), "fold_nd_kernel"),
    (dict(P=64, N=500_003, topo="torus_nd", dims=[4, 4, 4]), "fold_nd_kernel"),
    (dict(P=32, N=1_048_576, dtype="f16", topo="torus_nd", dims=[4, 4, 2]), "fold_nd_h2_kernel"),
    (dict(P=32, N=333_333, dtype="f16", topo="torus_nd", dims=[4, 4, 2]), "fold_lat_nd_kernel"),
    (dict(P=64, N=400_001, dtype="f16", topo="torus_nd", dims=[4, 4, 4]), "fold_nd_h2_kernel"),
]


@pytest.mark.parametrize("case,kernel", MID_SIZE, ids=[f"{i}-{k}" for i, (_, k) in enumerate(MID_SIZE)])
def test_mid_size_passes_match_oracle(ddl, case, kernel):
    w = _w(seed=29, **case)
    with ddl.Plan.for_workload(w) as plan:
        assert plan.kernel_name == kernel
    _check_exact(ddl, w)


@pytest.mark.parametrize("kernel", ["bulkload", "chunked"])
@pytest.mark.parametrize("P", [2, 4])
def test_small_p_with_a_staged_kernel_choice(ddl, kernel, P):
    """P <= 4 with a staged kernel chosen.  A staged tile once grew to 16 KB
    per rank at such P, more than the register pass covers, and the fused
    SGD pass runs the plan's items in the register pass's shape whatever the
    choice: the all-reduce and the SGD pass must match the oracle."""
    w = _w(P=P, N=200_003, seed=77)
    _check_exact(ddl, w, kernel=kernel)
    host = _host_inputs(w)
    p0 = np.linspace(-1, 1, w.N, dtype=np.float32)
    g_ref = [h.copy() for h in host]
    p_ref = [p0.copy() for _ in range(w.P)]
    oracle.sgd(oracle_cfg(w), g_ref, p_ref, None, w.scale, 0.1, 0.0, 0.0)
    grads = device_bufs_from_host(host, DEV)
    params = [torch.from_numpy(p0).to(DEV) for _ in range(w.P)]
    with ddl.Plan.for_workload(w, kernel=kernel) as plan:
        plan.allreduce_sgd(grads, params, None, w.scale, 0.1)
        torch.cuda.synchronize()
        plan.check()
    for r in range(w.P):
        assert np.array_equal(to_numpy_bits(grads[r]), g_ref[r]), r
        assert np.array_equal(params[r].cpu().numpy(), p_ref[r]), r


def test_allreduce_sgd_unaligned_and_errors(ddl):
    w = _w(P=6, N=12_345, seed=43)
    host = _host_inputs(w)
    p0 = np.linspace(-1, 1, w.N, dtype=np.float32)
    g_ref = [h.copy() for h in host]
    p_ref = [p0.copy() for _ in range(w.P)]
    m_ref = [np.zeros(w.N, np.float32) for _ in range(w.P)]
    oracle.sgd(oracle_cfg(w), g_ref, p_ref, m_ref, w.scale, 0.1, 0.5, 0.01)
    grads = device_bufs_from_host(host, DEV)
    big = [torch.zeros(w.N + 1, device=DEV) for _ in range(w.P)]       # parameters 4 bytes off 16-byte alignment
    params = [b[1:] for b in big]
    for q in params:
        q.copy_(torch.from_numpy(p0).to(DEV))
    moms = [torch.zeros(w.N, device=DEV) for _ in range(w.P)]
    with ddl.Plan.for_workload(w) as plan:
        plan.allreduce_sgd(grads, params, moms, w.scale, 0.1, 0.5, 0.01)
        torch.cuda.synchronize()
        for r in range(w.P):
            assert np.array_equal(params[r].cpu().numpy(), p_ref[r])
            assert np.array_equal(moms[r].cpu().numpy(), m_ref[r])
        with pytest.raises(ddl.DDLError) as ei:          # momentum without buffers
            plan.allreduce_sgd(grads, params, None, w.scale, 0.1, 0.5, 0.0)
        assert ei.value.status == ddl.DDL_ERR_INVALID_ARG
        with pytest.raises(ddl.DDLError):                # a parameter buffer that is a gradient buffer
            plan.allreduce_sgd(grads, [grads[0]] + params[1:], moms, w.scale, 0.1, 0.5, 0.0)
        with pytest.raises(ddl.DDLError):                # new gradients that overlap the cached parameters
            plan.allreduce_sgd([params[0]] + grads[1:], params, moms, w.scale, 0.1, 0.5, 0.0)
    with ddl.Plan(8, 1000, topo="torus_nd", dims=[2, 2, 2]) as plan:
        g8 = [torch.zeros(1000, device=DEV) for _ in range(8)]
        p8 = [torch.zeros(1000, device=DEV) for _ in range(8)]
        with pytest.raises(ddl.DDLError) as ei:
            plan.allreduce_sgd(g8, p8, None, 0.125, 0.1)
        assert ei.value.status == ddl.DDL_ERR_UNSUPPORTED


def test_oracle_binary16_rounding_equals_device_conversion():
    """The oracle's own binary32 -> binary16 rounding against the GPU's
    (torch .half() on the device: round to nearest even, subnormals kept,
    overflow to infinity) on all 2^32 binary32 bit patterns, 2^26 at a time;
    a NaN must give a NaN."""
    step = 1 << 26
    for lo in range(0, 1 << 32, step):
        mine = torch.from_numpy(oracle.f32_patterns_to_f16(lo, lo + step).view(np.int16)).to(DEV)
        p64 = torch.arange(lo, lo + step, dtype=torch.int64, device=DEV)
        x = torch.where(p64 >= (1 << 31), p64 - (1 << 32), p64).to(torch.int32).view(torch.float32)
        dev = x.half().view(torch.int16)
        nan = torch.isnan(x)
        assert torch.equal(dev[~nan], mine[~nan]), hex(lo)
        dn = dev[nan].to(torch.int32) & 0xFFFF
        assert bool((((dn & 0x7C00) == 0x7C00) & ((dn & 0x3FF) != 0)).all()), hex(lo)


def test_packed_hop_add_over_every_binary16_pair(ddl):
    """Every binary16 pair (a, b) through one hop add of the fused pass.

    A 3-rank fp16 ring whose rank 2 holds -0 everywhere, scale 1: chunk 0
    folds (a + b, rounded to binary16 for the next hop) + (-0), and that last
    add and the scale leave the hop value as it is.  So chunk 0 must equal
    fl16(fl32(a) + fl32(b)), computed here by torch on the device (widen, add
    in binary32, round to nearest even).  The pass takes this hop as a packed
    binary16 add; a NaN sum must give a NaN."""
    M = 1 << 28
    N = 3 * M
    bufs = [torch.zeros(N, dtype=torch.int16, device=DEV) for _ in range(3)]
    bufs[2].fill_(-0x8000)                                   # binary16 -0
    lo = torch.arange(M, dtype=torch.int32, device=DEV)

    def as16(v):
        return torch.where(v >= 0x8000, v - 0x10000, v).to(torch.int16)

    with ddl.Plan(3, N, "f16", "ring") as plan:
        for k in range(16):                                  # 2^28 pairs per pass, 2^32 in all
            a = as16(lo & 0xFFFF)
            b = as16((lo >> 16) + k * (M >> 16))
            bufs[0][:M] = a
            bufs[0][M:] = 0
            bufs[1][:M] = b
            bufs[1][M:] = 0
            bufs[2].fill_(-0x8000)
            plan.allreduce([t.view(torch.float16) for t in bufs], 1.0)
            want = (a.view(torch.float16).float() + b.view(torch.float16).float()).half()
            nan = torch.isnan(want)
            for r in range(3):
                got = bufs[r][:M]
                assert torch.equal(got[~nan], want.view(torch.int16)[~nan]), (k, r)
                assert bool(torch.isnan(got.view(torch.float16)[nan]).all()), (k, r)
        plan.check()


SLAB_CASES = [
    dict(P=4, N=50_003),
    dict(P=16, N=99_999, topo="torus", X=4, Y=4),
    dict(P=32, N=33_333, topo="torus", X=8, Y=4, dtype="f16"),
    dict(P=64, N=20_011, topo="multiring", k=4, bucket_bytes=30_000),
    dict(P=128, N=5_003),
    dict(P=12, N=40_000, topo="torus", X=3, Y=4, bucket_bytes=50_000, dtype="f16"),
    dict(P=8, N=30_001, topo="torus_nd", dims=[2, 2, 2]),
]


@pytest.mark.parametrize("kernel", ["ldg", "bulkload"])
@pytest.mark.parametrize("case", SLAB_CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_slab_matches_oracle(ddl, case, kernel):
    """Rank buffers in one slab (rank r at base + r * stride) give the
    oracle's bits, aligned or not."""
    w = _w(seed=71, **case)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    es = w.esize
    for pad in (0, 24):                           # pad 24 B: stride not a multiple of 16 -> element-wise path
        stride = (w.N * es + 255) // 256 * 256 + pad
        slab = torch.zeros(stride * w.P // 2 + 16, dtype=torch.int16, device=DEV)
        base = slab.data_ptr()
        bufs = []
        for r in range(w.P):
            t = slab.view(torch.uint8)[r * stride: r * stride + w.N * es].view(torch_dtype(w.dtype))
            t.copy_(device_bufs_from_host([host[r]], DEV)[0])
            bufs.append(t)
        with ddl.Plan.for_workload(w, kernel=kernel) as plan:
            plan.allreduce_slab(base, stride, w.scale)
            torch.cuda.synchronize()
            plan.check()
            for r in range(w.P):
                assert np.array_equal(to_numpy_bits(bufs[r]), ref[r]), (pad, r)
            with pytest.raises(ddl.DDLError):     # ranks would overlap
                plan.allreduce_slab(base, w.N * es - 16, w.scale)


def test_device_generator_matches_host(ddl):
    for dist, dtype, sigma in [("normal", "f32", 1e-3), ("normal", "f16", 1e-2), ("int1000", "f32", 1.0)]:
        w = _w(P=3, N=100_003, dtype=dtype, dist=dist, sigma=sigma, seed=99)
        dev = device_bufs_generated(w, DEV)
        torch.cuda.synchronize()
        for r in range(w.P):
            assert np.array_equal(to_numpy_bits(dev[r]), w.rank_values(r)), (dist, dtype, r)


@pytest.mark.parametrize("name", ["torus4x4_resnet50", "torus8x4_resnet50_f16", "multiring64_resnet101",
                                  "torus4x4x4_resnet101"])
def test_full_size_stepwise_sampled(ddl, name):
    """The stepwise mode (one launch per communication step) at full size:
    bit-exact with the oracle's closed form on sampled elements, ranks
    identical."""
    w = synth.WORKLOADS[name]
    bufs = device_bufs_generated(w, DEV)
    with ddl.Plan.for_workload(w, mode="stepwise") as plan:
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        plan.check()
    view = torch.int16 if w.dtype == "f16" else torch.int32
    for r in range(1, w.P):
        assert torch.equal(bufs[r].view(view), bufs[0].view(view)), r
    rng = np.random.default_rng(1234)
    idx = np.unique(np.concatenate([rng.integers(0, w.N, 30_000), edge_samples(w)]))
    x_rows = np.stack([w.rank_values(r, idx.astype(np.uint64)) for r in range(w.P)], axis=1)
    want = oracle.closed_form(oracle_cfg(w), x_rows, idx.astype(np.uint64), w.scale)
    got = to_numpy_bits(bufs[0][torch.from_numpy(idx).to(DEV)])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {idx.size} sampled elements differ, e.g. idx {idx[bad[:5]]}"
    del bufs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,tol", [("torus4x4_resnet50", 1e-6), ("torus8x4_resnet50_f16", 2e-3),
                                      ("ring16_lm300m", 1e-6), ("multiring64_resnet101", 1e-6)])
def test_full_size_rankorder_within_tolerance(ddl, name, tol):
    """The rank-order mode at full size: normwise error against the binary64
    sum of the stored inputs (times the scale) on sampled elements, within
    1e-6 (fp32) or 2e-3 (fp16), and every sampled element within the error
    bound of a P-term binary32 left fold (plus one binary16 rounding for
    fp16); ranks identical."""
    w = synth.WORKLOADS[name]
    bufs = device_bufs_generated(w, DEV)
    with ddl.Plan.for_workload(w, mode="rankorder") as plan:
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        plan.check()
    view = torch.int16 if w.dtype == "f16" else torch.int32
    for r in range(1, w.P):
        assert torch.equal(bufs[r].view(view), bufs[0].view(view)), r
    rng = np.random.default_rng(4321)
    idx = np.unique(rng.integers(0, w.N, 200_000))
    host = [w.rank_values(r, idx.astype(np.uint64)) for r in range(w.P)]
    got0 = to_numpy_bits(bufs[0][torch.from_numpy(idx).to(DEV)])
    norm, elem = rankorder_margins(host, got0, w.scale, w.dtype)
    assert norm <= tol, norm
    assert elem <= 1.0, elem
    del bufs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["torus4x4_resnet50", "torus8x4_resnet50_f16", "multiring64_resnet101"])
def test_full_size_sgd_sampled(ddl, name):
    """The all-reduce fused with momentum SGD at full size, as the bench's
    --sgd study runs it.  On sampled elements: the stored averaged gradient
    from the oracle's closed form; the update of two ranks' own parameters and
    momenta (different on each rank) from the oracle's SGD on a one-rank
    problem fed that gradient (a one-rank all-reduce with scale 1 leaves it
    unchanged, so only the update remains)."""
    w = synth.WORKLOADS[name]
    lr, mu, wd = 0.01, 0.9, 1e-4
    bufs = device_bufs_generated(w, DEV)
    params, moms = [], []
    for r in range(w.P):
        pt = torch.empty(w.N, dtype=torch.float32, device=DEV)
        mt = torch.empty(w.N, dtype=torch.float32, device=DEV)
        synth.fill_device(pt.data_ptr(), w.N, w.seed + 100, r, "normal", 1.0, "f32")
        synth.fill_device(mt.data_ptr(), w.N, w.seed + 200, r, "normal", 0.1, "f32")
        params.append(pt)
        moms.append(mt)
    with ddl.Plan.for_workload(w) as plan:
        plan.allreduce_sgd(bufs, params, moms, w.scale, lr, mu, wd, keep_grads=True)
        torch.cuda.synchronize()
        plan.check()
    rng = np.random.default_rng(99)
    idx = np.unique(np.concatenate([rng.integers(0, w.N, 20_000), edge_samples(w)[::7]]))
    x_rows = np.stack([w.rank_values(r, idx.astype(np.uint64)) for r in range(w.P)], axis=1)
    g = oracle.closed_form(oracle_cfg(w), x_rows, idx.astype(np.uint64), w.scale)
    t_idx = torch.from_numpy(idx).to(DEV)
    assert np.array_equal(to_numpy_bits(bufs[0][t_idx]), g)
    one = oracle.Config(1, idx.size, w.dtype, "ring")
    for r in (0, w.P - 1):
        p_want = synth.draw(w.seed + 100, r, idx.astype(np.uint64), "normal", 1.0, "f32").copy()
        m_want = synth.draw(w.seed + 200, r, idx.astype(np.uint64), "normal", 0.1, "f32").copy()
        oracle.sgd(one, [g.copy()], [p_want], [m_want], 1.0, lr, mu, wd)
        assert np.array_equal(params[r][t_idx].cpu().numpy(), p_want), ("params", r)
        assert np.array_equal(moms[r][t_idx].cpu().numpy(), m_want), ("moms", r)
    del bufs, params, moms
    torch.cuda.empty_cache()


# The largest P the plan takes (256: rank orders are stored as bytes) on every
# schedule, and the smallest buffers (fewer elements than ranks or chunks).
EXTREME = [
    dict(P=256, N=9_001),
    dict(P=256, N=20_011, topo="multiring", k=4),
    dict(P=256, N=12_345, topo="torus", X=16, Y=16),
    dict(P=256, N=7_777, topo="torus_nd", dims=[4, 4, 4, 4]),
    dict(P=5, N=1),
    dict(P=9, N=4, topo="torus", X=3, Y=3),
    dict(P=16, N=3, topo="multiring", k=2),
    dict(P=8, N=5, topo="torus_nd", dims=[2, 2, 2]),
]


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("case", EXTREME, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_extreme_shapes_match_oracle(ddl, case, dtype):
    _check_exact(ddl, _w(dtype=dtype, **case))


@pytest.mark.parametrize("kernel", ["auto", "chunked"])
def test_largest_p_at_size_sampled(ddl, kernel):
    """P = 256 ranks of 4,000,003 fp32 elements (4.1 GB resident), multi-ring
    k = 8 in 3 MiB buckets: every rank pointer of the kernel's parameter
    block in use at size.  Sampled against the oracle's closed form (random
    and at every edge); all ranks identical."""
    w = _w(P=256, N=4_000_003, topo="multiring", k=8, bucket_bytes=3 << 20, seed=256)
    bufs = device_bufs_generated(w, DEV)
    with ddl.Plan.for_workload(w, kernel=kernel) as plan:
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        plan.check()
    for r in range(1, w.P):
        assert torch.equal(bufs[r].view(torch.int32), bufs[0].view(torch.int32)), r
    rng = np.random.default_rng(256)
    idx = np.unique(np.concatenate([rng.integers(0, w.N, 20_000), edge_samples(w)]))
    x_rows = np.stack([w.rank_values(r, idx.astype(np.uint64)) for r in range(w.P)], axis=1)
    want = oracle.closed_form(oracle_cfg(w), x_rows, idx.astype(np.uint64), w.scale)
    got = to_numpy_bits(bufs[0][torch.from_numpy(idx).to(DEV)])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {idx.size} sampled elements differ, e.g. idx {idx[bad[:5]]}"
    del bufs
    torch.cuda.empty_cache()


def test_more_than_2_32_elements_per_rank_sampled(ddl):
    """Element indices past 2^32: a 3-rank fp16 ring of 2^32 + 12,345 elements
    per rank (8.6 GB each) in 3 GiB buckets, so bucket and chunk edges and
    work-item starts lie above 2^32.  Sampled against the oracle's closed
    form (random, at every edge, and around 2^31 and 2^32); ranks identical."""
    w = _w(P=3, N=(1 << 32) + 12_345, dtype="f16", bucket_bytes=3 << 30)
    free, _ = torch.cuda.mem_get_info()
    if free < 3 * w.N * 2 + (4 << 30):
        pytest.skip("needs about 30 GB of free device memory")
    bufs = device_bufs_generated(w, DEV)
    with ddl.Plan.for_workload(w) as plan:
        assert plan.num_buckets == 3
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        plan.check()
    for r in range(1, w.P):
        assert torch.equal(bufs[r].view(torch.int16), bufs[0].view(torch.int16)), r
    rng = np.random.default_rng(32)
    near = np.concatenate([np.arange(b - 40, b + 40) for b in ((1 << 31), (1 << 32), w.N - 40)])
    idx = np.unique(np.concatenate([rng.integers(0, w.N, 60_000), edge_samples(w), near]))
    idx = idx[(idx >= 0) & (idx < w.N)]
    x_rows = np.stack([w.rank_values(r, idx.astype(np.uint64)) for r in range(w.P)], axis=1)
    want = oracle.closed_form(oracle_cfg(w), x_rows, idx.astype(np.uint64), w.scale)
    got = to_numpy_bits(bufs[0][torch.from_numpy(idx).to(DEV)])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {idx.size} sampled elements differ, e.g. idx {idx[bad[:5]]}"
    del bufs
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# Full-size workloads, in the configuration the bench times: every rank's
# buffer compared on sampled elements (random and at every chunk edge) with
# the oracle's closed form, and all ranks bitwise identical.
# ---------------------------------------------------------------------------

FULL = ["ring4_int", "torus4x4_resnet50", "torus8x4_resnet50_f16", "multiring64_resnet101", "ring16_lm300m",
        "multiring16_lm300m", "torus4x4_lm300m", "torus4x4x4_resnet101", "torus4x4x2_resnet50_f16"]


@pytest.mark.parametrize("kernel", ["auto", "bulkload", "chunked"])
@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled(ddl, name, kernel):
    w = synth.WORKLOADS[name]
    bufs = device_bufs_generated(w, DEV)
    with ddl.Plan.for_workload(w, kernel=kernel) as plan:
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        plan.check()
    for r in range(1, w.P):
        assert torch.equal(bufs[r].view(torch.int16 if w.dtype == "f16" else torch.int32),
                           bufs[0].view(torch.int16 if w.dtype == "f16" else torch.int32)), r
    rng = np.random.default_rng(2017)
    n_rand = w.N if w.N <= 65_536 else 60_000
    idx = np.arange(w.N) if n_rand == w.N else np.unique(np.concatenate(
        [rng.integers(0, w.N, n_rand), edge_samples(w)]))
    x_rows = np.stack([w.rank_values(r, idx.astype(np.uint64)) for r in range(w.P)], axis=1)
    want = oracle.closed_form(oracle_cfg(w), x_rows, idx.astype(np.uint64), w.scale)
    got = to_numpy_bits(bufs[0][torch.from_numpy(idx).to(DEV)])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {idx.size} sampled elements differ, e.g. idx {idx[bad[:5]]}"
    if name == "ring4_int":
        # integer inputs: the exact int64 total
        ints = np.stack([w.rank_values(r) for r in range(w.P)]).astype(np.int64).sum(axis=0)
        assert np.array_equal(to_numpy_bits(bufs[0]), ints.astype(np.float32))
    del bufs
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# Bucket scheduler, host-buffer path, launches, argument checks on the GPU
# ---------------------------------------------------------------------------

def test_overlap_with_backward_matches_allreduce(ddl):
    """Buckets signalled from a producer stream, reduced on the plan's side
    stream, in reverse-layer order: same bits as the oracle."""
    w = _w(P=8, N=400_000, layers=[50_000] * 8, bucket_bytes=300_000, seed=5)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    bufs = [torch.zeros(w.N, dtype=torch.float32, device=DEV) for _ in range(w.P)]
    src = device_bufs_from_host(host, DEV)
    torch.cuda.synchronize()
    main = torch.cuda.Stream()
    with ddl.Plan.for_workload(w) as plan:
        nb = plan.num_buckets
        assert nb == 4
        with torch.cuda.stream(main):
            plan.overlap_begin(bufs, w.scale, stream=main)
            for b in range(nb):                     # "back-propagation": output layers first
                lo, hi = plan.bucket_range(b)
                for r in range(w.P):
                    bufs[r][lo:hi].copy_(src[r][lo:hi])
                plan.bucket_ready(b, stream=main)
            plan.overlap_end(stream=main)
        main.synchronize()
        torch.cuda.synchronize()
        plan.check()
        assert plan.launches == nb
    for r in range(w.P):
        assert np.array_equal(to_numpy_bits(bufs[r]), ref[r])


@pytest.mark.parametrize("signalled", [[0, 2], [], [3], [1, 2]])
def test_overlap_end_reduces_buckets_never_signalled(ddl, signalled):
    """ddl_overlap_end all-reduces, on the producer stream, every bucket that
    was never signalled: the result is the oracle's whichever buckets were."""
    w = _w(P=6, N=240_001, topo="torus", X=3, Y=2, layers=[60_000] * 3 + [60_001], bucket_bytes=200_000, seed=8)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    bufs = [torch.zeros(w.N, dtype=torch.float32, device=DEV) for _ in range(w.P)]
    src = device_bufs_from_host(host, DEV)
    torch.cuda.synchronize()
    main = torch.cuda.Stream()
    with ddl.Plan.for_workload(w) as plan:
        assert plan.num_buckets == 4
        with torch.cuda.stream(main):
            plan.overlap_begin(bufs, w.scale, stream=main)
            for b in range(plan.num_buckets):
                lo, hi = plan.bucket_range(b)
                for r in range(w.P):
                    bufs[r][lo:hi].copy_(src[r][lo:hi])
                if b in signalled:
                    plan.bucket_ready(b, stream=main)
            if signalled:
                with pytest.raises(ddl.DDLError):     # a bucket is signalled once per begin/end pair
                    plan.bucket_ready(signalled[0], stream=main)
            plan.overlap_end(stream=main)
        main.synchronize()
        torch.cuda.synchronize()
        plan.check()
    for r in range(w.P):
        assert np.array_equal(to_numpy_bits(bufs[r]), ref[r]), r


@pytest.mark.parametrize("mode", ["fused", "rankorder", "stepwise"])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("topo", [dict(topo="multiring", k=3), dict(topo="torus", X=4, Y=2)])
def test_overlap_equals_allreduce_in_every_mode(ddl, mode, dtype, topo):
    """The bucket scheduler (side-stream launches, the rank-chunked pass where
    the plan's kernel choice allows) gives, in every mode and dtype, the bits
    the same plan's ddl_allreduce gives."""
    es = 2 if dtype == "f16" else 4
    w = _w(P=8, N=300_007, dtype=dtype, layers=[60_000, 90_007, 50_000, 100_000], bucket_bytes=60_000 * es,
           seed=13, **topo)
    host = _host_inputs(w)
    a = device_bufs_from_host(host, DEV)
    b = device_bufs_from_host(host, DEV)
    torch.cuda.synchronize()
    main = torch.cuda.Stream()
    with ddl.Plan.for_workload(w, mode=mode) as plan:
        assert plan.num_buckets >= 3
        plan.allreduce(a, w.scale)
        torch.cuda.synchronize()
        with torch.cuda.stream(main):
            plan.overlap_begin(b, w.scale, stream=main)
            for q in range(plan.num_buckets):
                plan.bucket_ready(q, stream=main)
            plan.overlap_end(stream=main)
        main.synchronize()
        torch.cuda.synchronize()
        plan.check()
    for r in range(w.P):
        assert np.array_equal(to_numpy_bits(b[r]), to_numpy_bits(a[r])), r
    if mode != "rankorder":
        ref = [h.copy() for h in host]
        oracle.emulate(oracle_cfg(w), ref, w.scale)
        assert np.array_equal(to_numpy_bits(b[0]), ref[0])


@pytest.mark.parametrize("name", ["multiring64_resnet101", "torus4x4x4_resnet101"])
def test_full_size_overlap_sampled(ddl, name):
    """The bucket scheduler at full size: the 7 ResNet-101 buckets written
    from a producer stream in reverse-layer order and each signalled as it
    completes, reduced on the plan's side stream.  Sampled against the
    oracle's closed form (random and at every edge); ranks identical."""
    w = synth.WORKLOADS[name]
    src = device_bufs_generated(w, DEV)
    bufs = [torch.zeros(w.N, dtype=torch_dtype(w.dtype), device=DEV) for _ in range(w.P)]
    torch.cuda.synchronize()
    main = torch.cuda.Stream()
    with ddl.Plan.for_workload(w) as plan:
        nb = plan.num_buckets
        assert nb == 7
        with torch.cuda.stream(main):
            plan.overlap_begin(bufs, w.scale, stream=main)
            for b in range(nb):
                lo, hi = plan.bucket_range(b)
                for r in range(w.P):
                    bufs[r][lo:hi].copy_(src[r][lo:hi])
                plan.bucket_ready(b, stream=main)
            plan.overlap_end(stream=main)
        main.synchronize()
        torch.cuda.synchronize()
        plan.check()
    del src
    view = torch.int16 if w.dtype == "f16" else torch.int32
    for r in range(1, w.P):
        assert torch.equal(bufs[r].view(view), bufs[0].view(view)), r
    rng = np.random.default_rng(7)
    idx = np.unique(np.concatenate([rng.integers(0, w.N, 20_000), edge_samples(w)]))
    x_rows = np.stack([w.rank_values(r, idx.astype(np.uint64)) for r in range(w.P)], axis=1)
    want = oracle.closed_form(oracle_cfg(w), x_rows, idx.astype(np.uint64), w.scale)
    got = to_numpy_bits(bufs[0][torch.from_numpy(idx).to(DEV)])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {idx.size} sampled elements differ, e.g. idx {idx[bad[:5]]}"
    del bufs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["torus4x4_resnet50", "torus8x4_resnet50_f16"])
def test_full_size_zero_copy_sampled(ddl, name):
    """The end-to-end form as the bench times it: full-size gradients in
    page-locked host memory, reduced in place over the host link (the
    bulk-load pass over its own work items).  Sampled against the oracle's
    closed form; every rank's host buffer identical."""
    w = synth.WORKLOADS[name]
    dev = device_bufs_generated(w, DEV)
    host = [torch.empty(w.N, dtype=torch_dtype(w.dtype), pin_memory=True) for _ in range(w.P)]
    for r in range(w.P):
        host[r].copy_(dev[r])
    del dev
    torch.cuda.synchronize()
    with ddl.Plan.for_workload(w) as plan:
        plan.allreduce_host(host, None, w.scale)
        torch.cuda.synchronize()
        plan.check()
    view = torch.int16 if w.dtype == "f16" else torch.int32
    for r in range(1, w.P):
        assert torch.equal(host[r].view(view), host[0].view(view)), r
    rng = np.random.default_rng(11)
    idx = np.unique(np.concatenate([rng.integers(0, w.N, 20_000), edge_samples(w)]))
    x_rows = np.stack([w.rank_values(r, idx.astype(np.uint64)) for r in range(w.P)], axis=1)
    want = oracle.closed_form(oracle_cfg(w), x_rows, idx.astype(np.uint64), w.scale)
    got = to_numpy_bits(host[0][torch.from_numpy(idx)])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {idx.size} sampled elements differ, e.g. idx {idx[bad[:5]]}"
    del host


def test_allreduce_host_buffers(ddl):
    w = _w(P=6, N=50_001, topo="torus", X=3, Y=2, seed=8)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    pinned = [torch.from_numpy(h.copy()).pin_memory() for h in host]
    dev = [torch.empty(w.N, dtype=torch.float32, device=DEV) for _ in range(w.P)]
    with ddl.Plan.for_workload(w) as plan:
        plan.allreduce_host(pinned, dev, w.scale)
        torch.cuda.synchronize()
    for r in range(w.P):
        assert np.array_equal(pinned[r].numpy(), ref[r])


@pytest.mark.parametrize("case", [
    dict(P=4, N=3_000_001, bucket_bytes=5_000_000),                       # 12 ranges over 3 buckets
    dict(P=8, N=2_500_003, dtype="f16", topo="torus", X=4, Y=2),          # 5 ranges
    dict(P=6, N=1_000_000, topo="multiring", k=2, mode="stepwise"),       # whole-bucket path
])
def test_allreduce_host_pipelined(ddl, case):
    case = dict(case)
    mode = case.pop("mode", "fused")
    w = _w(seed=21, **case)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    tdt = torch_dtype(w.dtype)
    pinned = [torch.from_numpy(h.view(np.int16) if w.dtype == "f16" else h.copy()).clone().pin_memory()
              for h in host]
    dev = [torch.empty(w.N, dtype=tdt, device=DEV) for _ in range(w.P)]
    with ddl.Plan.for_workload(w, mode=mode) as plan:
        plan.allreduce_host(pinned, dev, w.scale)
        torch.cuda.synchronize()
        plan.check()
    for r in range(w.P):
        got = pinned[r].numpy()
        got = got.view(np.uint16) if w.dtype == "f16" else got
        assert np.array_equal(got, ref[r]), r


ZERO_COPY = [
    dict(P=8, N=400_003, topo="torus", X=4, Y=2),
    dict(P=16, N=300_001, topo="multiring", k=2, bucket_bytes=400_000),
    dict(P=64, N=100_003),
    dict(P=65, N=50_001),
]


@pytest.mark.parametrize("kernel", ["auto", "ldg"])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("case", ZERO_COPY, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_allreduce_host_zero_copy(ddl, case, dtype, kernel):
    """dev_bufs = NULL: the fused pass works on page-locked host memory in
    place (by default through the bulk-load pass over its own work items, up
    to P = 64; the register pass with kernel "ldg" or beyond P = 64); twice, so
    the second call reuses the zero-copy tables."""
    w = _w(dtype=dtype, seed=31, **case)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    ref2 = [h.copy() for h in ref]
    oracle.emulate(oracle_cfg(w), ref2, w.scale)
    pinned = [torch.from_numpy(h.view(np.int16) if w.dtype == "f16" else h.copy()).clone().pin_memory()
              for h in host]
    with ddl.Plan.for_workload(w, kernel=kernel) as plan:
        for want in (ref, ref2):
            plan.allreduce_host(pinned, None, w.scale)
            torch.cuda.synchronize()
            plan.check()
            for r in range(w.P):
                got = pinned[r].numpy()
                got = got.view(np.uint16) if w.dtype == "f16" else got
                assert np.array_equal(got, want[r]), r
        # memory the GPU cannot reach is refused, unless the system gives it coherent access
        plain = [np.zeros(w.N, dtype=np.float32 if dtype == "f32" else np.uint16) for _ in range(w.P)]
        try:
            plan.allreduce_host([a.ctypes.data for a in plain], None, w.scale)
            torch.cuda.synchronize()
        except ddl.DDLError as e:
            assert e.status == ddl.DDL_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_allreduce_host_zero_copy_unaligned(ddl, dtype):
    """Page-locked host buffers that start one element past a 16-byte
    boundary: the zero-copy pass takes its element-wise path (the bulk copies
    need 16-byte alignment) and still matches the oracle bit for bit."""
    w = _w(P=8, N=60_001, dtype=dtype, topo="torus", X=4, Y=2, seed=61)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    big = [torch.zeros(w.N + 1, dtype=torch.int16 if dtype == "f16" else torch.float32).pin_memory()
           for _ in range(w.P)]
    views = []
    for b, h in zip(big, host):
        v = b[1:]
        v.copy_(torch.from_numpy(h.view(np.int16) if dtype == "f16" else h))
        views.append(v)
    with ddl.Plan.for_workload(w) as plan:
        plan.allreduce_host(views, None, w.scale)
        torch.cuda.synchronize()
        plan.check()
    for r in range(w.P):
        got = views[r].numpy()
        got = got.view(np.uint16) if dtype == "f16" else got
        assert np.array_equal(got, ref[r]), r


def test_zero_copy_tables_follow_plan_changes(ddl):
    """The zero-copy pass's own work items are rebuilt when the plan changes:
    zero-copy, then a layer list (new buckets), zero-copy again, then
    rank-order mode, then stepwise (refused); each result against the oracle
    (rank order against the fp64 sum), launches counted on the plan."""
    w = _w(P=16, N=200_003, topo="multiring", k=2, bucket_bytes=300_000, seed=77)

    def pinned_inputs(wk):
        host = _host_inputs(wk)
        return host, [torch.from_numpy(h.copy()).pin_memory() for h in host]

    with ddl.Plan.for_workload(w) as plan:
        w2 = w.with_(layers=(50_000, 3, 80_000, 70_000))
        for wk in (w, w2):
            if wk is w2:
                ddl.ddl_plan_set_layers(plan.handle, list(wk.layers))
            host, pinned = pinned_inputs(wk)
            before = plan.launches
            plan.allreduce_host(pinned, None, wk.scale)
            torch.cuda.synchronize()
            plan.check()
            assert plan.launches - before == plan.num_buckets
            ref = [h.copy() for h in host]
            oracle.emulate(oracle_cfg(wk), ref, wk.scale)
            for r in range(wk.P):
                assert np.array_equal(pinned[r].numpy(), ref[r]), (wk.layers, r)
        plan.set_mode("rankorder")
        host, pinned = pinned_inputs(w2)
        plan.allreduce_host(pinned, None, w2.scale)
        torch.cuda.synchronize()
        ref = oracle.ref64(host, w2.scale, "f32")
        got = pinned[0].numpy().astype(np.float64)
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-6
        plan.set_mode("stepwise")
        with pytest.raises(ddl.DDLError) as ei:
            plan.allreduce_host(pinned, None, w2.scale)
        assert ei.value.status == ddl.DDL_ERR_UNSUPPORTED


@pytest.mark.parametrize("case", [dict(P=16, N=300_001, topo="torus", X=4, Y=4),
                                  dict(P=8, N=200_003, topo="torus_nd", dims=[2, 2, 2], dtype="f16"),
                                  dict(P=16, N=250_001, topo="multiring", k=2, bucket_bytes=300_000),
                                  dict(P=6, N=100_003, topo="torus", X=3, Y=2, mode="stepwise")],
                         ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_back_to_back_calls_and_producer_kernels(ddl, case):
    """Passes launched as programmatic dependents must still see every write
    of the kernel before them: three all-reduces queued back to back, with a
    torch kernel that rewrites every rank buffer (x -> 2x - 1, exact here)
    before the second, and no synchronisation between any of them."""
    case = dict(case)
    mode = case.pop("mode", "fused")
    w = _w(seed=88, **case)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    cfg = oracle_cfg(w)
    oracle.emulate(cfg, ref, w.scale)
    if w.dtype == "f16":
        ref = [oracle.f32_to_f16(2.0 * oracle.f16_to_f32(r) - 1.0) for r in ref]
    else:
        ref = [(np.float32(2.0) * r - np.float32(1.0)).astype(np.float32) for r in ref]
    oracle.emulate(cfg, ref, w.scale)
    oracle.emulate(cfg, ref, w.scale)
    bufs = device_bufs_from_host(host, DEV)
    torch.cuda.synchronize()
    with ddl.Plan.for_workload(w, mode=mode) as plan:
        plan.allreduce(bufs, w.scale)
        for b in bufs:
            b.mul_(2).sub_(1)
        plan.allreduce(bufs, w.scale)
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        plan.check()
    for r in range(w.P):
        assert np.array_equal(to_numpy_bits(bufs[r]), ref[r]), r


def test_two_plans_on_two_streams_concurrently(ddl):
    """Two plans (different schedules and dtypes) queued on two streams with no
    ordering between them, each on its own buffers: both results match the
    oracle (the plans share nothing on the device)."""
    wa = _w(P=16, N=300_001, topo="torus", X=4, Y=4, seed=71)
    wb = _w(P=12, N=250_003, dtype="f16", topo="multiring", k=2, bucket_bytes=200_000, seed=72)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    out = []
    with ddl.Plan.for_workload(wa) as pa, ddl.Plan.for_workload(wb) as pb:
        for w in (wa, wb):
            host = _host_inputs(w)
            ref = [h.copy() for h in host]
            oracle.emulate(oracle_cfg(w), ref, w.scale)
            out.append((w, device_bufs_from_host(host, DEV), ref))
        torch.cuda.synchronize()
        for _ in range(3):   # three rounds each, interleaved on the host, unordered on the GPU
            pa.allreduce(out[0][1], wa.scale, stream=sa)
            pb.allreduce(out[1][1], wb.scale, stream=sb)
        torch.cuda.synchronize()
        pa.check()
        pb.check()
    for w, bufs, ref in out:
        ref3 = [r.copy() for r in ref]
        oracle.emulate(oracle_cfg(w), ref3, w.scale)
        oracle.emulate(oracle_cfg(w), ref3, w.scale)
        for r in range(w.P):
            assert np.array_equal(to_numpy_bits(bufs[r]), ref3[r]), (w.topo, r)


def test_plans_driven_from_several_host_threads(ddl):
    """Four host threads, each creating its own plan and stream and running
    five all-reduces on its own buffers, all at once (the binding releases the
    interpreter lock during library calls).  The plans cover the register
    pass, the small-item pass and the latency pass (P >= 32, the first launch
    of it on the device among them), so the library's per-device launch
    caches are filled concurrently.  Every result matches five applications of
    the oracle."""
    import threading
    ws = [_w(P=16, N=300_001, topo="torus", X=4, Y=4, seed=81),
          _w(P=32, N=16_384, dtype="f16", topo="torus", X=8, Y=4, seed=82),
          _w(P=64, N=9_001, topo="multiring", k=4, seed=83),
          _w(P=4, N=65_536, dist="int1000", scale=1.0, seed=84)]
    reps = 5
    inputs = [_host_inputs(w) for w in ws]
    bufs = [device_bufs_from_host(h, DEV) for h in inputs]
    torch.cuda.synchronize()
    errors = [None] * len(ws)
    start = threading.Barrier(len(ws))

    def run(i):
        try:
            s = torch.cuda.Stream(DEV)
            s.wait_stream(torch.cuda.default_stream(DEV))
            with ddl.Plan.for_workload(ws[i]) as plan:
                start.wait(timeout=60)
                for _ in range(reps):
                    plan.allreduce(bufs[i], ws[i].scale, stream=s)
                s.synchronize()
                plan.check()
        except BaseException as e:  # reported on the main thread
            errors[i] = e
            start.abort()  # the others stop waiting at the barrier

    threads = [threading.Thread(target=run, args=(i,), daemon=True) for i in range(len(ws))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    for e in errors:
        if e is not None:
            raise e
    for w, host, got in zip(ws, inputs, bufs):
        ref = [h.copy() for h in host]
        for _ in range(reps):
            oracle.emulate(oracle_cfg(w), ref, w.scale)
        for r in range(w.P):
            assert np.array_equal(to_numpy_bits(got[r]), ref[r]), (w.topo, w.P, r)


def test_allreduce_captured_in_cuda_graph(ddl):
    """After a first (uploading) call, ddl_allreduce can be captured in a CUDA
    graph; each replay reduces whatever the buffers hold at that time."""
    w = _w(P=16, N=77_777, topo="torus", X=4, Y=4, bucket_bytes=100_000, seed=51)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    bufs = device_bufs_from_host(host, DEV)
    src = [b.clone() for b in bufs]
    with ddl.Plan.for_workload(w) as plan:
        plan.allreduce(bufs, w.scale)          # uploads the tables, outside the capture
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            plan.allreduce(bufs, w.scale, s)
        for _ in range(2):                     # replay twice on fresh inputs
            for b, x in zip(bufs, src):
                b.copy_(x)
            g.replay()
            torch.cuda.synchronize()
            for r in range(w.P):
                assert np.array_equal(to_numpy_bits(bufs[r]), ref[r]), r


@pytest.mark.parametrize("case", [dict(P=32, N=16_385, topo="torus", X=8, Y=4, dtype="f16"),
                                  dict(P=16, N=300_001, topo="torus", X=4, Y=4)],
                         ids=["staged-f16", "register-f32"])
def test_allreduce_sgd_captured_in_cuda_graph(ddl, case):
    """The fused all-reduce + momentum SGD captured in a CUDA graph (after a
    first call outside the capture): three replays equal three updates of the
    oracle, each on the gradients the buffers hold at that replay."""
    w = _w(seed=53, **case)
    host = _host_inputs(w)
    rng = np.random.default_rng(9)
    p0 = rng.standard_normal(w.N).astype(np.float32)
    v0 = (rng.standard_normal(w.N) * 0.1).astype(np.float32)
    lr, mu, wd = 0.05, 0.9, 1e-4
    p_ref = [p0.copy() for _ in range(w.P)]
    m_ref = [v0.copy() for _ in range(w.P)]
    grads = device_bufs_from_host(host, DEV)
    src = [g.clone() for g in grads]
    params = [torch.from_numpy(p0).to(DEV) for _ in range(w.P)]
    moms = [torch.from_numpy(v0).to(DEV) for _ in range(w.P)]
    with ddl.Plan.for_workload(w) as plan:
        g_ref = [h.copy() for h in host]
        oracle.sgd(oracle_cfg(w), g_ref, p_ref, m_ref, w.scale, lr, mu, wd)
        plan.allreduce_sgd(grads, params, moms, w.scale, lr, mu, wd)   # uploads, outside the capture
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            plan.allreduce_sgd(grads, params, moms, w.scale, lr, mu, wd, stream=s)
        for _ in range(3):
            for b, x in zip(grads, src):
                b.copy_(x)
            g_ref = [h.copy() for h in host]
            oracle.sgd(oracle_cfg(w), g_ref, p_ref, m_ref, w.scale, lr, mu, wd)
            graph.replay()
            torch.cuda.synchronize()
        plan.check()
    for r in range(w.P):
        assert np.array_equal(params[r].cpu().numpy(), p_ref[r]), ("params", r)
        assert np.array_equal(moms[r].cpu().numpy(), m_ref[r]), ("moms", r)
        assert np.array_equal(to_numpy_bits(grads[r]), g_ref[r]), ("grads", r)


def test_bounded_wait_timeout_is_reported_and_context_survives(ddl):
    """A wait that runs out (an mbarrier nothing arrives at, 50 ms limit)
    sets the error word; ddl_plan_check reports DDL_ERR_DEVICE_CHECK once,
    and the next all-reduce on the same context is still bit-exact."""
    w = _w(P=4, N=20_001, seed=61)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    with ddl.Plan.for_workload(w, kernel="bulkload") as plan:
        assert ddl.ddl_plan_check(plan.handle) == ddl.DDL_OK
        ddl.ddl_selftest_wait_timeout(plan.handle, 50_000)
        assert ddl.ddl_plan_check(plan.handle) == ddl.DDL_ERR_DEVICE_CHECK
        assert ddl.ddl_plan_check(plan.handle) == ddl.DDL_OK        # the word was cleared
        bufs = device_bufs_from_host(host, DEV)
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        assert ddl.ddl_plan_check(plan.handle) == ddl.DDL_OK
        for r in range(w.P):
            assert np.array_equal(to_numpy_bits(bufs[r]), ref[r])
        with pytest.raises(ddl.DDLError):
            ddl.ddl_selftest_wait_timeout(plan.handle, 0)


def test_injected_allocation_failure_returns_oom_and_the_plan_recovers(ddl, monkeypatch):
    """Host-side fault injection: with DDL_INJECT_ALLOC_FAILURE=1 the upload
    of the plan's device tables fails as if the device were out of memory.
    The all-reduce returns DDL_ERR_OOM and touches no buffer; once the
    variable is gone the same plan uploads its tables and is bit-exact."""
    w = _w(P=5, N=30_011, topo="multiring", k=2, seed=17)
    host = _host_inputs(w)
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    bufs = device_bufs_from_host(host, DEV)
    with ddl.Plan.for_workload(w) as plan:
        monkeypatch.setenv("DDL_INJECT_ALLOC_FAILURE", "1")
        with pytest.raises(ddl.DDLError) as ei:
            plan.allreduce(bufs, w.scale)
        assert ei.value.status == ddl.DDL_ERR_OOM
        torch.cuda.synchronize()
        for r in range(w.P):
            assert np.array_equal(to_numpy_bits(bufs[r]), host[r]), r   # nothing ran
        monkeypatch.delenv("DDL_INJECT_ALLOC_FAILURE")
        plan.allreduce(bufs, w.scale)
        torch.cuda.synchronize()
        plan.check()
    for r in range(w.P):
        assert np.array_equal(to_numpy_bits(bufs[r]), ref[r]), r


def test_launch_counts_and_checks(ddl):
    w = _w(P=16, N=100_000, topo="torus", X=4, Y=4, bucket_bytes=100_000)
    bufs = device_bufs_generated(w, DEV)
    with ddl.Plan.for_workload(w) as plan:
        nb = plan.num_buckets
        assert nb > 1
        plan.allreduce(bufs, w.scale)
        assert plan.launches == 1                      # every bucket in one fused launch
        for b in range(nb):
            plan.allreduce_bucket(b, bufs, w.scale)
        assert plan.launches == 1 + nb
        plan.set_mode("stepwise")
        plan.allreduce(bufs, w.scale)
        assert plan.launches == 1 + nb + nb * (2 * 3 + 2 * 3)
        torch.cuda.synchronize()
        plan.check()
        # a host pointer is not device memory: refused before any launch
        host = [np.zeros(w.N, dtype=np.float32) for _ in range(w.P)]
        with pytest.raises(ddl.DDLError) as ei:
            plan.allreduce([h.ctypes.data for h in host], w.scale)
        assert ei.value.status == ddl.DDL_ERR_INVALID_ARG
        # overlapping views of one tensor are refused
        big = torch.zeros(w.N * w.P, device=DEV)
        views = [big[i * (w.N - 1): i * (w.N - 1) + w.N] for i in range(w.P)]
        with pytest.raises(ddl.DDLError):
            plan.allreduce(views, w.scale)
