"""Randomised problems on the GPU, compared with the oracle.

test_random_problem_matches_oracle: small problems of every schedule, each
through the fused pass (a random kernel variant), the stepwise mode and the
zero-copy pass over page-locked host memory, bit for bit against the oracle's
step emulation.

test_random_entry_point_matches_oracle: each seed draws one problem -- P
(1..256), N (1 .. a few million elements in all), the schedule (ring,
multi-ring, 2D torus, n-D torus), the dtype, the mode, buckets or a layer
list, the kernel choice -- and the entry point that runs it: a plan's
all-reduce (aligned or misaligned rank buffers), the per-bucket call in a
random bucket order, the bucket scheduler with a random subset of buckets
signalled, the allocation-free entry point, or the zero-copy pass over
page-locked host memory.  Schedule-order modes must equal the oracle's step
emulation bit for bit; the rank-order mode must be within the element-wise
bound of a P-term binary32 left fold (plus one binary16 rounding for fp16)
with every rank identical.  The draws span the small-item, latency and
register passes and ragged tails; a fixed seed keeps each case reproducible.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from gpu_util import device_bufs_from_host, oracle_cfg, rankorder_margins, to_numpy_bits, torch_dtype
from test_random_tables import _random_problem

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
MAX_ELEMS = 8_000_000  # P * N of one case (32 MB of fp32 per copy)


@pytest.fixture(scope="module")
def ddl():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    from gradient_all_reduce_ddl_gb300 import ddl as mod
    return mod


@pytest.mark.parametrize("seed", range(32))
def test_random_problem_matches_oracle(ddl, seed):
    rng = np.random.default_rng(5000 + seed)
    kw = _random_problem(rng)
    kw["N"] = int(kw["N"]) * int(rng.integers(1, 12))      # up to ~30K elements: several tiles
    if "layers" in kw:
        kw["layers"] = kw["layers"][:-1] + [kw["layers"][-1] + kw["N"] - sum(kw["layers"])]
    w = synth.Workload(name="rand", P=kw["P"], N=kw["N"], dtype=kw["dtype"], topo=kw["topo"], k=kw.get("k", 1),
                       X=kw.get("X", 0), Y=kw.get("Y", 0), bucket_bytes=kw.get("bucket_bytes", 0),
                       layers=None if "layers" not in kw else tuple(kw["layers"]),
                       dims=None if "dims" not in kw else tuple(kw["dims"]),
                       scale=float(np.float32(1.0 / kw["P"])), sigma=1e-2 if kw["dtype"] == "f16" else 1e-3,
                       seed=seed)
    host = [w.rank_values(r) for r in range(w.P)]
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    kernel = str(rng.choice(["ldg", "bulkload", "chunked"]))
    for mode in ("fused", "stepwise"):
        bufs = device_bufs_from_host(host, "cuda:0")
        with ddl.Plan.for_workload(w, mode=mode, kernel=kernel if mode == "fused" else "auto") as plan:
            plan.allreduce(bufs, w.scale)
            torch.cuda.synchronize()
            plan.check()
        for r in range(w.P):
            assert np.array_equal(to_numpy_bits(bufs[r]), ref[r]), (kw, mode, kernel, r)
    pinned = [torch.from_numpy(h.view(np.int16) if w.dtype == "f16" else h.copy()).clone().pin_memory()
              for h in host]
    with ddl.Plan.for_workload(w) as plan:
        plan.allreduce_host(pinned, None, w.scale)
        torch.cuda.synchronize()
        plan.check()
    for r in range(w.P):
        got = pinned[r].numpy()
        got = got.view(np.uint16) if w.dtype == "f16" else got
        assert np.array_equal(got, ref[r]), (kw, "zero-copy", r)


def _divisors(n):
    return [d for d in range(1, n + 1) if n % d == 0]


def _draw_P(rng):
    r = rng.random()
    if r < 0.45:
        return int(rng.integers(1, 17))
    if r < 0.75:
        return int(rng.integers(17, 97))
    if r < 0.85:
        return int(rng.integers(97, 257))
    return int(rng.choice([32, 64, 128, 256]))


def _draw_N(rng, P):
    hi = max(2, min(400_000, MAX_ELEMS // P))
    if rng.random() < 0.35:  # several work items per rank
        return int(rng.integers(max(1, hi // 8), hi + 1))
    return int(math.exp(rng.uniform(0.0, math.log(hi))))  # down to a handful of elements


def random_case(seed):
    """One random problem and how to run it (plain data: the test runs it)."""
    rng = np.random.default_rng(77_000 + seed)
    P = _draw_P(rng)
    N = _draw_N(rng, P)
    dtype = "f16" if rng.random() < 0.4 else "f32"
    es = 2 if dtype == "f16" else 4
    topo = str(rng.choice(["ring", "multiring", "torus", "torus_nd"]))
    w = dict(P=P, N=N, dtype=dtype, topo=topo, k=1, X=0, Y=0, dims=None, bucket_bytes=0, layers=None)
    if topo == "multiring":
        phi = sum(1 for c in range(1, P) if math.gcd(c, P) == 1) if P > 1 else 1
        w["k"] = int(rng.integers(1, min(phi, 8) + 1))
    elif topo == "torus":
        X = int(rng.choice(_divisors(P)))
        w.update(X=X, Y=P // X)
    elif topo == "torus_nd":
        dims, rest = [], P
        for _ in range(int(rng.integers(1, 4))):
            d = int(rng.choice(_divisors(rest)))
            dims.append(d)
            rest //= d
        dims.append(rest)
        w["dims"] = tuple(dims)
    r = rng.random()
    if r < 0.3:
        w["bucket_bytes"] = int(rng.integers(es, es * N + 64))
    elif r < 0.5 and N > 1:
        n_cut = min(N - 1, int(rng.integers(0, 12)))
        cuts = np.sort(rng.choice(np.arange(1, N), size=n_cut, replace=False)) if n_cut else np.array([], int)
        edges = np.concatenate([[0], cuts, [N]]).astype(np.int64)
        w["layers"] = tuple(int(b - a) for a, b in zip(edges[:-1], edges[1:]))
        w["bucket_bytes"] = int(rng.integers(1, N + 2)) * es
    mode = str(rng.choice(["fused", "stepwise", "rankorder"], p=[0.6, 0.2, 0.2]))
    kernel = str(rng.choice(["auto", "ldg", "bulkload", "chunked"], p=[0.55, 0.15, 0.15, 0.15]))
    entries = ["plan", "misaligned", "buckets", "overlap"]
    if mode == "fused" and topo != "torus_nd" and kernel == "auto":
        entries.append("noalloc")
    if mode != "stepwise" and P * N * es <= (64 << 20):
        entries.append("host")
    entry = str(rng.choice(entries))
    if dtype == "f32" and rng.random() < 0.2:
        dist, sigma, scale = "int1000", 1.0, 1.0
    else:
        dist, sigma = "normal", (1e-2 if dtype == "f16" else 1e-3)
        scale = float(np.float32(1.0 / P)) if rng.random() < 0.7 else float(np.float32(rng.uniform(0.01, 2.0)))
    return dict(w=w, mode=mode, kernel=kernel, entry=entry, dist=dist, sigma=sigma, scale=scale,
                misalign=int(rng.integers(1, 4)), order_seed=int(rng.integers(0, 2**31)), seed=seed)


def _workload(c):
    w = c["w"]
    return synth.Workload(name=f"rand{c['seed']}", P=w["P"], N=w["N"], dtype=w["dtype"], topo=w["topo"], k=w["k"],
                          X=w["X"], Y=w["Y"], bucket_bytes=w["bucket_bytes"], layers=w["layers"], dims=w["dims"],
                          scale=c["scale"], dist=c["dist"], sigma=c["sigma"], seed=5000 + c["seed"])


def _run(ddl, c, w, host):
    """Runs the case's entry point; returns the P results in storage form."""
    entry, rng = c["entry"], np.random.default_rng(c["order_seed"])
    if entry == "host":
        pinned = [torch.from_numpy(h.view(np.int16) if w.dtype == "f16" else h).pin_memory() for h in host]
        with ddl.Plan.for_workload(w, mode=c["mode"], kernel=c["kernel"]) as plan:
            plan.allreduce_host(pinned, None, w.scale)
            torch.cuda.synchronize()
            plan.check()
        return [p.numpy().view(np.uint16) if w.dtype == "f16" else p.numpy() for p in pinned]
    if entry == "misaligned":
        bufs = []
        for h in host:
            big = torch.zeros(w.N + c["misalign"], dtype=torch_dtype(w.dtype), device=DEV)
            big[c["misalign"]:] = device_bufs_from_host([h], DEV)[0]
            bufs.append(big[c["misalign"]:])
    else:
        bufs = device_bufs_from_host(host, DEV)
    if entry == "noalloc":
        topo = ddl.ddl_topology_t({"ring": ddl.DDL_RING, "multiring": ddl.DDL_MULTIRING,
                                   "torus": ddl.DDL_TORUS}[w.topo], w.k, w.X, w.Y)
        try:
            ddl.ddl_allreduce_noalloc(w.P, w.N, ddl.DTYPES[w.dtype], topo, w.bucket_bytes,
                                      list(w.layers) if w.layers else None, bufs, w.scale)
        except ddl.DDLError as e:
            # tables larger than the static array are refused before any work
            assert e.status == ddl.DDL_ERR_UNSUPPORTED, e
            entry = "plan"
        else:
            torch.cuda.synchronize()
            ddl.ddl_noalloc_check()
            return [to_numpy_bits(b) for b in bufs]
    with ddl.Plan.for_workload(w, mode=c["mode"], kernel=c["kernel"]) as plan:
        if entry in ("plan", "misaligned"):
            plan.allreduce(bufs, w.scale)
        elif entry == "buckets":
            for b in rng.permutation(plan.num_buckets):
                plan.allreduce_bucket(int(b), bufs, w.scale)
        elif entry == "overlap":
            nb = plan.num_buckets
            signalled = sorted(int(b) for b in rng.choice(nb, size=int(rng.integers(0, nb + 1)), replace=False))
            side = torch.cuda.Stream(DEV)
            side.wait_stream(torch.cuda.current_stream(DEV))
            with torch.cuda.stream(side):
                plan.overlap_begin(bufs, w.scale, stream=side)
                for b in signalled:
                    plan.bucket_ready(b, stream=side)
                plan.overlap_end(stream=side)
            side.synchronize()
        torch.cuda.synchronize()
        plan.check()
    return [to_numpy_bits(b) for b in bufs]


CASES = [random_case(s) for s in range(256)]


def _case_id(c):
    w = c["w"]
    shape = {"multiring": f"k{w['k']}", "torus": f"{w['X']}x{w['Y']}",
             "torus_nd": "x".join(map(str, w["dims"] or ()))}.get(w["topo"], "")
    extra = "-layers" if w["layers"] else ("-b" if w["bucket_bytes"] else "")
    return f"{c['seed']}-P{w['P']}-N{w['N']}-{w['topo']}{shape}-{w['dtype']}-{c['mode']}-{c['kernel']}-" \
           f"{c['entry']}{extra}"


@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_random_entry_point_matches_oracle(ddl, case):
    w = _workload(case)
    host = [w.rank_values(r) for r in range(w.P)]
    got = _run(ddl, case, w, host)
    if case["mode"] == "rankorder":
        norm, elem = rankorder_margins(host, got[0], w.scale, w.dtype)
        assert elem <= 1.0, (elem, norm)
        for r in range(1, w.P):
            assert np.array_equal(got[r], got[0]), f"rank {r} differs from rank 0"
        return
    ref = [h.copy() for h in host]
    oracle.emulate(oracle_cfg(w), ref, w.scale)
    for r in range(w.P):
        if not np.array_equal(got[r], ref[r]):
            bad = np.nonzero(got[r] != ref[r])[0]
            raise AssertionError(f"rank {r}: {bad.size} elements differ, first at {bad[:8]}")


def test_random_draws_cover_every_path():
    """The fixed draw reaches every schedule, mode, kernel choice and entry
    point, and both dtypes, buckets and layer lists, P >= 32 and P = 1."""
    seen = lambda f: {f(c) for c in CASES}  # noqa: E731
    assert seen(lambda c: c["w"]["topo"]) == {"ring", "multiring", "torus", "torus_nd"}
    assert seen(lambda c: c["mode"]) == {"fused", "stepwise", "rankorder"}
    assert seen(lambda c: c["kernel"]) == {"auto", "ldg", "bulkload", "chunked"}
    assert seen(lambda c: c["entry"]) == {"plan", "misaligned", "buckets", "overlap", "noalloc", "host"}
    assert seen(lambda c: c["w"]["dtype"]) == {"f32", "f16"}
    assert any(c["w"]["layers"] for c in CASES) and any(c["w"]["bucket_bytes"] and not c["w"]["layers"]
                                                          for c in CASES)
    assert any(c["w"]["P"] >= 32 for c in CASES) and any(c["w"]["P"] > 128 for c in CASES)
