"""Randomised problems: the library's host tables (buckets, fold orders,
traffic, cost) against the oracle's, over every schedule, dtype and bucket
rule.  A fixed seed keeps the draw reproducible."""
import math

import numpy as np
import pytest

import oracle


def _random_problem(rng):
    P = int(rng.integers(1, 41))
    N = int(rng.integers(1, 2500))
    dtype = "f16" if rng.random() < 0.4 else "f32"
    kind = rng.choice(["ring", "multiring", "torus", "torus_nd"])
    kw = dict(P=P, N=N, dtype=dtype, topo=str(kind))
    if kind == "multiring":
        phi = sum(1 for c in range(1, P) if math.gcd(c, P) == 1) if P > 1 else 1
        kw["k"] = int(rng.integers(1, phi + 1))
    elif kind == "torus":
        divs = [d for d in range(1, P + 1) if P % d == 0]
        X = int(rng.choice(divs))
        kw.update(X=X, Y=P // X)
    elif kind == "torus_nd":
        dims, rest = [], P
        for _ in range(int(rng.integers(1, 4))):
            divs = [d for d in range(1, rest + 1) if rest % d == 0]
            d = int(rng.choice(divs))
            dims.append(d)
            rest //= d
        dims.append(rest)
        kw["dims"] = dims
    r = rng.random()
    if r < 0.3:
        kw["bucket_bytes"] = int(rng.integers(2, 4 * N + 8))
    elif r < 0.5:
        cuts = np.sort(rng.choice(np.arange(1, N), size=min(N - 1, int(rng.integers(0, 6))), replace=False)) \
            if N > 1 else np.array([], dtype=int)
        edges = np.concatenate([[0], cuts, [N]]).astype(int)
        kw["layers"] = [int(b - a) for a, b in zip(edges[:-1], edges[1:])]
        kw["bucket_bytes"] = int(rng.integers(1, 2 * N + 4)) * (2 if dtype == "f16" else 4)
    return kw


@pytest.mark.parametrize("seed", range(40))
def test_random_problem_tables_match_oracle(seed):
    from gradient_all_reduce_ddl_gb300.build import build
    build()
    from gradient_all_reduce_ddl_gb300 import ddl
    rng = np.random.default_rng(1000 + seed)
    kw = _random_problem(rng)
    cfg = oracle.Config(**kw)
    with ddl.Plan(**kw) as plan:
        assert plan.buckets() == oracle.buckets(cfg)
        assert plan.traffic() == oracle.traffic(cfg)
        links = int(rng.integers(1, 5))
        assert plan.cost(3e-6, 1e-10, links) == pytest.approx(oracle.cost(cfg, 3e-6, 1e-10, links), rel=1e-12,
                                                              abs=1e-18)
        for i in range(0, kw["N"], max(1, kw["N"] // 300)):
            o, inner, groups = oracle.fold_order(cfg, i)
            got = plan.fold_order(i)
            assert got[0] == o.tolist(), (kw, i)
            if kw["topo"] != "torus_nd":
                assert got[1:] == (inner, groups)


KERNEL_NAMES = {"fold_ldg_kernel", "fold_small_kernel", "fold_lat_kernel", "fold_lat_kernel (one group)",
                "fold_nd_kernel", "fold_nd_h2_kernel", "fold_lat_nd_kernel", "fold_bulk_kernel", "fold_chunked_kernel",
                "step_kernel"}


@pytest.mark.parametrize("seed", range(40))
def test_random_problem_kernel_name(seed):
    """ddl_plan_kernel_name answers for every drawn shape, mode and kernel
    choice with one of the library's passes, consistent with the plan's mode
    and choice (host-only)."""
    from gradient_all_reduce_ddl_gb300.build import build
    build()
    from gradient_all_reduce_ddl_gb300 import ddl
    rng = np.random.default_rng(3000 + seed)
    kw = _random_problem(rng)
    kw["N"] = int(kw["N"]) * int(rng.integers(1, 400))       # up to ~1M elements: every item size
    if "layers" in kw:
        kw["layers"] = kw["layers"][:-1] + [kw["layers"][-1] + kw["N"] - sum(kw["layers"])]
    mode = str(rng.choice(["fused", "stepwise", "rankorder"]))
    kernel = str(rng.choice(["auto", "ldg", "bulkload", "chunked"]))
    with ddl.Plan(mode=mode, kernel=kernel, **kw) as plan:
        name = plan.kernel_name
    assert name in KERNEL_NAMES, name
    if mode == "stepwise":
        assert name == "step_kernel"
    elif kw["topo"] == "torus_nd" and mode == "fused":
        assert name in {"fold_nd_kernel", "fold_nd_h2_kernel", "fold_lat_nd_kernel"}
    elif kernel in ("bulkload", "chunked"):
        assert name == {"bulkload": "fold_bulk_kernel", "chunked": "fold_chunked_kernel"}[kernel]
    else:
        assert name in {"fold_ldg_kernel", "fold_small_kernel", "fold_lat_kernel", "fold_lat_kernel (one group)"}
