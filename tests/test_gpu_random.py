"""Randomised small problems on the GPU, every schedule: the fused pass (a
random kernel variant), the stepwise mode and the zero-copy pass over
page-locked host memory must match the oracle's step emulation bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import device_bufs_from_host, oracle_cfg, to_numpy_bits
from test_random_tables import _random_problem

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


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
