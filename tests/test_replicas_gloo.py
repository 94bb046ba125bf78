"""The N > 1 path of bench.py (one replica per GPU, no collective on the data
path) on CPU: two gloo ranks agree on the slowest replica's time, the job
throughput counts every replica, and only rank 0 of the reference arm works."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    local_ms = [2.0, 3.5][rank]
    ms = bench.reduce_max(local_ms, ws)
    dist.barrier()
    q.put((r, ws, local, ms, bench.job_gbs(1_000_000_000, ws, ms)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica():
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[:3] for o in out] == [(0, 2, 0), (1, 2, 1)]
    for o in out:
        assert o[3] == 3.5                      # the slowest replica's time
        assert o[4] == pytest.approx(2e9 / 3.5e-3 / 1e9)   # both replicas' bytes


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.25, 1) == 1.25
    assert bench.job_gbs(3_271_300_096, 1, 0.475) == pytest.approx(6886.9, rel=1e-3)


def _short_rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), LOCAL_WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank 0 sees too little host memory for two replicas' buffers, rank 1 plenty
    avail = [30 << 30, 1 << 40][rank]
    why = bench.host_memory_short(20 << 30, world, avail=avail)
    both_ok = bench.host_memory_short(1 << 30, world, avail=avail)
    q.put((rank, why, both_ok))
    dist.destroy_process_group()


def test_e2e_memory_decision_is_the_same_on_every_rank():
    """A replica short of host memory for the end-to-end leg makes every
    replica skip it (a rank that ran it alone would wait forever in the
    max-over-ranks timing); when all have room, none skips."""
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_short_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0][1].startswith("host memory: ") and out[1][1] == "host memory short on another rank"
    assert out[0][2] is None and out[1][2] is None
