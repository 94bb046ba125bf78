"""Benchmark of the fused gradient all-reduce on one GB300 (or N replicas).

Metric: all-reduce GB/s on the algorithmic minimum of HBM traffic, 2*P*N*e
bytes per all-reduce (every rank element read once and written once), plus
elements/s, per schedule; and the fraction of the measured HBM copy bandwidth.

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--mode fused|stepwise|rankorder]
                    [--kernel auto|ldg|bulk] [--impl ours|reference] [--no-e2e] [--no-cpu]

A "step" is one ddl_allreduce of the whole gradient (every bucket).  The
default workload is the 4x4 2D-torus all-reduce of a ResNet-50 gradient
(P=16 ranks x 25,557,032 fp32, scale 1/16; 1.64 GB resident, well above the
129 MB L2, so every step streams from HBM).  With --gpus N > 1 (torchrun) the
path does not shard: each GPU runs an independent replica, and the reported
value is the total over all replicas.  --impl reference times the oracle (the
plain single-threaded CPU emulation) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "all-reduce GB/s and elems/s per schedule on 1 GB300; % of HBM roofline"
DEFAULT_WORKLOAD = "torus4x4_resnet50"

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the fused kernel,
# from one ncu capture, keyed by (workload, kernel variant, sha256[:16] of the
# kernel source it was taken on).  A changed kernel reports null.
NCU_TRAFFIC = {
    ("torus4x4_resnet50", "ldg", "0e52a75d29912526"): 1_635_956_224 + 1_575_996_160,
    ("torus4x4_resnet50", "ldg", "114f33c52577cd67"): 1_635_897_344 + 1_575_593_472,
    ("torus4x4_resnet50", "ldg", "316feed84c50fe44"): 1_636_111_360 + 1_575_655_424,
    ("torus4x4_resnet50", "ldg", "2e312619baf89fcd"): 1_636_190_976 + 1_575_729_664,
    ("torus4x4_resnet50", "ldg", "2c4e6c02dcdb9dcd"): 1_635_898_368 + 1_576_063_744,
    ("torus4x4_resnet50", "ldg", "8b82de61611a4d5b"): 1_635_897_088 + 1_575_497_728,
    ("torus4x4_resnet50", "ldg", "11c73895f5e07e69"): 1_635_897_344 + 1_575_480_064,
    ("torus4x4_resnet50", "ldg", "fcb0b1da26b97bdc"): 1_635_928_320 + 1_575_545_600,
    ("torus4x4_resnet50", "ldg", "b611438140eeb7a2"): 1_635_899_136 + 1_575_681_792,
}

KERNEL_SOURCES = ["gradient_all_reduce_ddl_gb300/csrc/fold_kernels.cu"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def sample_config(oracle, w, n: int):
    """The oracle's configuration for the first n elements of each rank of w:
    the same schedule (n-D dims included), bucket size, and the layer list cut
    at n."""
    layers = None
    if w.layers is not None:
        acc, layers = 0, []
        for v in w.layers:
            if acc >= n:
                break
            layers.append(min(v, n - acc))
            acc += layers[-1]
    return oracle.Config(w.P, n, w.dtype, w.topo, k=w.k, X=w.X, Y=w.Y, bucket_bytes=w.bucket_bytes, layers=layers,
                         dims=w.dims)


def host_link_study(host, bufs, stream, dev, reps: int = 3) -> dict:
    """Plain copies between the same page-locked host buffers and device
    buffers: the ceiling of the end-to-end paths.  `both_gbs` moves every rank
    in and every rank out with the two directions running at once (half of the
    ranks each way per phase, on two streams), in the e2e formula's units."""
    import torch
    P = len(host)
    nbytes = sum(h.numel() * h.element_size() for h in host)
    side = torch.cuda.Stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def h2d(ranks, st):
        with torch.cuda.stream(st):
            for r in ranks:
                bufs[r].copy_(host[r], non_blocking=True)

    def d2h(ranks, st):
        with torch.cuda.stream(st):
            for r in ranks:
                host[r].copy_(bufs[r], non_blocking=True)

    def both():
        lo, hi = range(P // 2), range(P // 2, P)
        side.wait_stream(stream)
        h2d(lo, stream)
        d2h(hi, side)
        stream.wait_stream(side)
        side.wait_stream(stream)
        h2d(hi, stream)
        d2h(lo, side)
        stream.wait_stream(side)

    def best_ms(fn):
        out = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            ev[0].record(stream)
            fn()
            ev[1].record(stream)
            torch.cuda.synchronize(dev)
            t = ev[0].elapsed_time(ev[1])
            out = t if out is None else min(out, t)
        return out

    t_in = best_ms(lambda: h2d(range(P), stream))
    t_out = best_ms(lambda: d2h(range(P), stream))
    t_both = best_ms(both)
    return {"h2d_gbs": round(nbytes / t_in / 1e6, 1), "d2h_gbs": round(nbytes / t_out / 1e6, 1),
            "both_gbs": round(2 * nbytes / t_both / 1e6, 1),
            "method": f"torch copies, page-locked host <-> device, best of {reps}; both = all ranks in and out, "
                      "the two directions concurrent on two streams"}


def schedule_name(w) -> str:
    if w.topo == "torus":
        return f"torus {w.X}x{w.Y}"
    if w.topo == "multiring":
        return f"multi-ring k={w.k}"
    if w.topo == "torus_nd":
        return "torus " + "x".join(str(d) for d in w.dims)
    return "ring"


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.6)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.3)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 - 1 <= r[0] <= self.t1 + 1] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm = [r[1] for r in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "reasons": sorted(reasons), "samples": len(inside)}


def cpu_baseline(w, target_s: float = 10.0, max_elems: int = 2_000_000):
    """The oracle as it stands (single thread) on a bounded sample of the
    workload: same P, schedule, dtype and value distribution, the first
    `max_elems` elements per rank as one bucket; repeated until `target_s`."""
    import oracle
    n = min(w.N, max_elems)
    host = [synth.draw_rank(w.seed, r, n, w.dist, w.sigma, w.dtype) for r in range(w.P)]
    cfg = sample_config(oracle, w, n)
    spent, reps = 0.0, 0
    while spent < target_s or reps < 1:
        bufs = [h.copy() for h in host]
        t = time.perf_counter()
        oracle.emulate(cfg, bufs, w.scale)
        spent += time.perf_counter() - t
        reps += 1
    per = spent / reps
    gbs = 2 * w.P * n * w.esize / per / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{w.P} ranks x {n} elements ({schedule_name(w)}, {w.dtype}), {reps} runs, "
                      f"{per * 1e3:.1f} ms per run, single-threaded step emulation",
            "elems_per_s": round(w.P * n / per, 1)}


def smi_gpu_id(local: int) -> str:
    """nvidia-smi --id for this process's GPU (index or UUID)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


def reduce_max(x: float, ws: int) -> float:
    """Largest value over the ranks (the job's time is its slowest replica)."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_replica_step: int, ws: int, ms_per_step: float) -> float:
    """Whole-job throughput: every replica moves its own bytes each step, and
    the step takes the slowest replica's time."""
    return bytes_per_replica_step * ws / (ms_per_step * 1e-3) / 1e9


def overlap_study(plan, bufs, w, stream, steps: int = 20, tokens: int = 2048):
    """Back-propagation overlapped with the bucketed all-reduce (Baidu
    write-up, opening paragraphs): a synthetic backward produces the buckets'
    gradients in reverse-layer order on `stream` -- per bucket a bf16 GEMM of
    2*tokens*params flops and the write of the bucket's
    gradients into all P rank buffers -- and either (a) all-reduces after the
    whole backward, or (b) signals each finished bucket (ddl_bucket_ready) so
    the plan's side stream reduces it while the next bucket is computed."""
    import torch
    nb = plan.num_buckets
    ranges = plan.buckets()
    dev = bufs[0].device
    pristine = [b.clone() for b in bufs]
    gemms = []
    for lo, hi in ranges:
        n = max(64, ((hi - lo) // 4096 + 63) // 64 * 64)
        gemms.append((torch.randn(tokens, 4096, device=dev, dtype=torch.bfloat16),
                      torch.randn(4096, n, device=dev, dtype=torch.bfloat16)))

    def backward_bucket(b):
        a, m = gemms[b]
        torch.matmul(a, m)
        lo, hi = ranges[b]
        for r in range(w.P):
            bufs[r][lo:hi].copy_(pristine[r][lo:hi])

    def seq():
        for b in range(nb):
            backward_bucket(b)
        plan.allreduce(bufs, w.scale, stream)

    def ovl():
        plan.overlap_begin(bufs, w.scale, stream)
        for b in range(nb):
            backward_bucket(b)
            plan.bucket_ready(b, stream)
        plan.overlap_end(stream)

    def backward_only():
        for b in range(nb):
            backward_bucket(b)

    out = {}
    with torch.cuda.stream(stream):
        for name, fn in [("backward_only", backward_only), ("sequential", seq), ("overlapped", ovl)]:
            for _ in range(3):
                fn()
            torch.cuda.synchronize(dev)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(steps):
                fn()
            s1.record(stream)
            torch.cuda.synchronize(dev)
            out[name + "_ms"] = round(s0.elapsed_time(s1) / steps, 4)
    out["allreduce_alone_ms"] = None
    out["saved_ms"] = round(out["sequential_ms"] - out["overlapped_ms"], 4)
    out["buckets"] = nb
    out["backward"] = (f"per bucket: bf16 GEMM {tokens}x4096 @ 4096x(params/4096) + gradient writes to all "
                       f"P ranks")
    del pristine, gemms
    return out


def sgd_study(plan, bufs, w, stream, steps: int = 50):
    """All-reduce + momentum-SGD update: the fused pass (ddl_allreduce_sgd)
    against the all-reduce followed by an unfused update of the P replicas'
    parameters (torch foreach kernels)."""
    import torch
    dev = bufs[0].device
    params = [torch.zeros(w.N, device=dev) for _ in range(w.P)]
    moms = [torch.zeros(w.N, device=dev) for _ in range(w.P)]
    lr, mu, wd = 0.01, 0.9, 1e-4

    def fused():
        plan.allreduce_sgd(bufs, params, moms, w.scale, lr, mu, wd, keep_grads=True, stream=stream)

    def unfused():
        plan.allreduce(bufs, w.scale, stream)
        g = [b.float() for b in bufs] if w.dtype == "f16" else bufs
        d = torch._foreach_add(g, params, alpha=wd)
        torch._foreach_mul_(moms, mu)
        torch._foreach_add_(moms, d)
        torch._foreach_add_(params, moms, alpha=-lr)

    out = {}
    with torch.cuda.stream(stream):
        for name, fn in [("fused", fused), ("unfused", unfused)]:
            for _ in range(3):
                fn()
            torch.cuda.synchronize(dev)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(steps):
                fn()
            s1.record(stream)
            torch.cuda.synchronize(dev)
            out[name + "_ms"] = round(s0.elapsed_time(s1) / steps, 4)
    algo = w.P * w.N * (2 * w.esize + 16)  # gradient read + write, parameter and momentum read + write
    out["fused_bytes_per_step"] = algo
    out["fused_GBps"] = round(algo / (out["fused_ms"] * 1e-3) / 1e9, 1)
    out["fused_frac_of_hbm"] = round(out["fused_GBps"] / measured_peak()[0], 4)
    out["update"] = "d = g + wd p; v = mu v + d; p = p - lr v on every rank's fp32 copy (lr 0.01, mu 0.9, wd 1e-4)"
    del params, moms
    return out


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    # per-step sample sized so that K + W steps take about two minutes at the
    # oracle's ~8 ns per rank-element (copies included)
    budget_s = 120.0
    n = int(budget_s / ((args.steps + args.warmup) * w.P * 8e-9))
    n = max(4096, min(n, w.N, 2_000_000))
    host = [synth.draw_rank(w.seed, r, n, w.dist, w.sigma, w.dtype) for r in range(w.P)]
    cfg = sample_config(oracle, w, n)
    times = []
    for i in range(args.warmup + args.steps):
        bufs = [h.copy() for h in host]
        t = time.perf_counter()
        oracle.emulate(cfg, bufs, w.scale)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    per = sum(times) / len(times)
    gbs = 2 * w.P * n * w.esize / per / 1e9
    sample = (f"oracle on {w.P} ranks x {n} elements of {w.name} ({schedule_name(w)}, {w.dtype}) per step, "
              f"single-threaded")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "config": {"workload": w.name, "P": w.P, "N": w.N, "schedule": schedule_name(w),
                                            "sample_elems_per_rank": n},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--mode", default="fused", choices=["fused", "stepwise", "rankorder"])
    ap.add_argument("--kernel", default="auto", choices=["auto", "ldg", "bulk", "bulkload", "tma", "chunked"])
    ap.add_argument("--slab", action="store_true",
                    help="rank buffers in one slab (ddl_allreduce_slab); needed by --kernel tma")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--elems", type=int, default=0,
                    help="run the workload with this many elements per rank (no layer list): small cases "
                         "for profiling")
    ap.add_argument("--overlap", action="store_true",
                    help="also time a synthetic backward overlapped with the bucketed all-reduce")
    ap.add_argument("--sgd", action="store_true",
                    help="also time the all-reduce fused with the momentum-SGD update")
    ap.add_argument("--overlap-tokens", type=int, default=2048,
                    help="GEMM rows of the synthetic backward (its compute per parameter)")
    ap.add_argument("--graph", action="store_true",
                    help="capture one ddl_allreduce in a CUDA graph and replay it each step")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = synth.WORKLOADS[args.workload]
    if args.elems:
        w = w.with_(N=args.elems, layers=None, name=f"{w.name}@{args.elems}")
    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    import torch.distributed as dist

    from gradient_all_reduce_ddl_gb300 import ddl

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)

    tdt = torch.float16 if w.dtype == "f16" else torch.float32
    bufs = []
    slab = None
    stride_elems = (w.N + 63) // 64 * 64  # 256-byte aligned rank rows in the slab
    if args.slab:
        slab = torch.empty(w.P * stride_elems, dtype=tdt, device=dev)
    for r in range(w.P):
        t = slab[r * stride_elems: r * stride_elems + w.N] if slab is not None else \
            torch.empty(w.N, dtype=tdt, device=dev)
        synth.fill_device(t.data_ptr(), w.N, w.seed, r, w.dist, w.sigma, w.dtype, stream=stream.cuda_stream)
        bufs.append(t)
    plan = ddl.Plan.for_workload(w, mode=args.mode, kernel=args.kernel)
    if slab is not None:
        slab_stride = stride_elems * w.esize
        plan.allreduce = (lambda b, sc, st=None, _p=plan:
                          _p.allreduce_slab(slab, slab_stride, sc, st))
    nbytes = w.min_bytes

    def barrier():
        if ws > 1:
            dist.barrier()

    for _ in range(args.warmup):
        plan.allreduce(bufs, w.scale, stream)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(smi_gpu_id(local if ws > 1 else 0))
    graph = None
    per_graph = 10  # all-reduces captured per graph, so one replay's overhead is shared
    if args.graph:
        if args.steps % per_graph:
            args.steps += per_graph - args.steps % per_graph
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        l0 = plan.launches
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(per_graph):
                plan.allreduce(bufs, w.scale, cap)
        graph_launches = (plan.launches - l0) // per_graph
        stream.wait_stream(cap)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(dev)

    clocks.start()
    launches0 = plan.launches
    barrier()
    torch.cuda.synchronize(dev)
    clocks.mark("t0")
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    if graph is not None:
        for _ in range(args.steps // per_graph):
            graph.replay()
    else:
        for _ in range(args.steps):
            plan.allreduce(bufs, w.scale, stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks.mark("t1")
    clk = clocks.stop()
    launches = plan.launches - launches0 if graph is None else graph_launches * args.steps
    local_ms = start.elapsed_time(end)
    total_ms = reduce_max(local_ms, ws)
    ms_per_step = total_ms / args.steps
    gbs = job_gbs(nbytes, ws, ms_per_step)
    elems = w.P * w.N * ws / (ms_per_step * 1e-3)

    # spread: 20 more steps, each bracketed by its own events (outside the
    # timed region; only where a step is long enough that two event records
    # per step do not distort it)
    step_median_ms = None
    if graph is None and ms_per_step > 0.05:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(21)]
        evs[0].record(stream)
        for i in range(20):
            plan.allreduce(bufs, w.scale, stream)
            evs[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        per = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(20))
        step_median_ms = {"median": round(0.5 * (per[9] + per[10]), 5), "min": round(per[0], 5),
                          "max": round(per[-1], 5), "steps": 20}

    # roofline of the dominant kernel: one fused launch per bucket
    nb = plan.num_buckets
    launches_per_call = max(1, launches // args.steps)
    # the step is one ddl_allreduce: its kernels back to back on one stream, so
    # the call's average device time is this replica's timed region / steps
    avg_call_ms = local_ms / args.steps
    peak, peak_kind = measured_peak()
    kernel_name = {"fused": {"bulk": "fold_bulk_kernel", "bulkload": "fold_bulk_kernel", "chunked": "fold_chunked_kernel",
                             "tma": "fold_tma_kernel" if args.slab else "fold_ldg_kernel"}.get(args.kernel,
                                                                                            "fold_ldg_kernel"),
                   "rankorder": "fold_ldg_kernel (rank order)", "stepwise": "step_kernel"}[args.mode]
    kernel_bytes = nbytes
    if args.mode == "stepwise":
        # the step kernels' own minimum: a reduce-scatter message element reads
        # two values and writes one, an all-gather element reads one and writes
        # one, and each half of the 2(P-1)N elements moved is one of the two
        moved = plan.traffic()[0]
        kernel_bytes = (moved // 2) * 5 * w.esize if moved else 2 * w.N * w.esize
    achieved = kernel_bytes / (avg_call_ms * 1e-3) / 1e9  # bytes of all launches / time of the call
    traffic = (NCU_TRAFFIC.get((w.name, args.kernel if args.kernel != "auto" else "ldg", kernel_hash()))
               if args.mode == "fused" else None)
    roofline = {"bound": "hbm", "kernel": kernel_name, "achieved": None if achieved is None else round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": None if achieved is None else round(achieved / peak, 4),
                "peak_kind": f"hbm_gbs of {peak_kind}", "traffic": traffic,
                "algorithmic_bytes_per_launch": kernel_bytes // max(1, launches_per_call),
                "launches_per_step": launches_per_call,
                "avg_call_ms": round(avg_call_ms, 4)}

    # end to end through the C ABI with page-locked host buffers
    e2e = None
    if not args.no_e2e:
        host = [torch.empty(w.N, dtype=tdt, pin_memory=True) for _ in range(w.P)]
        for r in range(w.P):
            host[r].copy_(bufs[r])
        torch.cuda.synchronize(dev)
        plan.allreduce_host(host, bufs, w.scale, stream)
        torch.cuda.synchronize(dev)
        barrier()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(args.e2e_steps):
            plan.allreduce_host(host, bufs, w.scale, stream)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = reduce_max(s0.elapsed_time(s1) / args.e2e_steps, ws)
        staged = {"value": round(job_gbs(nbytes, ws, e2e_ms), 2), "unit": "GB/s",
                  "h2d_bytes_per_step": w.P * w.N * w.esize, "d2h_bytes_per_step": w.P * w.N * w.esize,
                  "ms_per_step": round(e2e_ms, 3), "steps": args.e2e_steps,
                  "path": "ddl_allreduce_host with device staging: copy-in, fused pass, copy-out "
                          "pipelined over element ranges on three streams"}
        # zero-copy: the fused pass reads and writes the page-locked host buffers directly
        plan.allreduce_host(host, None, w.scale, stream)
        torch.cuda.synchronize(dev)
        barrier()
        s0.record(stream)
        for _ in range(args.e2e_steps):
            plan.allreduce_host(host, None, w.scale, stream)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        zc_ms = reduce_max(s0.elapsed_time(s1) / args.e2e_steps, ws)
        zero = {"value": round(job_gbs(nbytes, ws, zc_ms), 2), "unit": "GB/s",
                "h2d_bytes_per_step": w.P * w.N * w.esize, "d2h_bytes_per_step": w.P * w.N * w.esize,
                "ms_per_step": round(zc_ms, 3), "steps": args.e2e_steps,
                "path": "ddl_allreduce_host without staging: the fused pass loads and stores the page-locked "
                        "host buffers over the host link"}
        e2e, alt = (zero, staged) if zc_ms < e2e_ms else (staged, zero)
        e2e = dict(e2e, other_path=alt)
        link = host_link_study(host, bufs, stream, dev)
        link["e2e_frac_of_both"] = round(e2e["value"] / ws / link["both_gbs"], 4)
        e2e["host_link"] = link
        del host

    overlap = None
    if args.overlap:
        overlap = overlap_study(plan, bufs, w, stream, tokens=args.overlap_tokens)
        overlap["allreduce_alone_ms"] = round(ms_per_step, 4)

    sgd = sgd_study(plan, bufs, w, stream) if args.sgd else None

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu = cpu_baseline(w)

    # alpha-beta model of the same schedule on P real workers, at the Baidu
    # write-up's ~6 GB/s InfiniBand (alpha 0) and with 10 us of latency per step
    model = {"link_GBps": 6.0, "alpha0_s": round(plan.cost(0.0, 1 / 6e9), 6),
             "alpha10us_s": round(plan.cost(10e-6, 1 / 6e9), 6), "steps": plan.traffic()[1],
             "elements_sent_total": plan.traffic()[0]}

    if rank == 0:
        line = {"metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
                "config": {"workload": w.name, "P": w.P, "N": w.N, "schedule": schedule_name(w), "mode": args.mode,
                           "kernel": args.kernel, "buckets": nb, "bytes_per_step": nbytes,
                           "layout": "one slab (ddl_allreduce_slab)" if args.slab else "P separate buffers",
                           "launch": (f"CUDA graph replay, {per_graph} all-reduces per graph" if args.graph
                                      else "ddl_allreduce call per step"),
                           "elems_per_s": round(elems, 1), "frac_of_hbm": round(gbs / ws / peak, 4),
                           "frac_of_nominal_hbm": round(gbs / ws / 7900.0, 4),
                           "step_ms_spread": step_median_ms,
                           "l2": (f"inputs {w.P * w.N * w.esize / 1e9:.2f} GB per replica, larger than the 129 MB L2"
                                  if w.P * w.N * w.esize > 129e6 else
                                  f"inputs {w.P * w.N * w.esize / 1e6:.1f} MB fit in the 129 MB L2: back-to-back "
                                  f"steps run on a warm L2 (a latency measurement, not an HBM one)"),
                           "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU, P logical ranks"},
                "clocks": clk, "gpu_launches": launches, "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu,
                "cluster_model": model, "overlap": overlap, "sgd": sgd,
                "kernel_src": kernel_hash()}
        print(json.dumps(line), flush=True)
    plan.close()
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
