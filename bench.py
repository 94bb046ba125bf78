"""Benchmark of the fused gradient all-reduce on one GB300 (or N replicas).

Metric: all-reduce GB/s on the algorithmic minimum of HBM traffic, 2*P*N*e
bytes per all-reduce (every rank element read once and written once), plus
elements/s, per schedule; and the fraction of the measured HBM copy bandwidth.

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--mode fused|stepwise|rankorder]
                    [--kernel auto|ldg|bulk|bulkload|tma|chunked] [--impl ours|reference]
                    [--no-e2e] [--no-cpu] [--no-configs]

Default workload ("lm300m_sweep"): the three schedules the pages compare, on
the 300M-parameter language model's gradient of the Baidu write-up (P = 16
ranks x 300,000,000 fp32 = 1.2 GB per rank, 19.2 GB resident, values
N(0, 1e-4), scale 1/16): ring, multi-ring k=2 and 2D torus 4x4 over the same
buffers.  A step is one all-reduce under each of the three schedules; `value`
is their bytes over the step's time, and `per_schedule` splits it.  The
inputs are far larger than the 129 MB L2, so no flush is needed.

The same run also times the other four problems (the 2 MB integer ring, the
ResNet-50 4x4 torus, the fp16 8x4 torus of the ResNet-50 layout, the P=64
multi-ring of ResNet-101 in 25 MiB buckets) under `configs`.  The oracle (the
plain single-threaded CPU emulation) is run only in the `cpu_baseline` leg:
it is timed there on a bounded sample of the workload, and, in the same leg,
its closed form is compared bit for bit with the GPU's results at sampled
elements of every workload the run timed.

With --gpus N > 1 (torchrun) the path does not shard: each GPU runs an
independent replica, and the reported value is the total over all replicas.
--impl reference times the oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
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

# workloads timed together over one set of buffers (same P, N, dtype, inputs)
SWEEPS = {
    "lm300m_sweep": ("ring16_lm300m", "multiring16_lm300m", "torus4x4_lm300m"),
}
DEFAULT_WORKLOAD = "lm300m_sweep"
# the other problems, timed after the headline under `configs`
SECONDARY = ("ring4_int", "torus4x4_resnet50", "torus8x4_resnet50_f16", "multiring64_resnet101")

# dram__bytes_read.sum + dram__bytes_write.sum of one fused launch from one ncu
# capture, and the algorithmic bytes (2*P*n*e) of that launch, keyed by
# (schedule kind, dtype, kernel variant, sha256[:16] of the kernel source).
# A launch of another size reports the capture's traffic scaled by its
# algorithmic bytes; a changed kernel source reports null.
NCU_TRAFFIC = {
    # P = 16 x 20,000,000 fp32 (1.28 GB resident, above L2): 2.56 GB algorithmic per launch
    ("ring", "f32", "ldg", "878096f0134ae334"): (1_280_214_528 + 1_220_379_392, 2_560_000_000),
    ("multiring", "f32", "ldg", "878096f0134ae334"): (1_280_397_056 + 1_220_582_400, 2_560_000_000),
    ("torus", "f32", "ldg", "878096f0134ae334"): (1_280_243_200 + 1_220_768_000, 2_560_000_000),
}

KERNEL_SOURCES = ["gradient_all_reduce_ddl_gb300/csrc/fold_kernels.cu"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(w, kernel: str, launch_bytes: int):
    """Per-launch DRAM traffic from the stored capture, scaled to this launch."""
    hit = NCU_TRAFFIC.get((w.topo, w.dtype, kernel if kernel != "auto" else "ldg", kernel_hash()))
    if hit is None:
        return None
    traffic, algo = hit
    return int(round(traffic * launch_bytes / algo))


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


def full_config(oracle, w):
    return oracle.Config(w.P, w.N, w.dtype, w.topo, k=w.k, X=w.X, Y=w.Y, bucket_bytes=w.bucket_bytes,
                         layers=w.layers, dims=w.dims)


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


def host_cpu() -> dict:
    """The host cores the oracle legs run on: usable cores and the CPU model."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as fh:
                for line in fh:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    try:
        nproc = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        nproc = os.cpu_count()
    return {"nproc": nproc, "cpu_model": model or "unknown", "arch": platform.machine()}


class ClockSampler:
    """nvidia-smi clock/throttle samples every 50 ms while running; stop()
    keeps the samples taken between mark('t0') and mark('t1')."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.gpu = gpu_id
        self.period_ms = period_ms
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.6)

    def mark(self, which):
        setattr(self, which, time.time())

    @staticmethod
    def _stamp(text: str) -> float:
        base, _, frac = text.strip().partition(".")
        t = time.mktime(time.strptime(base, "%Y/%m/%d %H:%M:%S"))
        return t + (float("0." + frac) if frac.isdigit() else 0.0)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append((self._stamp(f[0]), float(f[2]), float(f[3]), float(f[4]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for n, v in zip(names, r[4]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm = [r[1] for r in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "power_w_max": max(r[3] for r in inside) if inside else None,
                "reasons": sorted(reasons), "samples": len(inside), "period_ms": self.period_ms,
                "timed_region_s": round(self.t1 - self.t0, 3)}


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


def _part_edges(lo, hi, m):
    n = hi - lo
    base, rem = divmod(n, m)
    return [lo + i * base + min(i, rem) for i in range(m + 1)]


def sample_indices(w, buckets, n_rand: int = 20_000, seed: int = 2017) -> np.ndarray:
    """Element indices to compare: all of them for small buffers, else random
    ones plus those at and next to every bucket, slice and chunk edge (bucket
    ranges as the plan reports them)."""
    if w.N <= 65_536:
        return np.arange(w.N, dtype=np.int64)
    edges = set()
    for lo, hi in buckets:
        if w.topo == "torus":
            for c0, c1 in zip(_part_edges(lo, hi, w.X)[:-1], _part_edges(lo, hi, w.X)[1:]):
                edges.update(_part_edges(c0, c1, w.Y))
        elif w.topo == "torus_nd":
            level = [(lo, hi)]
            for D in w.dims:
                nxt = []
                for a, b in level:
                    e = _part_edges(a, b, D)
                    edges.update(e)
                    nxt += list(zip(e[:-1], e[1:]))
                level = nxt
        elif w.topo == "multiring":
            for s0, s1 in zip(_part_edges(lo, hi, w.k)[:-1], _part_edges(lo, hi, w.k)[1:]):
                edges.update(_part_edges(s0, s1, w.P))
        else:
            edges.update(_part_edges(lo, hi, w.P))
    near = {e + d for e in edges for d in (-2, -1, 0, 1) if 0 <= e + d < w.N}
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.integers(0, w.N, n_rand), np.array(sorted(near), dtype=np.int64)]))


def gather_sample(w, bufs, idx) -> dict:
    """Rank 0's result bits at idx, and whether every rank equals rank 0."""
    import torch
    view = torch.int16 if w.dtype == "f16" else torch.int32
    same = all(torch.equal(b.view(view), bufs[0].view(view)) for b in bufs[1:])
    got = bufs[0][torch.from_numpy(idx).to(bufs[0].device)].view(view).cpu().numpy()
    got = got.view(np.uint16) if w.dtype == "f16" else got.view(np.float32)
    return {"idx": idx, "got": got, "ranks_identical": bool(same)}


def fill(w, bufs, stream):
    for r, t in enumerate(bufs):
        synth.fill_device(t.data_ptr(), w.N, w.seed, r, w.dist, w.sigma, w.dtype, stream=stream.cuda_stream)


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


# ---------------------------------------------------------------------------
# GPU legs
# ---------------------------------------------------------------------------

def alloc_bufs(w, dev, stream, slab: bool = False):
    """P rank buffers filled with w's inputs: separate tensors, or views of one
    slab with 256-byte aligned rank rows.  Returns (bufs, slab, stride bytes)."""
    import torch
    tdt = torch.float16 if w.dtype == "f16" else torch.float32
    stride = (w.N + 63) // 64 * 64
    base = torch.empty(w.P * stride, dtype=tdt, device=dev) if slab else None
    bufs = [base[r * stride: r * stride + w.N] if slab else torch.empty(w.N, dtype=tdt, device=dev)
            for r in range(w.P)]
    fill(w, bufs, stream)
    return bufs, base, stride * w.esize


def timed_steps(calls, stream, dev, steps: int, split: bool):
    """Runs `steps` steps, each the calls in order, between two events on
    `stream`.  Returns (total ms, per-call ms summed over the steps or None);
    the per-call split records one more event after every call."""
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = ([[torch.cuda.Event(enable_timing=True) for _ in calls] for _ in range(steps)]
             if split and len(calls) > 1 else None)
    start.record(stream)
    for s in range(steps):
        for j, c in enumerate(calls):
            c()
            if marks is not None:
                marks[s][j].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    total = start.elapsed_time(end)
    per = None
    if marks is not None:
        per = [0.0] * len(calls)
        prev = start
        for s in range(steps):
            for j in range(len(calls)):
                per[j] += prev.elapsed_time(marks[s][j])
                prev = marks[s][j]
    return total, per


def kernel_bytes_of(plan, w, mode: str) -> int:
    """Algorithmic bytes of one call's launches: 2*P*N*e for the one-pass
    modes; the step kernels' own minimum in stepwise mode (a reduce-scatter
    message element reads two values and writes one, an all-gather element
    reads one and writes one; each is half of the 2(P-1)N elements moved)."""
    if mode == "stepwise":
        moved = plan.traffic()[0]
        return (moved // 2) * 5 * w.esize if moved else 2 * w.N * w.esize
    return w.min_bytes


def host_memory_short(need: int, ws: int, avail: int | None = None) -> str | None:
    """Why the page-locked buffers of the e2e leg do not fit on this host, or
    None.  Every replica on a host pins its own buffers at once, and the
    answer is the same on every rank (a rank that skipped the leg would leave
    the others waiting in its max-over-ranks timing)."""
    if avail is None:
        try:
            with open("/proc/meminfo") as fh:
                avail = next(int(line.split()[1]) * 1024 for line in fh if line.startswith("MemAvailable:"))
        except (OSError, StopIteration, ValueError):
            avail = None
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    short = avail is not None and avail < need * local_ranks + (8 << 30)
    if reduce_max(1.0 if short else 0.0, ws) == 0:
        return None
    if short:
        return (f"host memory: {avail / 1e9:.1f} GB available, {need * local_ranks / 1e9:.1f} GB of page-locked "
                f"buffers needed")
    return "host memory short on another rank"


def e2e_leg(plans, wls, bufs, stream, dev, ws: int, e2e_steps: int) -> dict:
    """The same step through ddl_allreduce_host on page-locked host buffers:
    every call moves P*N*e bytes in and P*N*e out over the host link inside
    the timed region.  Both the zero-copy pass and the staged pipeline are
    timed; the faster is reported, the other beside it."""
    import torch
    w0 = wls[0]
    tdt = bufs[0].dtype
    why = host_memory_short(w0.P * w0.N * w0.esize, ws)
    if why:
        return {"value": None, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0, "skipped": why}
    host = [torch.empty(w0.N, dtype=tdt, pin_memory=True) for _ in range(w0.P)]
    for r in range(w0.P):
        host[r].copy_(bufs[r])
    torch.cuda.synchronize(dev)
    nbytes = sum(w.min_bytes for w in wls)
    io = {"h2d_bytes_per_step": w0.P * w0.N * w0.esize * len(wls),
          "d2h_bytes_per_step": w0.P * w0.N * w0.esize * len(wls)}

    def run(dev_bufs):
        for p, w in zip(plans, wls):
            p.allreduce_host(host, dev_bufs, w.scale, stream)
        torch.cuda.synchronize(dev)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(e2e_steps):
            for p, w in zip(plans, wls):
                p.allreduce_host(host, dev_bufs, w.scale, stream)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        return reduce_max(s0.elapsed_time(s1) / e2e_steps, ws)

    staged_ms = run(bufs)
    zc_ms = run(None)
    staged = dict(io, value=round(job_gbs(nbytes, ws, staged_ms), 2), unit="GB/s", ms_per_step=round(staged_ms, 3),
                  steps=e2e_steps, path="ddl_allreduce_host with device staging: copy-in, fused pass, copy-out "
                                        "pipelined over element ranges on three streams")
    zero = dict(io, value=round(job_gbs(nbytes, ws, zc_ms), 2), unit="GB/s", ms_per_step=round(zc_ms, 3),
                steps=e2e_steps, path="ddl_allreduce_host without staging: the fused pass loads and stores the "
                                      "page-locked host buffers over the host link")
    best, alt = (zero, staged) if zc_ms < staged_ms else (staged, zero)
    out = dict(best, other_path=alt)
    link = host_link_study(host, bufs, stream, dev)
    link["e2e_frac_of_both"] = round(out["value"] / ws / link["both_gbs"], 4)
    out["host_link"] = link
    del host
    return out


def secondary_leg(ddl, name: str, dev, stream, peak: float, samples: dict, target_ms: float = 250.0) -> dict:
    """One of the other problems, timed on its own after the headline: one
    all-reduce of fresh inputs (its result sampled for the oracle leg), three
    warm-up calls, then enough calls for about `target_ms` of device time.
    A bucketed problem also times its bucket scheduler against a synthetic
    backward (overlap_study)."""
    import torch
    w = synth.WORKLOADS[name]
    bufs, _, _ = alloc_bufs(w, dev, stream)
    plan = ddl.Plan.for_workload(w)
    try:
        with torch.cuda.stream(stream):
            plan.allreduce(bufs, w.scale, stream)
            torch.cuda.synchronize(dev)
            plan.check()
            samples[name] = gather_sample(w, bufs, sample_indices(w, plan.buckets()))
            call = (lambda: plan.allreduce(bufs, w.scale, stream))
            for _ in range(3):
                call()
            probe, _ = timed_steps([call], stream, dev, 5, False)
            steps = int(min(5000, max(20, target_ms / max(probe / 5, 1e-3))))
            l0 = plan.launches
            total, _ = timed_steps([call], stream, dev, steps, False)
            launches = plan.launches - l0
            ms = total / steps
            gbs = w.min_bytes / (ms * 1e-3) / 1e9
            out = {"P": w.P, "N": w.N, "dtype": w.dtype, "schedule": schedule_name(w), "buckets": plan.num_buckets,
                   "bytes_per_step": w.min_bytes, "steps": steps, "ms_per_step": round(ms, 5),
                   "GBps": round(gbs, 1), "elems_per_s": round(w.P * w.N / (ms * 1e-3), 1),
                   "frac_of_hbm": round(gbs / peak, 4), "gpu_launches": launches, "kernel": plan.kernel_name,
                   "l2": ("inputs larger than the 129 MB L2" if w.P * w.N * w.esize > 129e6 else
                          "inputs fit in the 129 MB L2: back-to-back calls run on a warm L2 (latency, not HBM)")}
            if w.P * w.N * w.esize <= 129e6:
                # the latency case: also per all-reduce in CUDA-graph replay
                per_graph = 10
                cap = torch.cuda.Stream(dev)
                cap.wait_stream(stream)
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=cap):
                    for _ in range(per_graph):
                        plan.allreduce(bufs, w.scale, cap)
                stream.wait_stream(cap)
                for _ in range(3):
                    graph.replay()
                torch.cuda.synchronize(dev)
                reps = 200
                g_total, _ = timed_steps([graph.replay], stream, dev, reps, False)
                out["us_per_call"] = round(ms * 1e3, 3)
                out["us_per_allreduce_graph_replay"] = round(g_total * 1e3 / (reps * per_graph), 3)
                del graph
            if plan.num_buckets > 1:
                # the bucket scheduler against the same step run sequentially
                out["overlap"] = overlap_study(plan, bufs, w, stream, steps=10)
                out["overlap"]["allreduce_alone_ms"] = round(ms, 4)
            torch.cuda.synchronize(dev)
    finally:
        plan.close()
        del bufs
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# Oracle legs (the only places this file runs the oracle)
# ---------------------------------------------------------------------------

def oracle_check(oracle, w, sample: dict) -> dict:
    """The oracle's closed form at the sampled elements against the GPU's
    result there: bit for bit (schedule-order modes)."""
    idx = sample["idx"].astype(np.uint64)
    x_rows = np.stack([w.rank_values(r, idx) for r in range(w.P)], axis=1)
    want = oracle.closed_form(full_config(oracle, w), x_rows, idx, w.scale)
    bad = int(np.count_nonzero(sample["got"] != want))
    out = {"elements": int(idx.size), "mismatches": bad, "bit_exact": bad == 0,
           "ranks_identical": sample["ranks_identical"], "against": "oracle closed form"}
    if w.dist == "int1000" and w.N == idx.size:
        ints = np.stack([w.rank_values(r) for r in range(w.P)]).astype(np.int64).sum(axis=0)
        out["equals_exact_int64_sums"] = bool(np.array_equal(sample["got"], (ints * w.scale).astype(np.float32)))
    return out


def cpu_baseline(wls, samples: dict, target_s: float = 10.0, max_elems: int = 2_000_000) -> dict:
    """The oracle as it stands (single thread) on a bounded sample of the
    step's workloads: same P, schedule, dtype and value distribution, the
    first `max_elems` elements per rank, each schedule repeated for about
    target_s / len(wls) seconds.  The same leg then checks the GPU's sampled
    results of every workload in `samples` against the oracle's closed form."""
    import oracle
    per_w, spent_all, bytes_all = {}, 0.0, 0
    for w in wls:
        n = min(w.N, max_elems)
        host = [synth.draw_rank(w.seed, r, n, w.dist, w.sigma, w.dtype) for r in range(w.P)]
        cfg = sample_config(oracle, w, n)
        spent, reps = 0.0, 0
        while spent < target_s / len(wls) or reps < 1:
            bufs = [h.copy() for h in host]
            t = time.perf_counter()
            oracle.emulate(cfg, bufs, w.scale)
            spent += time.perf_counter() - t
            reps += 1
        per = spent / reps
        per_w[w.name] = {"GBps": round(2 * w.P * n * w.esize / per / 1e9, 4), "ms_per_run": round(per * 1e3, 2),
                         "runs": reps, "elems_per_rank": n}
        spent_all += per
        bytes_all += 2 * w.P * n * w.esize
    hc = host_cpu()
    w0 = wls[0]
    n0 = min(w0.N, max_elems)
    out = {"value": round(bytes_all / spent_all / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "nproc": hc["nproc"], "cpu_model": hc["cpu_model"], "arch": hc["arch"],
           "sample": (f"{w0.P} ranks x {n0} elements per schedule ({', '.join(schedule_name(w) for w in wls)}; "
                      f"{w0.dtype}), single-threaded step emulation on 1 of {hc['nproc']} host cores"),
           "elems_per_s": round(sum(w.P * min(w.N, max_elems) for w in wls) / spent_all, 1),
           "per_schedule": per_w}
    by_name = {w.name: w for w in wls}
    checks = {}
    for name, sample in samples.items():
        w = by_name.get(name) or synth.WORKLOADS[name]
        checks[name] = oracle_check(oracle, w, sample)
    out["parity_sample"] = checks
    out["parity_all_bit_exact"] = all(c["bit_exact"] and c["ranks_identical"] for c in checks.values())
    return out


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def workloads_of(args):
    names = SWEEPS.get(args.workload, (args.workload,))
    wls = [synth.WORKLOADS[n] for n in names]
    if args.elems:
        wls = [w.with_(N=args.elems, layers=None, name=f"{w.name}@{args.elems}") for w in wls]
    return wls


def run_reference(args, wls):
    _, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    # per-step sample sized so that K + W steps take about two minutes at the
    # oracle's ~8 ns per rank-element (copies included)
    budget_s = 120.0
    w0 = wls[0]
    n = int(budget_s / ((args.steps + args.warmup) * len(wls) * w0.P * 8e-9))
    n = max(4096, min(n, w0.N, 2_000_000))
    host = [synth.draw_rank(w0.seed, r, n, w0.dist, w0.sigma, w0.dtype) for r in range(w0.P)]
    cfgs = [sample_config(oracle, w, n) for w in wls]
    times = []
    for i in range(args.warmup + args.steps):
        t_step = 0.0
        for w, cfg in zip(wls, cfgs):
            bufs = [h.copy() for h in host]
            t = time.perf_counter()
            oracle.emulate(cfg, bufs, w.scale)
            t_step += time.perf_counter() - t
        if i >= args.warmup:
            times.append(t_step)
    per = sum(times) / len(times)
    gbs = 2 * w0.P * n * w0.esize * len(wls) / per / 1e9
    hc = host_cpu()
    sample = (f"oracle on {w0.P} ranks x {n} elements per schedule ({', '.join(schedule_name(w) for w in wls)}; "
              f"{w0.dtype}) per step, single-threaded on 1 of {hc['nproc']} host cores ({hc['cpu_model']})")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w0.dtype,
            "data": "synthetic", "config": {"workload": args.workload, "P": w0.P, "N": w0.N,
                                            "schedules": [schedule_name(w) for w in wls],
                                            "sample_elems_per_rank": n},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "nproc": hc["nproc"], "cpu_model": hc["cpu_model"], "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS) + sorted(SWEEPS))
    ap.add_argument("--mode", default="fused", choices=["fused", "stepwise", "rankorder"])
    ap.add_argument("--kernel", default="auto", choices=["auto", "ldg", "bulkload", "chunked"])
    ap.add_argument("--slab", action="store_true", help="rank buffers in one slab (ddl_allreduce_slab)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other problems under `configs`")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--clock-ms", type=int, default=50, help="nvidia-smi clock sampling period during the timed region")
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
                    help="capture ten steps in a CUDA graph and replay it")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wls = workloads_of(args)
    w0 = wls[0]
    assert all((w.P, w.N, w.dtype, w.seed, w.dist, w.sigma) == (w0.P, w0.N, w0.dtype, w0.seed, w0.dist, w0.sigma)
               for w in wls), "a sweep's workloads share their buffers"
    if args.impl == "reference":
        return run_reference(args, wls)

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
    peak, peak_kind = measured_peak()
    oracle_legs = rank == 0 and ws == 1 and not args.no_cpu

    bufs, slab, slab_stride = alloc_bufs(w0, dev, stream, slab=args.slab)
    plans = [ddl.Plan.for_workload(w, mode=args.mode, kernel=args.kernel) for w in wls]

    def mk(plan, w):
        if slab is not None:
            return lambda: plan.allreduce_slab(slab, slab_stride, w.scale, stream)
        return lambda: plan.allreduce(bufs, w.scale, stream)

    calls = [mk(p, w) for p, w in zip(plans, wls)]
    n_buckets = plans[0].num_buckets

    # one all-reduce of fresh inputs per schedule, sampled for the oracle leg
    samples = {}
    if oracle_legs and args.mode != "rankorder":
        for j, (p, w, c) in enumerate(zip(plans, wls, calls)):
            if j:
                fill(w, bufs, stream)
            c()
            torch.cuda.synchronize(dev)
            p.check()
            samples[w.name] = gather_sample(w, bufs, sample_indices(w, p.buckets()))

    for _ in range(args.warmup):
        for c in calls:
            c()
    torch.cuda.synchronize(dev)

    def barrier():
        if ws > 1:
            dist.barrier()

    graph = None
    per_graph = 10  # steps captured per graph, so one replay's overhead is shared
    if args.graph:
        if args.steps % per_graph:
            args.steps += per_graph - args.steps % per_graph
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        l0 = sum(p.launches for p in plans)
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(per_graph):
                for p, w in zip(plans, wls):
                    p.allreduce(bufs, w.scale, cap)
        graph_launches = (sum(p.launches for p in plans) - l0) // per_graph
        stream.wait_stream(cap)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(smi_gpu_id(local if ws > 1 else 0), args.clock_ms)
    clocks.start()
    launches0 = sum(p.launches for p in plans)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.mark("t0")
    if graph is not None:
        local_ms, per_call = timed_steps([graph.replay], stream, dev, args.steps // per_graph, False)
        per_call = None
    else:
        local_ms, per_call = timed_steps(calls, stream, dev, args.steps, split=True)
    barrier()
    clocks.mark("t1")
    clk = clocks.stop()
    launches = (sum(p.launches for p in plans) - launches0) if graph is None else graph_launches * args.steps
    total_ms = reduce_max(local_ms, ws)
    ms_per_step = total_ms / args.steps
    nbytes = sum(w.min_bytes for w in wls)
    gbs = job_gbs(nbytes, ws, ms_per_step)
    elems = sum(w.P * w.N for w in wls) * ws / (ms_per_step * 1e-3)

    # spread: 20 more steps, each bracketed by its own events (outside the
    # timed region; only where a step is long enough that two event records
    # per step do not distort it)
    step_spread = None
    if graph is None and ms_per_step > 0.05:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(21)]
        evs[0].record(stream)
        for i in range(20):
            for c in calls:
                c()
            evs[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        per = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(20))
        step_spread = {"median": round(0.5 * (per[9] + per[10]), 5), "min": round(per[0], 5),
                       "max": round(per[-1], 5), "steps": 20}

    # roofline of the dominant kernel (the fused pass: one launch per call)
    launches_per_step = max(1, launches // args.steps)
    kernel_bytes = sum(kernel_bytes_of(p, w, args.mode) for p, w in zip(plans, wls))
    avg_launch_ms = local_ms / (args.steps * launches_per_step)
    achieved = (kernel_bytes / launches_per_step) / (avg_launch_ms * 1e-3) / 1e9
    # the kernel the library launches for these plans (its own dispatch rules)
    kernel_name = " / ".join(dict.fromkeys(p.kernel_name for p in plans))
    if args.mode == "rankorder":
        kernel_name += " (rank order)"
    traffic = None
    if args.mode == "fused" and launches_per_step == len(wls):
        per_launch = [ncu_traffic(w, args.kernel, w.min_bytes) for w in wls]
        if all(t is not None for t in per_launch):
            traffic = int(round(sum(per_launch) / len(per_launch)))
    roofline = {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": f"hbm_gbs of {peak_kind}", "traffic": traffic,
                "algorithmic_bytes_per_launch": kernel_bytes // launches_per_step,
                "launches_per_step": launches_per_step, "avg_launch_ms": round(avg_launch_ms, 4)}

    per_schedule = {}
    for j, (p, w) in enumerate(zip(plans, wls)):
        entry = {"workload": w.name, "schedule": schedule_name(w), "bytes_per_call": w.min_bytes,
                 "steps_per_call": p.traffic()[1]}
        if per_call is not None or len(wls) == 1:
            ms = per_call[j] / args.steps if per_call is not None else local_ms / args.steps
            g = w.min_bytes / (ms * 1e-3) / 1e9
            entry.update({"ms": round(ms, 5), "GBps": round(g, 1), "elems_per_s": round(w.P * w.N / (ms * 1e-3), 1),
                          "frac": round(g / peak, 4), "traffic": ncu_traffic(w, args.kernel, w.min_bytes)
                          if args.mode == "fused" else None})
        per_schedule[schedule_name(w)] = entry

    e2e = None
    if not args.no_e2e:
        with torch.cuda.stream(stream):
            e2e = e2e_leg(plans, wls, bufs, stream, dev, ws, args.e2e_steps)

    overlap = None
    if args.overlap:
        overlap = overlap_study(plans[0], bufs, w0, stream, tokens=args.overlap_tokens)
        overlap["allreduce_alone_ms"] = round(ms_per_step / len(wls), 4)
    sgd = sgd_study(plans[0], bufs, w0, stream) if args.sgd else None

    # alpha-beta model of each schedule on P real workers, at the Baidu
    # write-up's ~6 GB/s InfiniBand, with no latency and with 10 us per step:
    # one link per worker (every schedule on the same hardware), and for the
    # multi-ring also one link per ring
    def model_of(p, w):
        links = [1] + ([w.k] if w.topo == "multiring" and w.k > 1 else [])
        return {"steps": p.traffic()[1], "elements_sent_total": p.traffic()[0],
                **{f"links{L}": {"alpha0_s": round(p.cost(0.0, 1 / 6e9, L), 6),
                                 "alpha10us_s": round(p.cost(10e-6, 1 / 6e9, L), 6)} for L in links}}

    model = {"link_GBps": 6.0, "schedules": {schedule_name(w): model_of(p, w) for p, w in zip(plans, wls)}}

    for p in plans:
        p.close()
    del bufs, slab
    torch.cuda.empty_cache()

    configs = None
    if ws == 1 and not args.no_configs and args.workload == DEFAULT_WORKLOAD and not args.elems:
        configs = {}
        for name in SECONDARY:
            configs[name] = secondary_leg(ddl, name, dev, stream, peak, samples if oracle_legs else {})

    cpu = cpu_baseline(wls, samples) if oracle_legs else None
    if cpu is not None and configs:
        for name, c in configs.items():
            c["parity_sample"] = cpu["parity_sample"].get(name)

    if rank == 0:
        line = {"metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": w0.dtype, "data": "synthetic",
                "config": {"workload": args.workload if args.workload in SWEEPS else w0.name,
                           "schedules": [schedule_name(w) for w in wls], "P": w0.P, "N": w0.N,
                           "mode": args.mode, "kernel": args.kernel, "buckets": n_buckets,
                           "step": (f"one all-reduce under each of {len(wls)} schedules over the same buffers"
                                    if len(wls) > 1 else "one all-reduce"),
                           "bytes_per_step": nbytes,
                           "layout": "one slab (ddl_allreduce_slab)" if args.slab else "P separate buffers",
                           "launch": (f"CUDA graph replay, {per_graph} steps per graph" if args.graph
                                      else "one library call per all-reduce"),
                           "elems_per_s": round(elems, 1), "frac_of_hbm": round(gbs / ws / peak, 4),
                           "frac_of_nominal_hbm": round(gbs / ws / 7900.0, 4),
                           "step_ms_spread": step_spread,
                           "l2": (f"inputs {w0.P * w0.N * w0.esize / 1e9:.2f} GB per replica, larger than the "
                                  f"129 MB L2 (no flush needed)" if w0.P * w0.N * w0.esize > 129e6 else
                                  f"inputs {w0.P * w0.N * w0.esize / 1e6:.1f} MB fit in the 129 MB L2: back-to-back "
                                  f"steps run on a warm L2 (a latency measurement, not an HBM one)"),
                           "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU, P logical ranks"},
                "per_schedule": per_schedule, "clocks": clk, "gpu_launches": launches, "roofline": roofline,
                "e2e": e2e, "cpu_baseline": cpu, "configs": configs, "cluster_model": model, "overlap": overlap,
                "sgd": sgd, "kernel_src": kernel_hash()}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
