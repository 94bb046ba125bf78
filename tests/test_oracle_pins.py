"""Pins of the oracle against what the pages and the mathematics fix.

Each check below is chosen so that a plausible mistake in the oracle (a wrong
ring direction, a dropped rounding, a transposed grid, an off-by-one chunk
rule) fails at least one of them.  None compares the oracle with itself by
retyping its formula.
"""
import itertools
import math
import os
import zlib

import numpy as np
import pytest

import oracle
import synth
from golden_io import GOLDEN, load_buckets, load_trace

TRACES = ["ring3_n7_f32.txt", "torus2x2_n8_f32.txt", "ring3_n3_f16.txt", "torus2x2_n4_f16.txt"]


def _cfg(d, **kw):
    d = dict(d)
    d.update(kw)
    return oracle.Config(**d)


# --------------------------------------------------------------------------
# Hand traces (tests/golden)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", TRACES)
def test_hand_trace_final_and_counts(oracle_lib, name):
    cfgd, scale, ins, _, final, moved, steps = load_trace(name)
    cfg = _cfg(cfgd)
    bufs = [b.copy() for b in ins]
    m, s = oracle.emulate(cfg, bufs, scale)
    for r in range(cfg.P):
        assert np.array_equal(bufs[r], final), (name, r, bufs[r], final)
    assert (m, s) == (moved, steps)
    # the closed form is an independent witness of the same numbers
    assert np.array_equal(oracle.closed_form_full(cfg, ins, scale), final)


@pytest.mark.parametrize("name", ["ring3_n7_f32.txt", "torus2x2_n8_f32.txt"])
def test_hand_trace_intermediate_states(oracle_lib, name):
    cfgd, scale, ins, states, _, _, _ = load_trace(name)
    cfg = _cfg(cfgd)
    assert states
    for s, expect in states.items():
        bufs = [b.copy() for b in ins]
        oracle.emulate(cfg, bufs, scale, stop_after=s)
        for r in range(cfg.P):
            assert np.array_equal(bufs[r], expect[r]), (name, s, r, bufs[r], expect[r])


def test_hand_bucket_tables(oracle_lib):
    cases, expect = load_buckets()
    for name, c in cases.items():
        cfg = oracle.Config(P=2, N=c["N"], dtype=c["dtype"], topo="ring", bucket_bytes=c["bucket_bytes"],
                            layers=c["layers"])
        assert oracle.buckets(cfg) == expect[name], name


def test_resnet101_buckets_tensor_counts(oracle_lib):
    """25 MiB reverse-layer buckets of the ResNet-101 gradient: the packing
    rule gives 7 buckets of 14/12/39/54/54/54/87 tensors (output side first)."""
    w = synth.WORKLOADS["multiring64_resnet101"]
    cfg = oracle.Config(w.P, w.N, w.dtype, w.topo, k=w.k, bucket_bytes=w.bucket_bytes, layers=w.layers)
    bk = oracle.buckets(cfg)
    off = np.concatenate([[0], np.cumsum(w.layers)])
    counts = [int(np.sum((off[:-1] >= b) & (off[:-1] < e))) for b, e in bk]
    assert counts == [14, 12, 39, 54, 54, 54, 87]
    assert bk[0][1] == w.N and bk[-1][0] == 0
    assert all(bk[i][0] == bk[i + 1][1] for i in range(len(bk) - 1))
    for b, e in bk[:-1]:
        assert (e - b) * 4 >= 25 * 2 ** 20


def test_resnet_tensor_tables():
    assert (len(synth.RESNET50), sum(synth.RESNET50)) == (161, 25_557_032)
    assert (len(synth.RESNET101), sum(synth.RESNET101)) == (314, 44_549_160)


# --------------------------------------------------------------------------
# Exact sums: integer-valued fp32 inputs in [-1000, 1000] add exactly in any
# order for P <= 64 (|partial sums| < 2^24), so every schedule must give the
# brute-force int64 total.
# --------------------------------------------------------------------------

def _schedules(P):
    out = [dict(topo="ring")]
    phi = sum(1 for c in range(1, max(P, 2)) if math.gcd(c, P) == 1) if P > 1 else 1
    for k in sorted({1, 2, min(3, phi), phi}):
        if 1 <= k <= phi:
            out.append(dict(topo="multiring", k=k))
    for X in range(1, P + 1):
        if P % X == 0:
            out.append(dict(topo="torus", X=X, Y=P // X))
    return out


@pytest.mark.parametrize("P", [1, 2, 3, 4, 6, 8, 16])
def test_exact_integer_sums_all_schedules(oracle_lib, P):
    rng = np.random.default_rng(100 + P)
    for N in [1, 2, 3, P - 1 if P > 1 else 1, P, P + 1, 37, 100]:
        for sched in _schedules(P):
            for bucket_bytes in [0, 12]:
                cfg = oracle.Config(P=P, N=N, dtype="f32", bucket_bytes=bucket_bytes, **sched)
                ints = rng.integers(-1000, 1001, size=(P, N))
                bufs = [ints[r].astype(np.float32) for r in range(P)]
                moved, steps = oracle.emulate(cfg, bufs, 1.0)
                total = ints.sum(axis=0).astype(np.float32)
                for r in range(P):
                    assert np.array_equal(bufs[r], total), (P, N, sched, bucket_bytes, r)


def test_exact_integer_sums_p64_multiring(oracle_lib):
    rng = np.random.default_rng(7)
    P, N = 64, 1000
    cfg = oracle.Config(P=P, N=N, dtype="f32", topo="multiring", k=4, bucket_bytes=1024)
    ints = rng.integers(-1000, 1001, size=(P, N))
    bufs = [ints[r].astype(np.float32) for r in range(P)]
    oracle.emulate(cfg, bufs, 1.0)
    total = ints.sum(axis=0)
    assert np.all(np.abs(total) < 2 ** 24)
    for r in range(P):
        assert np.array_equal(bufs[r], total.astype(np.float32))


def test_ref64_exact_on_integers(oracle_lib):
    rng = np.random.default_rng(3)
    ints = rng.integers(-1000, 1001, size=(5, 50))
    bufs = [ints[r].astype(np.float32) for r in range(5)]
    assert np.array_equal(oracle.ref64(bufs, 0.25), ints.sum(axis=0) * 0.25)


# --------------------------------------------------------------------------
# Brute force over every rank's contribution (P <= 4, tiny N): a one-hot input
# (1 at one rank and element, 0 elsewhere) must reach exactly that element of
# every rank, scaled once, and nothing else.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("P", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_brute_force_one_hot(oracle_lib, P, dtype):
    scale = 0.5
    one = np.float16(1).view(np.uint16) if dtype == "f16" else np.float32(1)
    half = np.float16(0.5).view(np.uint16) if dtype == "f16" else np.float32(0.5)
    npdt = np.uint16 if dtype == "f16" else np.float32
    for N in [1, 2, 3, 5, 7]:
        for sched in _schedules(P):
            for src, i in itertools.product(range(P), range(N)):
                cfg = oracle.Config(P=P, N=N, dtype=dtype, **sched)
                bufs = [np.zeros(N, dtype=npdt) for _ in range(P)]
                bufs[src][i] = one
                oracle.emulate(cfg, bufs, scale)
                expect = np.zeros(N, dtype=npdt)
                expect[i] = half
                for r in range(P):
                    assert np.array_equal(bufs[r], expect), (P, N, sched, src, i, r)


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------

def _wide_random(rng, P, N, dtype):
    """Values of widely varying magnitude, so that the order of the adds shows
    in the rounded result."""
    x = rng.standard_normal((P, N)) * np.exp2(rng.integers(-12, 13, size=(P, N)))
    if dtype == "f16":
        return [x[r].astype(np.float16).view(np.uint16) for r in range(P)]
    return [x[r].astype(np.float32) for r in range(P)]


CASES = [
    dict(P=5, N=103, topo="ring"),
    dict(P=8, N=257, topo="ring", bucket_bytes=100),
    dict(P=16, N=1000, topo="multiring", k=2),
    dict(P=9, N=301, topo="multiring", k=5, bucket_bytes=400),
    dict(P=16, N=999, topo="torus", X=4, Y=4),
    dict(P=12, N=500, topo="torus", X=4, Y=3, bucket_bytes=300),
    dict(P=12, N=500, topo="torus", X=3, Y=4),
    dict(P=32, N=777, topo="torus", X=8, Y=4),
    dict(P=6, N=4, topo="torus", X=3, Y=2),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_emulation_equals_closed_form_and_ranks_identical(oracle_lib, case, dtype):
    rng = np.random.default_rng(zlib.crc32(repr((sorted(case.items()), dtype)).encode()))
    cfg = oracle.Config(dtype=dtype, **case)
    ins = _wide_random(rng, cfg.P, cfg.N, dtype)
    bufs = [b.copy() for b in ins]
    scale = float(np.float32(1.0 / cfg.P))
    oracle.emulate(cfg, bufs, scale)
    for r in range(1, cfg.P):
        assert np.array_equal(bufs[r], bufs[0])
    assert np.array_equal(oracle.closed_form_full(cfg, ins, scale), bufs[0])


def _py_fold(x_rows, order, inner, groups, f16_hops):
    """A third, independent fold in numpy float32 arithmetic (power check for
    the tests above: feeding it a wrong order must change the result)."""
    def rnd(v):
        return np.float32(np.float16(v)) if f16_hops else v
    outs = []
    for row in x_rows:
        outer = None
        for g in range(groups):
            acc = np.float32(row[order[g * inner]])
            for h in range(1, inner):
                last = groups == 1 and h == inner - 1
                acc = np.float32(acc + np.float32(row[order[g * inner + h]]))
                acc = acc if last else rnd(acc)
            outer = acc if g == 0 else (np.float32(outer + acc) if g == groups - 1 else rnd(np.float32(outer + acc)))
        outs.append(outer)
    return np.array(outs, dtype=np.float32)


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[4]])
def test_third_witness_and_wrong_orders_detected(oracle_lib, case):
    rng = np.random.default_rng(11)
    cfg = oracle.Config(dtype="f32", **case)
    ins = _wide_random(rng, cfg.P, cfg.N, "f32")
    got = oracle.closed_form_full(cfg, ins, 1.0)
    x = np.stack(ins, axis=1)
    same = differ_rev = differ_shift = 0
    for i in range(cfg.N):
        order, inner, groups = oracle.fold_order(cfg, i)
        v = _py_fold(x[i:i + 1], order, inner, groups, False)[0]
        same += v.tobytes() == got[i].tobytes()
        rev = _py_fold(x[i:i + 1], order[::-1].copy(), inner, groups, False)[0]
        differ_rev += rev.tobytes() != got[i].tobytes()
        sh = _py_fold(x[i:i + 1], np.roll(order, 1), inner, groups, False)[0]
        differ_shift += sh.tobytes() != got[i].tobytes()
    assert same == cfg.N
    # a reversed ring direction or an off-by-one start changes many results
    assert differ_rev > cfg.N // 4 and differ_shift > cfg.N // 4


def test_fold_orders_ring_and_torus_by_hand(oracle_lib):
    # ring P=3, N=7: chunks [0,3) [3,5) [5,7) start at ranks 0, 1, 2
    cfg = oracle.Config(P=3, N=7, topo="ring")
    assert [oracle.fold_order(cfg, i)[0].tolist() for i in (0, 2, 3, 4, 5, 6)] == \
        [[0, 1, 2], [0, 1, 2], [1, 2, 0], [1, 2, 0], [2, 0, 1], [2, 0, 1]]
    # 2x2 torus, N=8: (c, d) = (0,0) (0,1) (1,0) (1,1) at elements 0, 2, 4, 6
    cfg = oracle.Config(P=4, N=8, topo="torus", X=2, Y=2)
    assert [oracle.fold_order(cfg, i)[0].tolist() for i in (0, 2, 4, 6)] == \
        [[0, 1, 2, 3], [2, 3, 0, 1], [1, 0, 3, 2], [3, 2, 1, 0]]
    assert oracle.fold_order(cfg, 0)[1:] == (2, 2)
    # 3x2 torus (X=3, Y=2), N=6: row chunks of 2, sub-chunks of 1
    cfg = oracle.Config(P=6, N=6, topo="torus", X=3, Y=2)
    assert oracle.fold_order(cfg, 3)[0].tolist() == [4, 5, 3, 1, 2, 0]   # c=1, d=1
    # multi-ring P=5, k=2: slice 1 uses ring order t*2 mod 5 = 0,2,4,1,3
    cfg = oracle.Config(P=5, N=10, topo="multiring", k=2)
    assert oracle.ring_strides(5, 2) == [1, 2]
    assert oracle.fold_order(cfg, 5)[0].tolist() == [0, 2, 4, 1, 3]       # slice 1, chunk 0
    assert oracle.fold_order(cfg, 6)[0].tolist() == [2, 4, 1, 3, 0]       # slice 1, chunk 1


# --------------------------------------------------------------------------
# Traffic and steps
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", CASES)
def test_traffic_is_2_p_minus_1_n(oracle_lib, case):
    cfg = oracle.Config(dtype="f32", **case)
    moved, steps = oracle.traffic(cfg)
    assert moved == 2 * (cfg.P - 1) * cfg.N
    nb = len(oracle.buckets(cfg))
    if cfg.topo == "torus":
        assert steps == nb * (2 * (cfg.X - 1) + 2 * (cfg.Y - 1))
    else:
        assert steps == nb * 2 * (cfg.P - 1)


def test_page3_traffic_figure(oracle_lib):
    """300M parameters (1.2 GB fp32 gradient): each GPU sends and receives
    about 2.4 GB (Baidu write-up, the language-model example)."""
    for P in (40, 16):
        moved, steps = oracle.traffic(oracle.Config(P=P, N=300_000_000))
        per_rank_gb = moved * 4 / P / 1e9
        assert per_rank_gb == pytest.approx(2 * (P - 1) / P * 1.2)
        assert abs(per_rank_gb - 2.4) / 2.4 < 0.07
    moved, _ = oracle.traffic(oracle.Config(P=4096, N=300_000_000))
    assert moved * 4 / 4096 / 1e9 == pytest.approx(2.4, rel=1e-3)
    # the torus spends fewer steps than a ring of the same size
    _, ring_steps = oracle.traffic(oracle.Config(P=16, N=1000))
    _, torus_steps = oracle.traffic(oracle.Config(P=16, N=1000, topo="torus", X=4, Y=4))
    assert (ring_steps, torus_steps) == (30, 12)


def test_cost_model_closed_forms_and_page3_figure(oracle_lib):
    """alpha-beta cost from the emulation's own message lists.
    Baidu write-up, the 300M-parameter language model: a 1.2 GB gradient over
    ~6 GB/s InfiniBand takes about 2.4 GB / 6 GB/s = 400 ms per iteration."""
    beta = 1 / 6e9
    t40 = oracle.cost(oracle.Config(P=40, N=300_000_000), 0.0, beta)
    assert t40 == pytest.approx(2 * 39 / 40 * 1.2e9 / 6e9)        # 0.39 s
    assert abs(t40 - 0.400) / 0.400 < 0.03
    assert oracle.cost(oracle.Config(P=4000, N=300_000_000), 0.0, beta) == pytest.approx(0.4, rel=1e-3)
    # closed forms (n divisible): ring 2(P-1)(a + n/P e b); torus 2(X-1)(a + n/X e b) + 2(Y-1)(a + n/XY e b)
    a, b, n = 5e-6, 1e-10, 96_000
    assert oracle.cost(oracle.Config(P=16, N=n), a, b) == pytest.approx(30 * (a + n / 16 * 4 * b))
    assert oracle.cost(oracle.Config(P=16, N=n, topo="torus", X=4, Y=4), a, b) == \
        pytest.approx(6 * (a + n / 4 * 4 * b) + 6 * (a + n / 16 * 4 * b))
    # multi-ring: one link per ring (links = k) halves the bandwidth term;
    # one shared link keeps the ring's
    assert oracle.cost(oracle.Config(P=16, N=n, topo="multiring", k=2), a, b, links=2) == \
        pytest.approx(30 * (a + n / 32 * 4 * b))
    assert oracle.cost(oracle.Config(P=16, N=n, topo="multiring", k=2), a, b, links=1) == \
        pytest.approx(30 * (a + n / 16 * 4 * b))
    # fp16 halves the bandwidth term
    assert oracle.cost(oracle.Config(P=8, N=n, dtype="f16"), 0.0, b) == pytest.approx(14 * n / 8 * 2 * b)
    # the torus keeps the ring's bandwidth term, 2(X-1)/X + 2(Y-1)/XY = 2(P-1)/P
    # (both bandwidth-optimal), and cuts the steps from 30 to 12
    ring = oracle.Config(P=16, N=n)
    torus = oracle.Config(P=16, N=n, topo="torus", X=4, Y=4)
    assert oracle.cost(torus, 0.0, b) == pytest.approx(oracle.cost(ring, 0.0, b))
    assert oracle.cost(torus, 1e-3, 0.0) == pytest.approx(12e-3)
    assert oracle.cost(ring, 1e-3, 0.0) == pytest.approx(30e-3)
    # ring and torus send one message per worker per step: extra links change nothing
    assert oracle.cost(ring, a, b, links=4) == oracle.cost(ring, a, b, links=1)
    assert oracle.cost(torus, a, b, links=4) == oracle.cost(torus, a, b, links=1)
    with pytest.raises(Exception):
        oracle.cost(ring, a, b, links=0)


def _load_cost_cases():
    out = []
    with open(os.path.join(GOLDEN, "cost_multiring4_k2_n10.txt")) as fh:
        for line in fh:
            tok = line.split()
            if tok and tok[0] == "case":
                out.append((tok[2], int(tok[3]), int(tok[4]), int(tok[5]), int(tok[6])))
    return out


@pytest.mark.parametrize("topo,k,links,steps,elems", _load_cost_cases())
def test_cost_model_hand_worked_shared_link(oracle_lib, topo, k, links, steps, elems):
    """The P = 4, k = 2 multi-ring of tests/golden/cost_multiring4_k2_n10.txt,
    worked out by hand: with one link per worker a step costs its busiest
    worker's summed messages, with a link per ring its largest message."""
    cfg = oracle.Config(P=4, N=10, topo=topo, k=k)
    assert oracle.cost(cfg, 1.0, 0.0, links=links) == steps
    assert oracle.cost(cfg, 0.0, 1.0, links=links) == elems * 4


# --------------------------------------------------------------------------
# Special cases that reduce to a simpler schedule or a plain operation
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_special_cases(oracle_lib, dtype):
    rng = np.random.default_rng(5)
    scale = float(np.float32(1 / 3))
    # P = 1: out = round(x * scale)
    ins = _wide_random(rng, 1, 50, dtype)
    bufs = [ins[0].copy()]
    oracle.emulate(oracle.Config(P=1, N=50, dtype=dtype), bufs, scale)
    if dtype == "f16":
        expect = (oracle.f16_to_f32(ins[0]) * np.float32(scale)).astype(np.float32)
        expect = expect.astype(np.float16).view(np.uint16)
    else:
        expect = (ins[0] * np.float32(scale)).astype(np.float32)
    assert np.array_equal(bufs[0], expect)
    # torus X=1 == ring of Y; torus Y=1 == ring of X; multi-ring k=1 == ring
    for P, other in [(6, dict(topo="torus", X=1, Y=6)), (6, dict(topo="torus", X=6, Y=1)),
                     (7, dict(topo="multiring", k=1))]:
        for bucket_bytes in (0, 40):
            ins = _wide_random(rng, P, 123, dtype)
            a = [b.copy() for b in ins]
            b = [b.copy() for b in ins]
            oracle.emulate(oracle.Config(P=P, N=123, dtype=dtype, bucket_bytes=bucket_bytes), a, scale)
            oracle.emulate(oracle.Config(P=P, N=123, dtype=dtype, bucket_bytes=bucket_bytes, **other), b, scale)
            assert all(np.array_equal(a[r], b[r]) for r in range(P))


def test_invalid_configurations_rejected(oracle_lib):
    with pytest.raises(oracle.OracleError):
        oracle.traffic(oracle.Config(P=6, N=10, topo="torus", X=4, Y=2))
    with pytest.raises(oracle.OracleError):
        oracle.traffic(oracle.Config(P=16, N=10, topo="multiring", k=9))   # phi(16) = 8
    with pytest.raises(oracle.OracleError):
        oracle.traffic(oracle.Config(P=4, N=10, layers=[3, 3]))
    with pytest.raises(oracle.OracleError):
        oracle.traffic(oracle.Config(P=4, N=0))


# --------------------------------------------------------------------------
# binary16 conversion, against independent implementations
# --------------------------------------------------------------------------

def test_f16_widening_exhaustive(oracle_lib):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _narrow_check(pats):
    mine = oracle.f32_to_f16(pats.view(np.float32))
    f = pats.view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all((mine[nan] & 0x7C00) == 0x7C00) and np.all((mine[nan] & 0x3FF) != 0)


def test_f16_narrowing_structured_vs_numpy(oracle_lib):
    """Every sign, exponent and top-11-bit mantissa prefix (2^20 prefixes)
    combined with the low-12-bit patterns that decide rounding (exact tie,
    just above and below a tie, all ones) and random ones, against numpy's
    float32 -> float16 conversion (round to nearest even, subnormals kept).
    The tie bit of every binary16 quantum lies in the prefix or is bit 12."""
    rng = np.random.default_rng(1)
    lows = np.concatenate([[0x000, 0x001, 0x7FF, 0x800, 0x801, 0xFFF], rng.integers(0, 4096, 10)])
    prefix = np.arange(1 << 20, dtype=np.uint32) << np.uint32(12)
    for low in lows:
        _narrow_check(prefix | np.uint32(low))


@pytest.mark.slow
@pytest.mark.skipif(not __import__("os").environ.get("DDL_SLOW_TESTS"), reason="set DDL_SLOW_TESTS=1")
def test_f16_narrowing_exhaustive_vs_numpy(oracle_lib):
    """All 2^32 binary32 patterns (about two minutes)."""
    step = 1 << 26
    base = np.arange(step, dtype=np.uint32)
    for lo in range(0, 1 << 32, step):
        _narrow_check(base + np.uint32(lo))


def test_f16_narrowing_vs_compiler_float16(oracle_lib, tmp_path):
    """A second independent witness: the C compiler's _Float16 conversion, on
    a strided sample of every binary32 pattern plus all values near binary16
    rounding boundaries."""
    import subprocess
    src = tmp_path / "h.c"
    src.write_text(
        "#include <stdint.h>\n#include <string.h>\n"
        "void conv(const uint32_t* in, uint16_t* out, long n){for(long i=0;i<n;++i){float f;"
        "memcpy(&f,&in[i],4);_Float16 h=(_Float16)f;memcpy(&out[i],&h,2);}}\n")
    so = tmp_path / "h.so"
    try:
        subprocess.check_call(["gcc", "-O1", "-shared", "-fPIC", "-o", str(so), str(src)])
    except (subprocess.CalledProcessError, FileNotFoundError):
        pytest.skip("compiler without _Float16")
    import ctypes
    lib = ctypes.CDLL(str(so))
    pats = np.arange(0, 1 << 32, 4099, dtype=np.uint64).astype(np.uint32)
    # every binary16 midpoint, and its two binary32 neighbours
    h = np.arange(0x7C00, dtype=np.uint32).astype(np.uint16)
    mids = ((h.view(np.float16).astype(np.float64)[:-1] + h.view(np.float16).astype(np.float64)[1:]) / 2)
    m32 = mids.astype(np.float32).view(np.uint32)
    pats = np.concatenate([pats, m32, m32 + 1, m32 - 1, m32 | 0x80000000]).astype(np.uint32)
    out = np.empty(pats.size, dtype=np.uint16)
    lib.conv(ctypes.c_void_p(pats.ctypes.data), ctypes.c_void_p(out.ctypes.data), ctypes.c_long(pats.size))
    mine = oracle.f32_to_f16(pats.view(np.float32))
    nan = np.isnan(pats.view(np.float32))
    assert np.array_equal(mine[~nan], out[~nan])


# --------------------------------------------------------------------------
# The input generator: host and workload sanity (device equality is a GPU test)
# --------------------------------------------------------------------------

def test_generator_statistics_and_counter_access():
    x = synth.draw_rank(123, 5, 200_000, "normal", 1e-3)
    assert abs(float(x.mean())) < 1e-5 and abs(float(x.std()) - 1e-3) < 2e-5
    assert np.max(np.abs(x)) <= 6e-3
    i = synth.draw_rank(1, 0, 100_000, "int1000")
    assert i.min() == -1000 and i.max() == 1000 and np.all(i == np.round(i))
    # counter based: any window equals the same window of the full draw
    assert np.array_equal(synth.draw_rank(9, 3, 50, "normal", 0.1, start=1000),
                          synth.draw_rank(9, 3, 1050, "normal", 0.1)[1000:])
    h = synth.draw_rank(9, 3, 1000, "normal", 1e-2, "f16")
    assert h.dtype == np.uint16
    # SplitMix64 published first output for seed 0 (state 0 + gamma)
    assert int(synth._mix(np.array([0x9E3779B97F4A7C15], dtype=np.uint64))[0]) == 0xE220A8397B1DCDAF


# --------------------------------------------------------------------------
# n-D torus (generalising the 2D torus of the Sony page's "2D-Torus
# All-reduce" to the multi-level rings of "[论文解读] PowerAI DDL")
# --------------------------------------------------------------------------

ND_CASES = [
    dict(P=8, N=77, dims=[2, 2, 2]),
    dict(P=12, N=500, dims=[2, 3, 2], bucket_bytes=600),
    dict(P=64, N=1001, dims=[4, 4, 4]),
    dict(P=24, N=333, dims=[2, 3, 2, 2]),
    dict(P=16, N=100, dims=[4, 1, 4]),
]


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("dims,other", [([4, 4], dict(topo="torus", X=4, Y=4)), ([16], dict(topo="ring")),
                                        ([3, 4, 1], dict(topo="torus", X=3, Y=4)), ([1, 12], dict(topo="ring")),
                                        ([12, 1, 1], dict(topo="ring")), ([4, 1, 3], dict(topo="torus", X=4, Y=3))])
def test_nd_torus_reduces_to_torus_and_ring(oracle_lib, dtype, dims, other):
    P = int(np.prod(dims))
    rng = np.random.default_rng(P * 7 + len(dims))
    for bucket_bytes in (0, 300):
        ins = _wide_random(rng, P, 257, dtype)
        a = [b.copy() for b in ins]
        b = [b.copy() for b in ins]
        ma = oracle.emulate(oracle.Config(P=P, N=257, dtype=dtype, topo="torus_nd", dims=dims,
                                          bucket_bytes=bucket_bytes), a, 1 / P)
        mb = oracle.emulate(oracle.Config(P=P, N=257, dtype=dtype, bucket_bytes=bucket_bytes, **other), b, 1 / P)
        assert ma == mb
        assert all(np.array_equal(a[r], b[r]) for r in range(P))


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("case", ND_CASES)
def test_nd_torus_emulation_equals_closed_form(oracle_lib, case, dtype):
    rng = np.random.default_rng(zlib.crc32(repr((sorted(case.items()), dtype)).encode()))
    cfg = oracle.Config(dtype=dtype, topo="torus_nd", **case)
    ins = _wide_random(rng, cfg.P, cfg.N, dtype)
    bufs = [b.copy() for b in ins]
    oracle.emulate(cfg, bufs, 1 / cfg.P)
    for r in range(1, cfg.P):
        assert np.array_equal(bufs[r], bufs[0])
    assert np.array_equal(oracle.closed_form_full(cfg, ins, 1 / cfg.P), bufs[0])


@pytest.mark.parametrize("case", ND_CASES)
def test_nd_torus_exact_sums_traffic_steps(oracle_lib, case):
    rng = np.random.default_rng(3)
    cfg = oracle.Config(topo="torus_nd", **case)
    ints = rng.integers(-1000, 1001, size=(cfg.P, cfg.N))
    bufs = [ints[r].astype(np.float32) for r in range(cfg.P)]
    moved, steps = oracle.emulate(cfg, bufs, 1.0)
    for r in range(cfg.P):
        assert np.array_equal(bufs[r], ints.sum(axis=0).astype(np.float32))
    nb = len(oracle.buckets(cfg))
    assert moved == 2 * (cfg.P - 1) * cfg.N
    assert steps == nb * sum(2 * (d - 1) for d in case["dims"])


@pytest.mark.parametrize("dims", [[2, 2], [2, 1, 2], [1, 2, 2], [2, 2, 1], [4], [1, 1, 1, 3]])
def test_nd_torus_brute_force_one_hot(oracle_lib, dims):
    P = int(np.prod(dims))
    for dtype in ("f32", "f16"):
        one = np.float16(1).view(np.uint16) if dtype == "f16" else np.float32(1)
        half = np.float16(0.5).view(np.uint16) if dtype == "f16" else np.float32(0.5)
        npdt = np.uint16 if dtype == "f16" else np.float32
        for N in (1, 3, 7):
            for src, i in itertools.product(range(P), range(N)):
                cfg = oracle.Config(P=P, N=N, dtype=dtype, topo="torus_nd", dims=dims)
                bufs = [np.zeros(N, dtype=npdt) for _ in range(P)]
                bufs[src][i] = one
                oracle.emulate(cfg, bufs, 0.5)
                expect = np.zeros(N, dtype=npdt)
                expect[i] = half
                assert all(np.array_equal(b, expect) for b in bufs), (dims, dtype, N, src, i)


def test_nd_torus_2x2x2_fold_order_by_hand(oracle_lib):
    """2x2x2 cube, N=8: each element is its own chunk tuple.  Element 5 has
    chunks (c0, c1, c2) = (1, 0, 1) (halves of 8, then of 4, then of 2).  Its
    fold visits x_k = (c_k + g_k) mod 2, g_0 fastest, rank = x0 + 2 x1 + 4 x2:
    ranks 5, 4, 7, 6, 1, 0, 3, 2, grouped ((5+4)+(7+6)) + ((1+0)+(3+2))."""
    cfg = oracle.Config(P=8, N=8, topo="torus_nd", dims=[2, 2, 2])
    assert oracle.fold_order(cfg, 5)[0].tolist() == [5, 4, 7, 6, 1, 0, 3, 2]
    assert oracle.fold_order(cfg, 0)[0].tolist() == [0, 1, 2, 3, 4, 5, 6, 7]
    # E = 2^24: nested groups give (E+1 -> E) + (1+1) = E+2, then + 0; a flat
    # left fold over the same order would give ((E+1)+1)+1 -> E
    E = 16777216.0
    vals = np.zeros((8, 8), dtype=np.float32)
    vals[5, 5], vals[4, 5], vals[7, 5], vals[6, 5] = E, 1, 1, 1
    bufs = [vals[r].copy() for r in range(8)]
    oracle.emulate(cfg, bufs, 1.0)
    assert bufs[0][5] == E + 2 and bufs[3][5] == E + 2


def test_nd_torus_invalid_dims(oracle_lib):
    for dims in ([3, 3], [0, 8], [2, 2, 2, 1, 1]):
        with pytest.raises(oracle.OracleError):
            oracle.traffic(oracle.Config(P=8, N=10, topo="torus_nd", dims=dims))


# --------------------------------------------------------------------------
# Momentum SGD after the all-reduce
# --------------------------------------------------------------------------

def test_sgd_exact_dyadic_values(oracle_lib):
    """Values that are short binary fractions make every product and sum
    exact, so the result must equal the rational arithmetic exactly:
    g = mean of the ranks' gradients, d = g + wd p, v = mu v + d, p = p - lr v."""
    from fractions import Fraction as F
    P, N = 4, 16
    rng = np.random.default_rng(9)
    grads = [(rng.integers(-64, 65, N) / 8).astype(np.float32) for _ in range(P)]
    p0 = (rng.integers(-32, 33, N) / 4).astype(np.float32)
    v0 = (rng.integers(-32, 33, N) / 16).astype(np.float32)
    params = [p0.copy() for _ in range(P)]
    moms = [v0.copy() for _ in range(P)]
    lr, mu, wd = 0.125, 0.5, 0.25
    inputs = [g.copy() for g in grads]
    oracle.sgd(oracle.Config(P, N), grads, params, moms, 0.25, lr, mu, wd)
    for i in range(N):
        g = F(1, 4) * sum(F(float(inputs[r][i])) for r in range(P))   # the mean gradient
        assert all(F(float(grads[r][i])) == g for r in range(P))       # stored on every rank
        d = g + F(wd) * F(float(p0[i]))
        v = F(mu) * F(float(v0[i])) + d
        p = F(float(p0[i])) - F(lr) * v
        for r in range(P):
            assert F(float(moms[r][i])) == v and F(float(params[r][i])) == p


def test_sgd_matches_torch_optimizer(oracle_lib):
    """torch.optim.SGD (momentum, weight decay) on the oracle's all-reduced
    gradient: an independent implementation; it may fuse a multiply-add, so
    agreement is to within a couple of binary32 roundings."""
    torch = pytest.importorskip("torch")
    P, N = 3, 2000
    rng = np.random.default_rng(4)
    grads = [rng.standard_normal(N).astype(np.float32) for _ in range(P)]
    p0 = rng.standard_normal(N).astype(np.float32)
    params = [p0.copy() for _ in range(P)]
    moms = [np.zeros(N, dtype=np.float32) for _ in range(P)]
    cfg = oracle.Config(P, N, topo="ring")
    lr, mu, wd = 0.05, 0.9, 1e-4
    g_ref = [g.copy() for g in grads]
    oracle.emulate(cfg, g_ref, 1.0 / 3)
    oracle.sgd(cfg, grads, params, moms, 1.0 / 3, lr, mu, wd)
    w = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.SGD([w], lr=lr, momentum=mu, weight_decay=wd)
    w.grad = torch.from_numpy(g_ref[0].copy())
    opt.step()
    got = w.detach().numpy()
    assert np.allclose(params[0], got, rtol=4e-7, atol=1e-7)
    assert np.array_equal(grads[0], g_ref[0])
    # lr = 0 leaves the parameters alone; mu = 0 with no momentum buffer is d
    params2 = [p0.copy() for _ in range(P)]
    grads2 = [g.copy() for g in g_ref]
    oracle.sgd(oracle.Config(P, N), grads2, params2, None, 1.0, 0.0, 0.0, 0.0)
    assert all(np.array_equal(p, p0) for p in params2)
