"""Reader for the hand-written fixtures in tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def to_storage(values, dtype):
    a = np.array(values, dtype=np.float64)
    if dtype == "f16":
        h = a.astype(np.float16)
        assert np.all(h.astype(np.float64) == a), "fixture value not exact in binary16"
        return h.view(np.uint16)
    f = a.astype(np.float32)
    assert np.all(f.astype(np.float64) == a), "fixture value not exact in binary32"
    return f


def load_trace(name):
    params, inputs, states, final, moved, steps = {}, {}, {}, None, None, None
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "param":
                params[tok[1]] = tok[2]
            elif tok[0] == "input":
                inputs[int(tok[1])] = [float(v) for v in tok[2:]]
            elif tok[0] == "state":
                states.setdefault(int(tok[1]), {})[int(tok[2])] = [float(v) for v in tok[3:]]
            elif tok[0] == "final":
                final = [float(v) for v in tok[1:]]
            elif tok[0] == "moved":
                moved = int(tok[1])
            elif tok[0] == "steps":
                steps = int(tok[1])
    P, N = int(params["P"]), int(params["N"])
    dt = params["dtype"]
    cfg = dict(P=P, N=N, dtype=dt, topo=params["topo"], X=int(params.get("X", 0)),
               Y=int(params.get("Y", 0)), k=int(params.get("k", 1)))
    scale = float(np.float32(float(params["scale"])))
    ins = [to_storage(inputs[r], dt) for r in range(P)]
    sts = {s: [to_storage(v[r], dt) for r in range(P)] for s, v in states.items()}
    return cfg, scale, ins, sts, to_storage(final, dt), moved, steps


def load_buckets(name="buckets_hand.txt"):
    cases, expect = {}, {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "case":
                layers = None if tok[5] == "-" else [int(v) for v in tok[5].split(",")]
                cases[tok[1]] = dict(dtype=tok[2], N=int(tok[3]), bucket_bytes=int(tok[4]), layers=layers)
                expect[tok[1]] = []
            elif tok[0] == "bucket":
                expect[tok[1]].append((int(tok[2]), int(tok[3])))
    return cases, expect
