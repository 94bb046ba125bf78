"""Helpers for the GPU tests: rank buffers on the device and comparisons."""
import numpy as np

import oracle
import synth


def torch_dtype(dtype):
    import torch
    return torch.float16 if dtype == "f16" else torch.float32


def to_numpy_bits(t):
    """Device tensor -> numpy in the oracle's storage form (float32 / uint16 bits)."""
    import torch
    if t.dtype == torch.float16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def from_numpy_bits(a, device):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).to(device).view(torch.float16)
    return torch.from_numpy(a.copy()).to(device)


def device_bufs_from_host(host, device):
    return [from_numpy_bits(h, device) for h in host]


def device_bufs_generated(w, device, pad_elems=0):
    """P rank buffers filled on the device by the seeded generator."""
    import torch
    bufs = []
    for r in range(w.P):
        t = torch.empty(w.N + pad_elems, dtype=torch_dtype(w.dtype), device=device)
        synth.fill_device(t.data_ptr(), w.N, w.seed, r, w.dist, w.sigma, w.dtype,
                          stream=torch.cuda.current_stream().cuda_stream)
        bufs.append(t[:w.N] if pad_elems else t)
    return bufs


def oracle_cfg(w):
    return oracle.Config(w.P, w.N, w.dtype, w.topo, k=w.k, X=w.X, Y=w.Y, bucket_bytes=w.bucket_bytes,
                         layers=w.layers, dims=w.dims)


def part_edges(lo, hi, m):
    """Positions where a split of [lo, hi) into m parts changes part (for
    choosing sample points near chunk edges)."""
    n = hi - lo
    base, rem = divmod(n, m)
    return [lo + i * base + min(i, rem) for i in range(m + 1)]


def edge_samples(w):
    """Element indices at and next to every bucket, slice and chunk edge."""
    cfg = oracle_cfg(w)
    edges = set()
    for lo, hi in oracle.buckets(cfg):
        if w.topo == "torus":
            for c0, c1 in zip(part_edges(lo, hi, w.X)[:-1], part_edges(lo, hi, w.X)[1:]):
                edges.update(part_edges(c0, c1, w.Y))
        elif w.topo == "torus_nd":
            level = [(lo, hi)]
            for D in w.dims:
                nxt = []
                for a, b in level:
                    e = part_edges(a, b, D)
                    edges.update(e)
                    nxt += list(zip(e[:-1], e[1:]))
                level = nxt
        elif w.topo == "multiring":
            for s0, s1 in zip(part_edges(lo, hi, w.k)[:-1], part_edges(lo, hi, w.k)[1:]):
                edges.update(part_edges(s0, s1, w.P))
        else:
            edges.update(part_edges(lo, hi, w.P))
    out = set()
    for e in edges:
        for d in (-9, -8, -5, -4, -3, -2, -1, 0, 1, 2, 3, 4, 7, 8):
            if 0 <= e + d < w.N:
                out.add(e + d)
    return np.array(sorted(out), dtype=np.int64)


def rankorder_margins(host, got_bits, scale, dtype):
    """Error of a rank-order result against the binary64 sum of the stored
    inputs (times the scale), normwise and element by element.

    host: P arrays of stored inputs (float32, or uint16 binary16 bits) at the
    elements of got_bits (the result in storage form).  Element-wise bound:
    the left fold of P binary32 values is within gamma_{P-1} * sum|x| of the
    exact sum (gamma_n = n u / (1 - n u), u = 2^-24; recursive summation,
    Higham, Accuracy and Stability of Numerical Algorithms, ch. 4); the
    multiply by the scale adds one rounding (u |result|); the binary64
    reference itself is within P 2^-53 sum|x|; for binary16 storage the result
    is rounded once more, by at most 2^-11 of its magnitude (2^-25 absolute
    below the binary16 normal range).  Returns (normwise relative error,
    largest element-wise |got - ref64| / bound)."""
    P = len(host)
    wide = [oracle.f16_to_f32(h).astype(np.float64) if dtype == "f16" else h.astype(np.float64) for h in host]
    ref = oracle.ref64(host, scale, dtype)
    got = (oracle.f16_to_f32(got_bits) if dtype == "f16" else got_bits).astype(np.float64)
    abs_sum = np.abs(np.stack(wide)).sum(axis=0) * abs(float(scale))
    u = 2.0 ** -24
    gamma = (P - 1) * u / (1 - (P - 1) * u)
    bound = gamma * abs_sum + u * (np.abs(ref) + gamma * abs_sum) + P * 2.0 ** -52 * abs_sum + 2.0 ** -149
    if dtype == "f16":
        bound = bound + np.maximum(2.0 ** -11 * (np.abs(ref) + bound), 2.0 ** -25)
    err = np.abs(got - ref)
    norm = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    return norm, float(np.max(err / bound))
