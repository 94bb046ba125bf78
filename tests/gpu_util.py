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
