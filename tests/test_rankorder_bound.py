"""The element-wise error bound the rank-order GPU tests apply (CPU only).

A rank-order result is a binary32 left fold of the P stored values, times the
scale, rounded to the storage type.  The bound must hold for such a fold
(computed here with numpy's binary32 adds) and must reject plausible
mistakes: a rank left out, a rank added twice, a result rounded to binary16
twice over a coarse grid, a scale applied twice.
"""
import numpy as np

import oracle
from gpu_util import rankorder_margins


def _inputs(P, n, dtype, seed, sigma):
    rng = np.random.default_rng(seed)
    # wide magnitudes, so the fold's rounding is visible
    x = (rng.standard_normal((P, n)) * sigma * np.exp(rng.uniform(-6, 6, (P, n)))).astype(np.float32)
    if dtype == "f16":
        return [oracle.f32_to_f16(r) for r in x]
    return list(x)


def _rank_order_fold(host, scale, dtype, skip=None, twice=None):
    wide = [oracle.f16_to_f32(h) if dtype == "f16" else h for h in host]
    acc = np.array(wide[0], dtype=np.float32)
    for r in range(1, len(wide)):
        if r == skip:
            continue
        acc = (acc + wide[r]).astype(np.float32)
        if r == twice:
            acc = (acc + wide[r]).astype(np.float32)
    out = (acc * np.float32(scale)).astype(np.float32)
    return oracle.f32_to_f16(out) if dtype == "f16" else out


def test_bound_holds_for_a_binary32_left_fold():
    for dtype, sigma in (("f32", 1e-3), ("f16", 1e-2)):
        for P in (2, 16, 64, 256):
            host = _inputs(P, 5000, dtype, P, sigma)
            scale = float(np.float32(1.0 / P))
            norm, elem = rankorder_margins(host, _rank_order_fold(host, scale, dtype), scale, dtype)
            assert elem <= 1.0, (dtype, P, elem)
            assert norm <= (1e-6 if dtype == "f32" else 2e-3), (dtype, P, norm)


def test_bound_rejects_planted_mistakes():
    for dtype, sigma in (("f32", 1e-3), ("f16", 1e-2)):
        P = 16
        host = _inputs(P, 5000, dtype, 99, sigma)
        scale = float(np.float32(1.0 / P))
        for kw in (dict(skip=5), dict(twice=7)):
            _, elem = rankorder_margins(host, _rank_order_fold(host, scale, dtype, **kw), scale, dtype)
            assert elem > 1.0, (dtype, kw, elem)
        good = _rank_order_fold(host, scale, dtype)
        _, elem = rankorder_margins(host, _rank_order_fold(host, scale * scale, dtype), scale, dtype)
        assert elem > 1.0
        if dtype == "f32":
            # a second rounding on a grid 2^10 times coarser than binary32's
            coarse = oracle.f16_to_f32(oracle.f32_to_f16(good * np.float32(2.0 ** 20))) / np.float32(2.0 ** 20)
            _, elem = rankorder_margins(host, coarse.astype(np.float32), scale, dtype)
            assert elem > 1.0
