"""Element-wise comparison of GPU results with the oracle.

Rules (fp32 outputs within 1e-5 relative, bf16 within 1e-2, with a floor
per output kind where the fp32 error scales with something other than the
value itself, as noted beside each entry of TOL):
  * NaN must sit exactly where the oracle has NaN; +-inf must match exactly;
  * otherwise |g - o| <= rtol * max(|o|, floor) element by element;
  * integer results (indices, gathered bf16 values) are compared bit for bit.
"""
from __future__ import annotations

import numpy as np

# (rtol, floor) per output kind
TOL = {
    "f32": (1e-5, 1e-30),       # sums, softmax probabilities, rstd
    "mean": (1e-5, 0.1),        # LayerNorm mean: fp32 error scales with the row's spread
    "loss": (1e-5, 1.0),        # LSE - x_t: fp32 error scales with |LSE|, not with the loss
    "bf16": (1e-2, 1e-3),       # LayerNorm y after rounding to bf16
}


def assert_close(got, ref, kind: str = "f32", what: str = ""):
    rtol, floor = TOL[kind]
    g = np.asarray(got, dtype=np.float64)
    o = np.asarray(ref, dtype=np.float64)
    assert g.shape == o.shape, f"{what}: shape {g.shape} vs {o.shape}"
    gn, on = np.isnan(g), np.isnan(o)
    bad_nan = gn != on
    assert not bad_nan.any(), f"{what}: NaN mismatch at {np.argwhere(bad_nan)[:5].tolist()}"
    gi, oi = np.isinf(g), np.isinf(o)
    bad_inf = (gi | oi) & ~(gn | on) & (g != o)
    assert not bad_inf.any(), f"{what}: inf mismatch at {np.argwhere(bad_inf)[:5].tolist()}"
    fin = ~(gn | on | gi | oi)
    err = np.abs(g[fin] - o[fin])
    lim = rtol * np.maximum(np.abs(o[fin]), floor)
    if err.size and not (err <= lim).all():
        idx = np.argwhere(fin)[np.argmax(err / lim)]
        k = tuple(idx)
        raise AssertionError(f"{what}: worst at {list(k)}: gpu {g[k]!r} oracle {o[k]!r} "
                             f"(rel {abs(g[k] - o[k]) / max(abs(o[k]), floor):.3g} > {rtol})")


def assert_bits_equal(got, ref, what: str = ""):
    g, o = np.asarray(got), np.asarray(ref)
    assert g.shape == o.shape and g.dtype == o.dtype, f"{what}: {g.shape}/{g.dtype} vs {o.shape}/{o.dtype}"
    if g.dtype.kind == "f":
        g, o = g.view(np.uint8), o.view(np.uint8)
    neq = g != o
    assert not neq.any(), f"{what}: {int(neq.sum())} mismatches, first {np.argwhere(neq)[:5].tolist()}"


def bf16_nearest_bits(ref) -> np.ndarray:
    """bf16 bit patterns nearest (ties to even) to fp64 values, by way of fp32
    (the double rounding can move a value by at most one bf16 step)."""
    f = np.asarray(ref, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[np.isnan(f)] = 0x7FC0
    return r


def assert_bf16_within_steps(got_bits, ref, steps: int = 1, what: str = ""):
    """Non-negative bf16 results (uint16 bit patterns) within `steps` bf16
    steps of the nearest bf16 to the oracle's fp64 value; NaN where the oracle
    has NaN."""
    g = np.asarray(got_bits, dtype=np.uint16)
    o = np.asarray(ref, dtype=np.float64)
    assert g.shape == o.shape, f"{what}: shape {g.shape} vs {o.shape}"
    gn = (g & 0x7FFF) > 0x7F80
    on = np.isnan(o)
    bad = gn != on
    assert not bad.any(), f"{what}: NaN mismatch at {np.argwhere(bad)[:5].tolist()}"
    assert (o[~on] >= 0).all() and not (g[~gn] & 0x8000).any(), f"{what}: negative values"
    d = np.abs(g[~gn].astype(np.int64) - bf16_nearest_bits(o[~on]).astype(np.int64))
    if d.size and d.max() > steps:
        k = tuple(np.argwhere(~gn)[np.argmax(d)])
        raise AssertionError(f"{what}: worst at {list(k)}: gpu bits {int(g[k]):#06x} "
                             f"oracle {o[k]!r} ({int(d.max())} bf16 steps > {steps})")
