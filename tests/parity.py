"""Comparison helpers for GPU-vs-oracle parity (test infrastructure).

Tolerance policy of the path (stated once, used by every parity test):
  * E8M0 scale codes and static-path (C) codes: bit-exact;
  * kv bf16 outputs of (B): bit-exact;
  * (A)/(B) E4M3 codes: identical except one-code differences (adjacent in
    value order, +-0 counted equal) on at most 1e-4 of the elements, the
    budget left for reduction-order effects;
  * per-token fp32 scales of (A): relative difference <= 1e-6;
  * dequantised values decode(code) * scale agree at atol = rtol = 1e-3 on
    every element outside the one-code set (the pages' own check).
The kernels are designed to meet these exactly; the helpers report the
observed counts so a test log shows how far from the budget a run was.
"""
from __future__ import annotations

import numpy as np

import oracle as O

CODE_FRAC_BUDGET = 1e-4
SCALE_RTOL = 1e-6


def _e4m3_table() -> np.ndarray:
    return np.array([O.e4m3_to_double(c) for c in range(256)], dtype=np.float64)


E4M3 = _e4m3_table()


def rank(codes: np.ndarray) -> np.ndarray:
    """Position of each E4M3 code in value order (+0 and -0 share rank 0)."""
    c = codes.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def compare_codes(got: np.ndarray, want: np.ndarray, budget: float = CODE_FRAC_BUDGET) -> dict:
    """Check E4M3 codes against the tolerance policy; return the counts."""
    got = np.asarray(got, dtype=np.uint8).reshape(-1)
    want = np.asarray(want, dtype=np.uint8).reshape(-1)
    assert got.shape == want.shape
    diff = got != want
    n_diff = int(diff.sum())
    if n_diff:
        r = np.abs(rank(got[diff]) - rank(want[diff]))
        assert int(r.max()) <= 1, "a code differs by more than one step: %s vs %s" % (
            got[diff][r > 1][:8], want[diff][r > 1][:8])
    assert n_diff <= budget * got.size, "%d of %d codes differ (budget %g)" % (
        n_diff, got.size, budget)
    return {"elements": int(got.size), "code_diffs": n_diff}


def compare_scales(got: np.ndarray, want: np.ndarray, rtol: float = SCALE_RTOL) -> dict:
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    want = np.asarray(want, dtype=np.float64).reshape(-1)
    both_nan = np.isnan(got) & np.isnan(want)
    ok = both_nan | (np.abs(got - want) <= rtol * np.abs(want)) | (got == want)
    assert ok.all(), "scales differ: got %s want %s" % (got[~ok][:4], want[~ok][:4])
    return {"scales": int(got.size), "scale_exact": int((got == want).sum())}


def compare_dequant(codes_got, scale_got, codes_want, scale_want) -> None:
    """decode(code) * scale within 1e-3 outside the one-code set."""
    cg = np.asarray(codes_got, dtype=np.uint8)
    cw = np.asarray(codes_want, dtype=np.uint8)
    same = rank(cg) == rank(cw)
    sg = np.asarray(scale_got, dtype=np.float64).reshape(-1, *([1] * (cg.ndim - 1)))
    sw = np.asarray(scale_want, dtype=np.float64).reshape(-1, *([1] * (cw.ndim - 1)))
    dg = E4M3[cg] * sg
    dw = E4M3[cw] * sw
    fin = np.isfinite(dw) & same
    assert np.allclose(dg[fin], dw[fin], atol=1e-3, rtol=1e-3)
