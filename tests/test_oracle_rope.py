"""Pins for the oracle's inverse RoPE + MXFP8 (CPU only).

* hand-worked rows (tests/golden/inv_rope_rows.json, each with its
  derivation): quarter turns in both pair layouts, a span at an offset, and
  the IEEE signs of zero of the rotation's sums;
* brute force on small random rows against the exact-rational checker
  (tests/exact_ref.py), both layouts, real cos/sin tables;
* special cases that reduce to other pinned operations: the zero angle is the
  MX quantiser of (B) applied to the input, and the fused call is its two
  steps composed.
"""
import json
import os
import random
import struct
from fractions import Fraction

import numpy as np
import pytest

import exact_ref as X
import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bf16_of(v) -> int:
    """bf16 bits of a small exactly representable number ("-0" allowed)."""
    if v == "-0":
        return 0x8000
    return struct.unpack("<I", struct.pack("<f", float(v)))[0] >> 16


def test_golden_inv_rope_rows():
    with open(os.path.join(GOLDEN, "inv_rope_rows.json")) as f:
        g = json.load(f)
    for row in g["rows"]:
        H, D, R = row["H"], row["D"], row["R"]
        x = np.array([bf16_of(v) for v in row["x"]], np.uint16).reshape(1, H, D)
        cs = np.array([[row["cos"]] * (R // 2) + [row["sin"]] * (R // 2)], np.float32)
        pos = np.zeros(1, np.int32)
        y = O.inv_rope_bf16(x, pos, cs, row["rope_off"], R, row["interleaved"])
        assert y[0].tolist() == [bf16_of(v) for v in row["y"]], row["name"]
        codes, scale = O.inv_rope_quant_mx(x, pos, cs, row["rope_off"], R, row["interleaved"])
        assert codes[0].tolist() == [int(c, 16) for c in row["codes"]], row["name"]
        assert scale[0].tolist() == [int(c, 16) for c in row["scale"]], row["name"]


def _cache(rng, P, R):
    ang = np.array([[rng.uniform(-40.0, 40.0) for _ in range(R // 2)] for _ in range(P)])
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


@pytest.mark.parametrize("H,D,rope_off,R,interleaved", [
    (1, 32, 0, 32, False), (2, 64, 32, 32, True), (3, 96, 16, 64, False), (1, 32, 8, 16, True),
])
def test_inv_rope_matches_exact_checker(H, D, rope_off, R, interleaved):
    rng = random.Random(H * 100 + D + R + interleaved)
    P, T = 5, 3
    cs = _cache(rng, P, R)
    pos = np.array([rng.randrange(P) for _ in range(T)], np.int32)
    vals = [[X.bf16_bits(Fraction(rng.gauss(0.0, 1.0) * (30.0 if rng.random() < 0.05 else 1.0)))
             for _ in range(H * D)] for _ in range(T)]
    o = np.array(vals, np.uint16).reshape(T, H, D)
    y = O.inv_rope_bf16(o, pos, cs, rope_off, R, interleaved)
    codes, scales = O.inv_rope_quant_mx(o, pos, cs, rope_off, R, interleaved)
    for t in range(T):
        want = X.inv_rope_row(vals[t], H, D, rope_off, R, interleaved, cs[pos[t]].tolist())
        assert y[t].tolist() == want, t
        for b in range(H * D // 32):
            sc, cb = X.mx_block(want[32 * b:32 * b + 32])
            assert scales[t, b] == sc and codes[t, 32 * b:32 * b + 32].tolist() == cb, (t, b)


def test_inv_rope_zero_angle_is_the_mx_quantiser():
    """cos = 1, sin = 0 leaves every value (the sign of a zero can change:
    -0 + +0 = +0); away from zeros the result is (B)'s MX quantiser of o."""
    w = synth.InvRopeWorkload("t", T=16, H=2, D=64, rope_off=32, rope_dim=32)
    o = w.o()
    o[o & 0x7FFF == 0] = 0x3F80
    cs = np.concatenate([np.ones((1, 16)), np.zeros((1, 16))], axis=1).astype(np.float32)
    pos = np.zeros(16, np.int32)
    for inter in (False, True):
        codes, scales = O.inv_rope_quant_mx(o, pos, cs, 32, 32, inter)
        want_c, want_s = O.quant_mx(o.reshape(16, -1))
        assert np.array_equal(codes, want_c) and np.array_equal(scales, want_s)


def test_inv_rope_fused_is_its_steps():
    w = synth.InvRopeWorkload("t", T=32, H=3, D=96, rope_off=32, rope_dim=64, P=64)
    o, pos, cs = w.o(), w.positions(), w.cos_sin()
    for inter in (False, True):
        codes, scales = O.inv_rope_quant_mx(o, pos, cs, 32, 64, inter)
        want_c, want_s = O.quant_mx(O.inv_rope_bf16(o, pos, cs, 32, 64, inter))
        assert np.array_equal(codes, want_c) and np.array_equal(scales, want_s)


def test_inv_rope_workload_inputs():
    """The synthetic workload's positions and cache: in range, the table's
    rows are cos/sin of p * base^(-2i/R) (position 0: cos 1, sin 0)."""
    w = synth.workloads()["inv_rope_mx"]
    pos, cs = w.positions(), w.cos_sin()
    assert pos.shape == (w.T,) and pos.min() >= 0 and pos.max() < w.P
    assert cs.shape == (w.P, w.rope_dim) and cs.dtype == np.float32
    assert np.all(cs[0, :32] == 1.0) and np.all(cs[0, 32:] == 0.0)
    assert np.allclose(cs[:, :32] ** 2 + cs[:, 32:] ** 2, 1.0, atol=1e-6)


# Two rotations from the o-projection workload whose sum lies so close to a
# bf16 rounding boundary that rounding x1*c + x2*s once (a fused multiply-add)
# gives the other bf16 neighbour than rounding the product and the sum apart:
# (x1, x2, cos, sin) as bf16 / binary32 bit patterns, and the two results.
CONTRACTION_CASES = [
    (0x3E8E, 0xBF05, 0x3F73BDEA, 0x3E9C8953, 0x3DD8, 0x3DD7),
    (0x3D8B, 0x3FB1, 0xBF7FB319, 0x3D465E5E, 0xBA58, 0xBA57),
]


def contraction_row():
    """One token, one head of 32 with the two cases as pairs 0 and 1."""
    o = np.zeros((1, 1, 32), np.uint16)
    cs = np.zeros((1, 32), np.float32)
    cs[0, :16] = 1.0
    for i, (x1, x2, c, s, _, _) in enumerate(CONTRACTION_CASES):
        o[0, 0, i], o[0, 0, 16 + i] = x1, x2
        cs[0, i] = np.array([c], np.uint32).view(np.float32)[0]
        cs[0, 16 + i] = np.array([s], np.uint32).view(np.float32)[0]
    return o, cs


def test_inv_rope_rounds_product_and_sum_apart():
    o, cs = contraction_row()
    y = O.inv_rope_bf16(o, np.zeros(1, np.int32), cs, 0, 32, False)
    want = X.inv_rope_row(o.reshape(-1).tolist(), 1, 32, 0, 32, False, cs[0].tolist())
    assert y[0].tolist() == want
    for i, (_, _, _, _, apart, fused) in enumerate(CONTRACTION_CASES):
        assert y[0, i] == apart and apart != fused
