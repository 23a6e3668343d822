"""Pins for the oracle's codecs, activation and mean square (CPU only).

Each oracle routine is compared with something other than itself: the
independent exact-rational checker (tests/exact_ref.py), library casts in
torch, the OCP bit layouts, or exhaustive enumeration.
"""
import math
import random
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact_ref as X
import oracle as O


def f32(u):
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def f32_bits(f):
    return struct.unpack("<I", struct.pack("<f", f))[0]


def random_finite_f32(rng, n, emin=-149, emax=127):
    """Random finite binary32 values spread over binades (and subnormals)."""
    out = []
    while len(out) < n:
        e = rng.randint(emin, emax)
        m = rng.getrandbits(23)
        if e < -126:
            u = rng.getrandbits(23)
            v = f32(u)
        else:
            v = f32(((e + 127) << 23) | m)
        if rng.random() < 0.5:
            v = -v
        if math.isfinite(v):
            out.append(v)
    return out


# ---------------------------------------------------------------------------
# bf16
# ---------------------------------------------------------------------------

def test_bf16_from_binary32_matches_torch_cast():
    """binary32 -> bf16 nearest-even equals torch's bfloat16 cast."""
    rng = random.Random(1)
    vals = random_finite_f32(rng, 200000)
    # exact ties (low 16 bits == 0x8000) with odd and even kept parts
    for hi in (0x3F80, 0x3F81, 0x0001, 0x7F7E, 0x7F7F, 0x8001):
        vals.append(f32((hi << 16) | 0x8000))
        vals.append(f32((hi << 16) | 0x7FFF))
        vals.append(f32((hi << 16) | 0x8001))
    vals = [v for v in vals if math.isfinite(v)]
    a = np.array(vals, dtype=np.float32)
    ours = O.bf16_from_float_n(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_from_double_matches_exact_rounding():
    """double -> bf16 is one rounding (no detour through binary32)."""
    rng = random.Random(2)
    cases = []
    for _ in range(3000):
        b = rng.randrange(0x0001, 0x7F7F)
        lo, hi = X.bf16_to_frac(b), X.bf16_to_frac(b + 1)
        mid = (lo + hi) / 2
        # the midpoint itself, and one double ulp either side of it
        m = float(mid)
        cases += [m, math.nextafter(m, 0), math.nextafter(m, math.inf)]
        cases.append(rng.uniform(float(lo), float(hi)))
    for v in cases:
        for s in (1, -1):
            want = X.bf16_bits(Fraction(s * v), neg_zero=s < 0)
            assert O.bf16_from_double(s * v) == want, (s * v)


def test_bf16_overflow_and_specials():
    assert O.bf16_from_double(3.0e38) == 0x7F62
    assert O.bf16_from_double(3.4e38) == 0x7F80          # rounds past the largest finite
    assert O.bf16_from_double(-1e300) == 0xFF80
    assert O.bf16_from_double(float("nan")) == 0x7FC0
    assert O.bf16_from_double(-0.0) == 0x8000
    assert O.bf16_from_double(2.0 ** -133) == 0x0001      # smallest subnormal
    assert O.bf16_from_double(2.0 ** -134) == 0x0000      # tie to even (zero)
    assert O.bf16_from_double(1.5 * 2.0 ** -134) == 0x0001


# ---------------------------------------------------------------------------
# E4M3
# ---------------------------------------------------------------------------

def test_e4m3_decode_matches_ocp_layout():
    for c in range(256):
        v = O.e4m3_to_double(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(v)
        else:
            assert Fraction(v) == X.E4M3_VALUE[c], hex(c)


def test_e4m3_ocp_table_facts():
    assert O.e4m3_to_double(0x7E) == 448.0                # largest finite
    assert O.e4m3_to_double(0x01) == 2.0 ** -9            # smallest subnormal
    assert O.e4m3_to_double(0x08) == 2.0 ** -6            # smallest normal
    assert O.e4m3_to_double(0x38) == 1.0
    assert O.e4m3_to_double(0x80) == 0.0 and math.copysign(1, O.e4m3_to_double(0x80)) < 0


def test_e4m3_roundtrip_all_codes():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert O.e4m3_from_float(O.e4m3_to_double(c)) == c, hex(c)


def test_e4m3_ties_saturation_and_specials():
    cases = [
        (1.0625, 0x38),          # tie between 1.0 (m=0) and 1.125 (m=1): even
        (1.1875, 0x3A),          # tie between 1.125 (m=1) and 1.25 (m=2): even
        (-1.1875, 0xBA),
        (2.0 ** -10, 0x00),      # half the smallest subnormal: tie to zero
        (3 * 2.0 ** -11, 0x01),
        (-(2.0 ** -11), 0x80),   # underflow keeps the sign
        (448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E),
        (-500.0, 0xFE), (float("inf"), 0x7E), (float("-inf"), 0xFE),
        (float("nan"), 0x7F), (-0.0, 0x80), (0.0, 0x00),
        (0.10009765625, 0x1D),   # 12.8 quanta of 2^-7 -> 13
    ]
    for v, c in cases:
        assert O.e4m3_from_float(v) == c, (v, hex(O.e4m3_from_float(v)), hex(c))


def test_e4m3_encode_matches_exact_rounding():
    rng = random.Random(3)
    vals = random_finite_f32(rng, 20000, emin=-14, emax=10)
    a = np.array(vals, dtype=np.float32)
    ours = O.e4m3_from_float_n(a)
    for v, c in zip(a.tolist(), ours.tolist()):
        assert c == X.e4m3_code(Fraction(v), v < 0 or (v == 0 and math.copysign(1, v) < 0)), v


def test_e4m3_encode_matches_torch_cast_in_range():
    """torch's float8_e4m3fn cast is nearest-even but not saturating, so
    compare on |v| < 448 only."""
    rng = random.Random(4)
    vals = [v for v in random_finite_f32(rng, 200000, emin=-20, emax=8) if abs(v) < 448]
    a = np.array(vals, dtype=np.float32)
    ours = O.e4m3_from_float_n(a)
    ref = torch.from_numpy(a).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------------------
# activation: exhaustive over every bf16 gate
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("act,name", [(O.ACT_SIGMOID, "sigmoid"), (O.ACT_SILU, "silu")])
def test_activation_exhaustive_against_decimal(act, name):
    ours = O.act_table(act)
    for g in range(65536):
        if not X.bf16_is_finite(g):
            continue
        want = X.act_exact(g, name)
        assert ours[g] == want, (name, hex(g), hex(int(ours[g])), hex(want))


def test_activation_specials():
    S, L = O.ACT_SIGMOID, O.ACT_SILU
    assert O.act_bf16(0x0000, S) == 0x3F00                # sigmoid(0) = 1/2
    assert O.act_bf16(0x0000, L) == 0x0000                # silu(0) = 0
    assert O.act_bf16(0x7F80, S) == 0x3F80 and O.act_bf16(0xFF80, S) == 0x0000
    assert O.act_bf16(0x7F80, L) == 0x7F80 and O.act_bf16(0xFF80, L) == 0x8000
    assert O.act_bf16(0x7FC0, S) == 0x7FC0 and O.act_bf16(0xFFC1, L) == 0x7FC0
    # sigmoid(-x) = 1 - sigmoid(x): check on values where both sides are exact
    # enough in bf16 (|x| <= 1 keeps both in [0.27, 0.73])
    for g in range(0x3C00, 0x3F80, 7):
        a = O.bf16_to_float([O.act_bf16(g, S)])[0]
        b = O.bf16_to_float([O.act_bf16(g | 0x8000, S)])[0]
        assert abs(float(a) + float(b) - 1.0) <= 2.0 ** -8


def test_activation_matches_torch_within_one_ulp():
    """torch's own bf16 sigmoid/silu (fp32 evaluation, then rounding) may
    differ from the correctly rounded value by at most one bf16 ulp where the
    result is a normal number and sigmoid(g) is too: torch's fp32 path
    flushes subnormal sigmoids (g below about -87.3) to zero, also inside its
    silu.  The decimal check above covers those gates."""
    g = np.arange(65536, dtype=np.uint16)
    gt = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16)
    gval = O.bf16_to_float(g)
    for act, fn in ((O.ACT_SIGMOID, torch.sigmoid), (O.ACT_SILU, torch.nn.functional.silu)):
        table = O.act_table(act)
        finite = (((g & 0x7F80) != 0x7F80) & (((table & 0x7F80) != 0) | ((table & 0x7FFF) == 0))
                  & ~(gval < -87.0))
        ours = table[finite].astype(np.int32)
        ref = fn(gt.float()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[finite]
        ref = ref.astype(np.int32)
        same_sign = (ours & 0x8000) == (ref & 0x8000)
        d = np.abs(ours - ref)
        assert np.all(d[same_sign] <= 1)


# ---------------------------------------------------------------------------
# mean square and r
# ---------------------------------------------------------------------------

def _rand_bf16_vec(rng, n, spread):
    out = []
    for _ in range(n):
        e = rng.randint(127 - spread, 127 + spread // 4)
        e = max(0, min(254, e))
        out.append((rng.getrandbits(1) << 15) | (e << 7) | rng.getrandbits(7))
    return out


@pytest.mark.parametrize("n", [1, 2, 3, 8, 40, 128, 1536])
def test_mean_square_matches_exact(n):
    rng = random.Random(n)
    for spread in (2, 20, 80, 200):
        for _ in range(15 if n > 200 else 40):
            xs = _rand_bf16_vec(rng, n, spread)
            want = X.mean_square(xs)
            got = O.mean_square(np.array(xs, dtype=np.uint16))
            assert Fraction(got) == want, (n, spread)


def test_mean_square_subnormals_and_zero():
    assert O.mean_square(np.zeros(8, np.uint16)) == 0.0
    xs = [0x0001, 0x0003, 0x8002, 0x0000]                 # bf16 subnormals
    assert Fraction(O.mean_square(np.array(xs, np.uint16))) == X.mean_square(xs)
    xs = [0x2000, 0x2080, 0xA100]                         # squares below 2^-126
    assert Fraction(O.mean_square(np.array(xs, np.uint16))) == X.mean_square(xs)
    assert math.isnan(O.mean_square(np.array([0x3F80, 0x7FC0], np.uint16)))
    assert math.isinf(O.mean_square(np.array([0x3F80, 0xFF80], np.uint16)))


def test_mean_square_is_order_independent():
    rng = random.Random(7)
    xs = _rand_bf16_vec(rng, 128, 60)
    ref = O.mean_square(np.array(xs, dtype=np.uint16))
    for _ in range(20):
        rng.shuffle(xs)
        assert O.mean_square(np.array(xs, dtype=np.uint16)) == ref


def test_rms_factor_matches_exact():
    rng = random.Random(8)
    for eps in (1e-6, 1e-5, 0.0, 1.0):
        for _ in range(300):
            ms = f32(((rng.randint(60, 200)) << 23) | rng.getrandbits(23))
            want = X.rms_factor(Fraction(ms), X.rn32(Fraction(eps)))
            assert Fraction(O.rms_factor(ms, eps)) == want


def test_rms_factor_closed_form_unit_mean_square():
    """ms = 1, eps = 1e-6: v = 1 + 2^-20 (1e-6 is 8.39 ulps of 2^-23),
    sqrt rounds to 1 + 2^-21, and 1/(1 + 2^-21) rounds to 1 - 2^-21."""
    assert O.rms_factor(1.0, 1e-6) == 1.0 - 2.0 ** -21


# ---------------------------------------------------------------------------
# E8M0
# ---------------------------------------------------------------------------

def test_e8m0_code_all_positive_bf16():
    for b in range(0x0001, 0x7F80):
        want = max(-127, min(127, X.floor_log2(X.bf16_to_frac(b)) - 8)) + 127
        assert O.e8m0_code(b) == want, hex(b)
    assert O.e8m0_code(0x0000) == 0
    assert O.e8m0_code(0x7F80) == 0xFF and O.e8m0_code(0x7FC0) == 0xFF
    assert O.e8m0_code(0x3F80) == 119                     # amax 1.0 -> 2^-8


def test_e8m0_block_max_lands_in_256_to_448():
    """With scale 2^(floor(log2 A) - 8), the block maximum scaled by 2^-e lies
    in [256, 512) and encodes to a code of magnitude 256..448, unless the
    exponent is clamped at -127 (amax below 2^-119)."""
    for b in range(0x0001, 0x0400):                       # amax < 2^-119: clamped
        assert O.e8m0_code(b) == 0
    for b in range(0x0400, 0x7F80, 3):                    # amax >= 2^-119
        e = O.e8m0_code(b) - 127
        scaled = float(X.bf16_to_frac(b)) * 2.0 ** (-e)
        assert 256.0 <= scaled < 512.0
        c = O.e4m3_from_float(scaled)
        assert 256.0 <= O.e4m3_to_double(c) <= 448.0
