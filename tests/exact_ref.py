"""Independent exact-arithmetic restatement of the three operations.

Pure Python standard library (``fractions``, ``decimal``, ``struct``).  It
shares nothing with the C oracle: every rounding is done on exact rationals
by one generic round-to-nearest-even routine, square roots by integer square
root, and the gate activation by ``decimal`` at 60 significant digits.  It is
slow and meant for tiny inputs (1-4 rows) that pin the oracle.

Values are returned as bit patterns / codes so that comparisons are exact.
"""
from __future__ import annotations

import math
import struct
from decimal import Decimal, localcontext
from fractions import Fraction

HALF = Fraction(1, 2)


# ---------------------------------------------------------------------------
# generic binary rounding on exact rationals
# ---------------------------------------------------------------------------

def floor_log2(a: Fraction) -> int:
    """floor(log2(a)) for a > 0, exactly."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    # a in [2^(e-1), 2^(e+1)); fix up
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_rne(a: Fraction, p: int, emin: int) -> Fraction:
    """Nearest-even rounding of a >= 0 to p significant bits, gradual
    underflow below 2^emin (quantum 2^(emin-p+1) there).  No overflow check."""
    if a == 0:
        return Fraction(0)
    E = max(floor_log2(a), emin)
    q = Fraction(2) ** (E - p + 1)
    s = a / q
    n = s.numerator // s.denominator
    rem = s - n
    if rem > HALF or (rem == HALF and n % 2 == 1):
        n += 1
    return n * q


# ---------------------------------------------------------------------------
# formats
# ---------------------------------------------------------------------------

def f32_bits_to_frac(u: int) -> Fraction:
    f = struct.unpack("<f", struct.pack("<I", u))[0]
    assert math.isfinite(f)
    return Fraction(f)


def bf16_to_frac(b: int) -> Fraction:
    return f32_bits_to_frac((b & 0xFFFF) << 16)


def bf16_is_finite(b: int) -> bool:
    return (b & 0x7F80) != 0x7F80


def rn32(v: Fraction) -> Fraction:
    """IEEE binary32 round-to-nearest-even (finite results only)."""
    r = round_rne(abs(v), 24, -126)
    assert r < Fraction(2) ** 128, "binary32 overflow outside the checked domain"
    return r if v >= 0 else -r


def bf16_bits(v: Fraction, neg_zero: bool = False) -> int:
    """bf16 bit pattern of the nearest-even rounding of v (finite only)."""
    r = round_rne(abs(v), 8, -126)
    assert r < Fraction(2) ** 128
    sign = 0x8000 if (v < 0 or (v == 0 and neg_zero)) else 0
    if r == 0:
        return sign
    f = struct.unpack("<I", struct.pack("<f", float(r)))[0]
    assert Fraction(struct.unpack("<f", struct.pack("<I", f))[0]) == r
    return sign | (f >> 16)


def _e4m3_table():
    """Value of every finite E4M3 code, from the OCP OFP8 bit layout:
    sign | 4-bit exponent (bias 7) | 3-bit mantissa; exponent 0 subnormal;
    S.1111.111 is NaN (no infinities)."""
    tab = {}
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        if e == 0:
            v = Fraction(m, 8) * Fraction(2) ** -6
        else:
            v = (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        tab[c] = -v if s else v
    return tab


E4M3_VALUE = _e4m3_table()
E4M3_MAX = Fraction(448)


def e4m3_code(v: Fraction, negative: bool) -> int:
    """Saturating nearest-even E4M3 code of v; `negative` carries the sign
    (also for zero results)."""
    a = abs(v)
    if a >= E4M3_MAX:
        r = E4M3_MAX
    else:
        r = round_rne(a, 4, -6)
    sign = 0x80 if negative else 0
    for c in range(128):
        if c in E4M3_VALUE and E4M3_VALUE[c] == r:
            return sign | c
    raise AssertionError("no code for %s" % r)


# ---------------------------------------------------------------------------
# elementary steps
# ---------------------------------------------------------------------------

def sqrt_rn32(v: Fraction) -> Fraction:
    """Correctly rounded binary32 square root of v >= 0 (v normal binary32)."""
    if v == 0:
        return Fraction(0)
    E = floor_log2(v) // 2  # leading exponent of sqrt(v), up to one
    for Eg in (E - 1, E, E + 1):
        if Fraction(2) ** (2 * Eg) <= v < Fraction(2) ** (2 * Eg + 2):
            E = Eg
            break
    qexp = E - 23
    scaled = v / Fraction(2) ** (2 * qexp)  # sqrt(scaled) in [2^23, 2^24)
    n = math.isqrt(scaled.numerator // scaled.denominator)
    mid = (Fraction(n) + HALF) ** 2
    if scaled > mid or (scaled == mid and n % 2 == 1):
        n += 1
    return n * Fraction(2) ** qexp


def mean_square(xs) -> Fraction:
    fs = [bf16_to_frac(b) for b in xs]
    return rn32(sum((f * f for f in fs), Fraction(0)) / len(fs))


def rms_factor(ms: Fraction, eps: Fraction) -> Fraction:
    v = rn32(ms + eps)
    s = sqrt_rn32(v)
    return rn32(1 / s)


def act_exact(g: int, act: str) -> int:
    """bf16 of sigmoid(g) or silu(g) = g*sigmoid(g), correctly rounded, with
    60 significant decimal digits of working precision."""
    assert bf16_is_finite(g)
    x = bf16_to_frac(g)
    neg = (g & 0x8000) != 0
    if abs(x) > 200:
        # |x| > 200: e^-|x| < 2^-288, far below half a bf16 step anywhere
        if act == "sigmoid":
            return 0x3F80 if x > 0 else 0x0000
        return bf16_bits(x) if x > 0 else 0x8000
    with localcontext() as ctx:
        ctx.prec = 60
        dx = Decimal(x.numerator) / Decimal(x.denominator)
        sig = Decimal(1) / (Decimal(1) + (-dx).exp())
        val = sig if act == "sigmoid" else dx * sig
    fv = Fraction(val)
    return bf16_bits(fv, neg_zero=(act == "silu" and neg))


def act_table_exact(act: str):
    """act_exact over every finite bf16 pattern; None for inf/NaN patterns."""
    return [act_exact(g, act) if bf16_is_finite(g) else None for g in range(65536)]


# ---------------------------------------------------------------------------
# the three operations (finite inputs)
# ---------------------------------------------------------------------------

def gated_token(x_tok, gate_tok, weight, H, D, eps: float, act: str, act_tab=None,
                ms_given=None):
    """Operation (A) on one token: x_tok, gate_tok flat lists [H*D] of bf16
    bits, weight [D].  ms_given: None, or binary32 mean squares [H] to use in
    place of the exact ones.  Returns (y bits, codes, scale as Fraction)."""
    epsf = rn32(Fraction(eps))
    y = []
    for h in range(H):
        xs = x_tok[h * D:(h + 1) * D]
        ms = mean_square(xs) if ms_given is None else Fraction(float(ms_given[h]))
        r = rms_factor(ms, epsf)
        for d in range(D):
            xn = rn32(bf16_to_frac(xs[d]) * r)
            xnb = bf16_bits(xn, neg_zero=(xs[d] & 0x8000) != 0)
            u = bf16_bits(bf16_to_frac(xnb) * bf16_to_frac(weight[d]),
                          neg_zero=((xnb ^ weight[d]) & 0x8000) != 0)
            g = act_tab[gate_tok[h * D + d]] if act_tab else act_exact(gate_tok[h * D + d], act)
            y.append(bf16_bits(bf16_to_frac(u) * bf16_to_frac(g),
                               neg_zero=((u ^ g) & 0x8000) != 0))
    amax = max(abs(bf16_to_frac(b)) for b in y)
    scale = rn32(amax / 448)
    codes = []
    for b in y:
        neg = (b & 0x8000) != 0
        if amax == 0:
            codes.append(0x80 if neg else 0)
        else:
            codes.append(e4m3_code(rn32(bf16_to_frac(b) / scale), neg))
    return y, codes, scale


def rmsnorm_row(xs, w, eps: float):
    epsf = rn32(Fraction(eps))
    r = rms_factor(mean_square(xs), epsf)
    out = []
    for b, wb in zip(xs, w):
        xn = rn32(bf16_to_frac(b) * r)
        xnb = bf16_bits(xn, neg_zero=(b & 0x8000) != 0)
        out.append(bf16_bits(bf16_to_frac(xnb) * bf16_to_frac(wb),
                             neg_zero=((xnb ^ wb) & 0x8000) != 0))
    return out


def mx_block(yq):
    """E8M0 code and E4M3 codes of one 32-element block of bf16 bits."""
    amax = max(abs(bf16_to_frac(b)) for b in yq)
    if amax == 0:
        e = -127
    else:
        e = max(-127, min(127, floor_log2(amax) - 8))
    codes = [e4m3_code(bf16_to_frac(b) * Fraction(2) ** (-e), (b & 0x8000) != 0) for b in yq]
    return e + 127, codes


def static_quant(x_bits, descale: float):
    d = Fraction(descale)
    return [e4m3_code(rn32(bf16_to_frac(b) / d), (b & 0x8000) != 0) for b in x_bits]


def quant_row(y_bits):
    """Per-token quantisation of a bf16 row: (codes, scale)."""
    amax = max(abs(bf16_to_frac(b)) for b in y_bits)
    scale = rn32(amax / 448)
    codes = []
    for b in y_bits:
        neg = (b & 0x8000) != 0
        codes.append((0x80 if neg else 0) if amax == 0 else e4m3_code(rn32(bf16_to_frac(b) / scale), neg))
    return codes, scale


def gated_quant_row(x_bits, g_bits, act: str, act_tab=None):
    """y = bf16(x * bf16(act(g))) per element, then the per-token quantisation."""
    y = []
    for xb, gb in zip(x_bits, g_bits):
        g = act_tab[gb] if act_tab else act_exact(gb, act)
        y.append(bf16_bits(bf16_to_frac(xb) * bf16_to_frac(g), neg_zero=((xb ^ g) & 0x8000) != 0))
    codes, scale = quant_row(y)
    return y, codes, scale


def head_amax(x_bits):
    """max |x| over a head's values (finite inputs)."""
    return max(abs(bf16_to_frac(b)) for b in x_bits)


def dynamic_quant(x_bits_head):
    """descale = RN32(amax / 448) of the head, codes of x / descale (signed
    zeros for a zero head)."""
    d = rn32(head_amax(x_bits_head) / 448)
    if d == 0:
        return d, [0x80 if b & 0x8000 else 0 for b in x_bits_head]
    return d, [e4m3_code(rn32(bf16_to_frac(b) / d), (b & 0x8000) != 0) for b in x_bits_head]


# ---------------------------------------------------------------------------
# inverse RoPE (binary32 products and sums, IEEE signs of zero), then MX
# ---------------------------------------------------------------------------

def _signed(v: Fraction, neg: bool):
    """A value with the sign of zero kept: (v, negative)."""
    return (v, (v < 0) or (v == 0 and neg))


def _rn32_signed(x):
    v, neg = x
    r = rn32(v)
    return (r, (r < 0) or (r == 0 and neg))


def _mul32(a, b):
    return _rn32_signed(_signed(a[0] * b[0], a[1] != b[1]))


def _add32(a, b):
    v = a[0] + b[0]
    # an exact zero sum is -0 only when both addends are -0 (round to nearest)
    return _rn32_signed(_signed(v, a[1] and b[1]))


def _neg(a):
    return (-a[0], not a[1])


def _f32(x: float):
    import math
    return (Fraction(x), math.copysign(1.0, x) < 0)


def inv_rope_row(o_bits, H, D, rope_off, R, interleaved, cs):
    """One token: o_bits flat [H*D] bf16 bits; cs [R] binary32 cos then sin.
    Returns the bf16 bits of the rotated-back row."""
    y = list(o_bits)
    half = R // 2
    for h in range(H):
        for i in range(half):
            j1 = h * D + (rope_off + 2 * i if interleaved else rope_off + i)
            j2 = h * D + (rope_off + 2 * i + 1 if interleaved else rope_off + half + i)
            x1 = _signed(bf16_to_frac(o_bits[j1]), (o_bits[j1] & 0x8000) != 0)
            x2 = _signed(bf16_to_frac(o_bits[j2]), (o_bits[j2] & 0x8000) != 0)
            c, s = _f32(float(cs[i])), _f32(float(cs[half + i]))
            y1 = _add32(_mul32(x1, c), _mul32(x2, s))
            y2 = _add32(_mul32(x2, c), _neg(_mul32(x1, s)))
            y[j1] = bf16_bits(y1[0], neg_zero=y1[1])
            y[j2] = bf16_bits(y2[0], neg_zero=y2[1])
    return y
