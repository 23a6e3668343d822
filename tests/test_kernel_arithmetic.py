"""Host-side proofs about arithmetic identities the CUDA kernels rely on
(exhaustive where the input set is finite; CPU only, exact rationals)."""
import struct
from fractions import Fraction

import exact_ref as X


def rn32(v: Fraction) -> Fraction:
    return X.rn32(v)


def test_scale_division_by_448_is_exact_for_every_bf16_amax():
    """The gated kernel forms scale = RN32(amax / 448) as q0 = RN(amax * r),
    e = RN(amax - q0 * 448) (one FMA), q = RN(e * r + q0) (one FMA) with the
    constant r = RN(1/448).  amax is a bf16 value, so all 32,640 positive
    finite patterns are checked against the IEEE quotient."""
    r = rn32(Fraction(1, 448))
    for b in range(1, 0x7F80):
        a = X.bf16_to_frac(b)
        q0 = rn32(a * r)
        e = rn32(a - q0 * 448)
        q = rn32(e * r + q0)
        assert q == rn32(a / 448), hex(b)


def test_markstein_quotient_on_ties():
    """q0 = RN(x * RN(1/d)) can miss an E4M3 tie that x / d hits exactly
    (x = 1.3671875, d = 7 gives 0.1953125); the FMA correction restores the
    IEEE quotient."""
    x, d = Fraction(1.3671875), Fraction(7)
    rd = rn32(1 / d)
    q0 = rn32(x * rd)
    assert q0 != x / d
    e = rn32(q0 * d - x)          # exact: the remainder fits binary32
    assert e == q0 * d - x
    q = rn32(q0 - e * rd)
    assert q == rn32(x / d) == Fraction(0.1953125)


def test_fastdiv_constants():
    """(umulhi(n, m) + n) >> l == n // d for the static kernel's divisors
    (chunks per row and head counts) over n < 2^31, spot-checked densely
    near multiples of d and exhaustively for small n."""
    import random
    rng = random.Random(3)
    for d in list(range(1, 300)) + [1024, 1536, 2048, 4095, 65535]:
        l = 0
        while (1 << l) < d:
            l += 1
        m = ((1 << 32) * ((1 << l) - d)) // d + 1
        assert m < (1 << 32)
        ns = list(range(0, 3000)) + [rng.randrange(0, 1 << 31) for _ in range(3000)]
        ns += [k * d + j for k in (1 << 20, (1 << 31) // d - 1) for j in (-1, 0, 1) if 0 <= k * d + j < (1 << 31)]
        for n in ns:
            assert ((((n * m) >> 32) + n) >> l) == n // d, (d, n)
