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


def _e4m3(v: Fraction) -> int:
    return X.e4m3_code(v, v < 0)


def _bf16_values_near_midpoints(s: Fraction, rng, n: int):
    """bf16 numerators y whose quotient y / s lies on or next to an E4M3
    rounding boundary (midpoints between neighbouring codes, and 448), plus
    uniformly drawn magnitudes up to 448 s."""
    codes = sorted(v for c, v in X.E4M3_VALUE.items() if c < 0x7F)
    mids = [(a + b) / 2 for a, b in zip(codes, codes[1:])] + [Fraction(448)]
    out = []
    for _ in range(n):
        if rng.random() < 0.7:
            m = mids[rng.randrange(len(mids))]
        else:
            m = Fraction(rng.uniform(2.0 ** -12, 448.0))
        if m * s >= X.bf16_to_frac(0x7F7F):
            continue
        b = X.bf16_bits(m * s)
        b += rng.choice((-1, 0, 0, 1)) if (b & 0x7FFF) > 1 else 0
        b |= 0x8000 if rng.random() < 0.5 else 0
        out.append(b)
    return out


def test_token_quotient_residual_is_exact_above_2_to_minus_60():
    """The per-token quantiser computes RN32(y / s) as q0 = RN(-y * -RN(1/s)),
    e = RN(q0 s - y) (one FMA), q = RN(q0 - e RN(1/s)), with y and s first
    multiplied by 2^64 when s < 2^-60.  Emulated on exact rationals (subnormal
    binary32 results included), the codes equal e4m3(RN32(y / s)) for scales
    across the whole range, near every E4M3 rounding boundary."""
    import random
    rng = random.Random(17)
    for e in list(range(-149, -120, 4)) + list(range(-100, 120, 9)) + [-61, -60, -59]:
        s = rn32(Fraction(2) ** e * Fraction(rng.uniform(1.0, 2.0)))
        if s == 0:
            continue
        sc, k = (s * Fraction(2) ** 64, Fraction(2) ** 64) if s < Fraction(2) ** -60 else (s, 1)
        nrs = -rn32(1 / sc)
        for yb in _bf16_values_near_midpoints(s, rng, 150):
            y = X.bf16_to_frac(yb) if (yb & 0x7F80) != 0x7F80 else None
            if y is None or abs(y) > 448 * s * 2:
                continue
            ny = -y * k
            q0 = rn32(ny * nrs)
            r = rn32(q0 * sc + ny)
            q = rn32(r * nrs + q0)
            want = rn32(y / s)
            got_code = X.e4m3_code(q, q < 0 or (q == 0 and (yb & 0x8000) != 0))
            want_code = X.e4m3_code(want, want < 0 or (want == 0 and (yb & 0x8000) != 0))
            assert got_code == want_code, (e, hex(yb))


def test_static_quotient_fast_path_range():
    """The static quantiser takes the same reciprocal-plus-FMA quotient for
    descales 2^-92 <= d <= 2^126, after clamping |x| to RU_bf16(512 d); its
    codes equal e4m3(RN32(x / d)) at both ends of that range."""
    import random
    rng = random.Random(23)
    for e in (-92, -91, -80, -40, 0, 40, 100, 125, 126):
        d = rn32(Fraction(2) ** e * Fraction(rng.uniform(1.0, 2.0)))
        if d > Fraction(2) ** 126:
            d = Fraction(2) ** 126
        nrd = -rn32(1 / d)
        T = X.round_rne(512 * d, 8, -126)
        if T < 512 * d:
            T = T + Fraction(2) ** (X.floor_log2(T) - 7)
        for xb in _bf16_values_near_midpoints(d, rng, 150) + [0x7F7F, 0xFF7F, 0x0001, 0x8000]:
            x = X.bf16_to_frac(xb)
            xc = max(-T, min(T, x))
            nx = -xc
            q0 = rn32(nx * nrd)
            r = rn32(q0 * d + nx)
            q = rn32(r * nrd + q0)
            want = rn32(x / d) if abs(x / d) < Fraction(2) ** 128 else (448 if x > 0 else -448)
            neg = (xb & 0x8000) != 0
            assert X.e4m3_code(q, neg) == X.e4m3_code(Fraction(want), neg), (e, hex(xb))


def test_token_quotient_exact_ties_need_the_2_to_minus_60_rescale():
    """Exact E4M3 ties y / s = midpoint, with scales of short mantissa: with
    the rescale taken only below 2^-126 the residual underflows and one tie is
    lost (s = 7 * 2^-123, y = 0x005B: y / s = 13/1024 rounds to even, while the
    uncorrected q0 lies above the tie); with the rescale below 2^-60 every tie
    is kept."""
    from fractions import Fraction as F
    codes = sorted(v for c, v in X.E4M3_VALUE.items() if c < 0x7F)
    mids = [(a + b) / 2 for a, b in zip(codes, codes[1:])]

    def misses(threshold):
        bad = []
        for e in range(-125, -40, 2):
            for mant in (F(9, 8), F(7, 4), F(11, 8), F(3, 2), F(13, 8), F(5, 4)):
                s = F(2) ** e * mant
                k = F(2) ** 64 if s < threshold else 1
                nrs = -rn32(1 / (s * k))
                for m in mids:
                    y = m * s
                    if X.round_rne(y, 8, -126) != y:
                        continue
                    q0 = rn32(-y * k * nrs)
                    r = rn32(q0 * s * k - y * k)
                    q = rn32(r * nrs + q0)
                    if X.e4m3_code(q, False) != X.e4m3_code(rn32(y / s), False):
                        bad.append((e, mant, m))
        return bad

    assert misses(F(2) ** -126) == [(-121, F(7, 4), F(13, 1024))]
    assert misses(F(2) ** -60) == []


# ---------------------------------------------------------------------------
# the mean square: device sum of squares, emulated operation by operation
# ---------------------------------------------------------------------------

def _two_sum(a, b):
    s = rn32(a + b)
    bb = rn32(s - a)
    return s, rn32(rn32(a - rn32(s - bb)) + rn32(b - bb))


def _fast_two_sum(a, b):
    s = rn32(a + b)
    return s, rn32(b - rn32(s - a))


def _df_add(a, b):
    s, e = _two_sum(a[0], b[0])
    return _fast_two_sum(s, rn32(e + rn32(a[1] + b[1])))


def _sumsq2(values):
    """One packed lane of the device accumulator on exact rationals."""
    s = c = Fraction(0)
    for x in values:
        q = x * x
        t = rn32(q + s)                      # mixed-precision FMA
        nz = rn32(s - t)
        a = rn32(s - rn32(t + nz))
        b = rn32(q + nz)                     # mixed-precision FMA
        c = rn32(c + rn32(a + b))
        s = t
    return s, c


def _kahan(values):
    """One packed lane of an ordinary Kahan sum of squares (the earlier
    accumulator), for comparison."""
    s = cn = Fraction(0)
    for x in values:
        y = rn32(x * x + cn)
        t = rn32(s + y)
        cn = rn32(y - rn32(t - s))
        s = t
    return s, cn


def _device_head(xs, head, lane_sum=None):
    """Double-float S of one head of 128 values as the staged kernel forms it
    for D = 128 (four threads of four 8-element chunks): thread j = 4 head + i
    reads chunk (c + j / 2) % 4 at step c into chain c % 2, each chain with
    two packed lanes (even / odd elements); the chains meet in one df_add and
    the four threads in an xor butterfly."""
    lane_sum = lane_sum or _sumsq2
    parts = []
    for i in range(4):
        j = 4 * head + i
        chunks = [xs[32 * i + 8 * c: 32 * i + 8 * c + 8] for c in range(4)]
        order = [chunks[(c + j // 2) % 4] for c in range(4)]
        chains = []
        for ch in (order[0] + order[2], order[1] + order[3]):
            e, o = lane_sum(ch[0::2]), lane_sum(ch[1::2])
            chains.append(_df_add(_fast_two_sum(*e), _fast_two_sum(*o)))
        parts.append(_df_add(chains[0], chains[1]))
    for m in (1, 2):
        parts = [_df_add(parts[i], parts[i ^ m]) for i in range(4)]
    return parts[0]


def _single_chain_head(xs, head, lane_sum):
    """The earlier layout: one chain per thread over the four rotated chunks."""
    parts = []
    for i in range(4):
        j = 4 * head + i
        chunks = [xs[32 * i + 8 * c: 32 * i + 8 * c + 8] for c in range(4)]
        seg = sum((chunks[(c + j // 2) % 4] for c in range(4)), [])
        e, o = lane_sum(seg[0::2]), lane_sum(seg[1::2])
        parts.append(_df_add(_fast_two_sum(*e), _fast_two_sum(*o)))
    for m in (1, 2):
        parts = [_df_add(parts[i], parts[i ^ m]) for i in range(4)]
    return parts[0]


def _ms_uncertain(S, n, ms, err):
    h, l = S
    if not (Fraction(2) ** -100 <= ms <= Fraction(2) ** 120):
        return False
    rd = rn32(rn32(h - ms * n) + l)           # the FMA residual is exact
    half = Fraction(2) ** (X.floor_log2(ms) - 24) * n
    tol = rn32(err + rn32(abs(rd) * Fraction(2) ** -22))
    near = abs(rn32(abs(rd) - half)) <= tol
    if ms == Fraction(2) ** X.floor_log2(ms) and rd < 0:
        near |= abs(rn32(-rd - half / 2)) <= tol
    return near


def test_mean_square_is_decided_or_flagged():
    """For heads of 128 values (the staged kernel's layout and bound),
    including heavy outliers and the head that exposed an ordinary Kahan sum,
    the binary32 mean square from the device double-float either equals
    RN32(S / 128) of the exact S or is flagged for the double-double path, by
    either of the two flag tests the kernels use."""
    import numpy as np
    import synth
    k, adds = 8, 5
    rel = Fraction((k * k + 4 * adds + 16)) * Fraction(2) ** -48
    rng = np.random.default_rng(4)
    heads = []
    x = synth.bf16_normal(11, 528, 700 * 32 * 128, outlier_p=0.01,
                          outlier_scale=60.0).reshape(700, 32, 128)
    heads.append(x[551, 29])                                   # lost by plain Kahan
    heads += [x[t, h] for t, h in zip(rng.integers(0, 700, 60), rng.integers(0, 32, 60))]
    y = synth.bf16_normal(12, 9, 40 * 128, sigma=1.0, outlier_p=0.2, outlier_scale=1e4)
    heads += list(y.reshape(40, 128))
    heads.append(np.full(128, 0x3FC0, np.uint16))              # constant head: exact S
    z = synth.bf16_normal(13, 9, 60 * 128, sigma=0.3, mean=1.5).reshape(60, 128)
    heads += list(z)                                           # narrow range: exact sums, ties
    flagged = certified = 0
    for n_head, hx in enumerate(heads):
        xs = [X.bf16_to_frac(int(b)) for b in hx]
        S_exact = sum((v * v for v in xs), Fraction(0))
        head = 29 if n_head == 0 else n_head % 32
        S = _device_head(xs, head)
        ms = rn32(rn32(S[0] + S[1]) / 128)
        err = rn32(S[0] * rel + 128 * Fraction(2) ** -149)
        # the staged kernel's test: RN32 at both ends of the error interval
        probe = S[0] != 0 and rn32(S[0] + rn32(S[1] + err)) != rn32(S[0] + rn32(S[1] - err))
        # the other kernels' test: the residual's distance to a boundary
        near = _ms_uncertain(S, 128, ms, err)
        # the exactness certificate (smallest nonzero exponent against S)
        emin = min(((int(b) >> 7) & 0xFF) for b in hx if int(b) & 0x7FFF)
        E = X.floor_log2(S[0]) + 127
        if emin >= 60 and 2 * emin >= E + 95 + 2:
            certified += 1
            assert S[0] + S[1] == S_exact
        elif probe or near:
            flagged += 1
        if not probe or not near:
            assert ms == rn32(S_exact / 128)
        if n_head == 0:   # an ordinary Kahan sum (one chain per thread) misses it by one ulp
            K = _single_chain_head(xs, head, _kahan)
            assert rn32(rn32(K[0] + K[1]) / 128) != ms
    assert flagged <= 3 and certified >= 50


def _resolve_exact(S, n, ms):
    """The kernels' binary32 resolve of RN32(S / n) for an exact double-float S."""
    h, l = S
    for _ in range(4):
        r1 = rn32(h - ms * n)                       # FMA, exact
        up = X.f32_bits_to_frac(_bits(ms) + 1)
        dn = X.f32_bits_to_frac(_bits(ms) - 1) if ms > 0 else Fraction(0)
        hu = rn32(rn32(rn32(up - ms) / 2) * n)
        hd = rn32(rn32(rn32(ms - dn) / 2) * n)
        du = rn32(rn32(r1 - hu) + l)
        dl = rn32(rn32(r1 + hd) + l)
        odd = _bits(ms) & 1
        if du > 0 or (du == 0 and odd):
            ms = up
        elif ms > 0 and (dl < 0 or (dl == 0 and odd)):
            ms = dn
        else:
            break
    return ms


def _bits(v: Fraction) -> int:
    return struct.unpack("<I", struct.pack("<f", float(v)))[0]


def test_binary32_resolve_of_exact_sums():
    """For exact double-float sums S (up to 48 significant bits, including
    exact ties of S / n) and row lengths n that are not powers of two, the
    binary32 resolve steps any start within two ulps to RN32(S / n)."""
    import random
    rng = random.Random(31)
    for n in (1536, 40, 96, 120, 512, 16384):
        for _ in range(300):
            e = rng.randrange(-20, 40)
            S = Fraction(rng.getrandbits(47) | (1 << 47), 1 << 47) * Fraction(2) ** e
            if rng.random() < 0.3:                  # an exact tie of S / n
                q = rn32(S / n)
                ulp = Fraction(2) ** (X.floor_log2(q) - 23)
                S = (q + ulp / 2) * n
                if X.round_rne(S, 48, -1000) != S:
                    continue
            h = rn32(S)
            l = rn32(S - h)
            assert h + l == S
            want = rn32(S / n)
            for k in (-2, -1, 0, 1, 2):
                start = X.f32_bits_to_frac(_bits(want) + k)
                assert _resolve_exact((h, l), n, start) == want, (n, S, k)


def _ms_int(bits, log2n):
    """The kernels' integer mean square, step by step: squares as integers
    m^2 4^(e - emin), their sum rounded to binary32 at scale
    2^(2(emin - 134) - log2n); None when the exponents span too much."""
    nz = [b for b in bits if b & 0x7FFF]
    if not nz:
        return Fraction(0)
    e1 = lambda b: max((b >> 7) & 0xFF, 1)
    emin, emax = min(map(e1, nz)), max(map(e1, nz))
    if 2 * (emax - emin) > 98:
        return None
    acc = 0
    for b in nz:
        m = (b & 0x7F) | (0x80 if b & 0x7F80 else 0)
        acc += (m * m) << (2 * (e1(b) - emin))
    base = 2 * (emin - 134) - log2n
    msb = acc.bit_length() - 1
    eres = msb + base
    if eres > 127:
        return None  # infinity
    q = max(eres - 23, -149)
    sh = q - base
    if sh <= 0:
        M = acc << -sh
    else:
        M, rem, half = acc >> sh, acc & ((1 << sh) - 1), 1 << (sh - 1)
        if rem > half or (rem == half and M & 1):
            M += 1
    return M * Fraction(2) ** q


def test_integer_mean_square_is_the_rounding_of_the_exact_sum():
    """The integer path equals RN32(S / 2^k) of the exact sum on heads with
    wide exponent spreads, subnormals, zeros and exact ties."""
    import random
    rng = random.Random(41)
    cases = 0
    for _ in range(400):
        n = rng.choice((8, 16, 128))
        lo = rng.randrange(1, 200)
        hi = min(254, lo + rng.randrange(0, 50))
        sub = 0.05 if lo < 40 else 0.0                       # subnormals with small exponents
        bits = []
        for _ in range(n):
            r = rng.random()
            if r < 0.1:
                bits.append(0)
            elif r < 0.1 + sub:
                bits.append(rng.randrange(1, 0x80))          # subnormal
            else:
                bits.append((rng.randrange(lo, hi + 1) << 7) | rng.randrange(0, 128))
        log2n = n.bit_length() - 1
        got = _ms_int(bits, log2n)
        if got is None:
            continue
        S = sum((X.bf16_to_frac(b) ** 2 for b in bits), Fraction(0))
        assert got == X.round_rne(S / n, 24, -126), (bits, log2n)
        cases += 1
    for hx in TIE_HEADS_HOST:
        S = sum((X.bf16_to_frac(b) ** 2 for b in hx), Fraction(0))
        assert _ms_int(hx, 3) == X.round_rne(S / 8, 24, -126)
    assert cases > 300


# heads whose exact mean square is a binary32 tie, and the same plus a 2^-40
TIE_HEADS_HOST = [
    [0x3F93, 0x3F98, 0x3D37, 0x3D37, 0, 0, 0, 0],
    [0x3F93, 0x3F98, 0x3D37, 0x3D37, 0x2B80, 0, 0, 0],
]
