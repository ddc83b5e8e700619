"""Host checks of the integer and binary32 recipes the kernels compute with,
each against an independent definition (the oracle's E4M3 decode, exact
integer arithmetic, exact rationals): the E4M3 -> bf16 widening of the
weight-only kernels and its NaN test, the decode GEMM's exact split of a
k-block partial into integer parts, and the TwoSum accumulation of the
blockwise paths.  The recipes are restated here in numpy so that a wrong
constant, shift or sign fails on the CPU; the GPU tests run the kernels
themselves (test_w16_every_code_exact, the exact-sum decode tests, the
blockwise tests).  No GPU needed."""
import numpy as np

import oracle

TWO120 = 2.0 ** 120


def widen_lane(code):
    """One E4M3 code as the widening builds it: the code in the low byte of a
    16-bit lane with its sign byte replicated above (the byte permute), shifted
    left by 4 and masked to the sign and the 7 magnitude bits -- a bf16 pattern
    of the value times 2^-120 -- then the exact bf16 multiply by 2^120."""
    code = np.asarray(code, np.uint32)
    lane = np.where(code & 0x80, 0xFF00, 0x0000).astype(np.uint32) | code
    bits = (lane << 4) & 0x87F0
    # bf16 pattern -> binary32 -> value; times 2^120 is exact in binary64
    f = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return f * TWO120


def nan_flags(words):
    """The widening's NaN test on 32-bit words of four codes: bit 7 of each
    byte of ((w & 0x7F7F7F7F) + 0x01010101) & 0x80808080 is set exactly when
    that byte's low 7 bits are all ones."""
    w = np.asarray(words, np.uint64)
    return ((w & 0x7F7F7F7F) + 0x01010101) & 0x80808080


def test_widening_every_code():
    codes = np.arange(256, dtype=np.uint32)
    got = widen_lane(codes)
    want = oracle.e4m3_decode(codes.astype(np.uint8))
    finite = (codes & 0x7F) != 0x7F
    assert np.array_equal(got[finite], want[finite])
    # signed zeros keep their sign; subnormal codes come out exactly
    assert np.signbit(got[0x80]) and not np.signbit(got[0x00])
    assert got[0x01] == 2.0 ** -9 and got[0x07] == 7 * 2.0 ** -9 and got[0x7E] == 448.0
    # the NaN codes come out as 480: finite, so the kernels test for them separately
    assert np.all(got[~finite] == np.where(codes[~finite] & 0x80, -480.0, 480.0))


def test_nan_test_every_byte_and_position():
    for pos in range(4):
        for c in range(256):
            other = 0x3C  # a finite code in the other three bytes
            w = 0
            for p in range(4):
                w |= (c if p == pos else other) << (8 * p)
            flags = int(nan_flags([w])[0])
            is_nan = (c & 0x7F) == 0x7F
            assert flags == ((0x80 << (8 * pos)) if is_nan else 0), (pos, hex(c))


def test_nan_test_random_words():
    g = np.random.default_rng(8100)
    w = g.integers(0, 2 ** 32, 200000, dtype=np.uint64)
    flags = nan_flags(w)
    b = (w[:, None] >> (8 * np.arange(4, dtype=np.uint64))) & 0xFF
    want = np.zeros_like(w)
    for p in range(4):
        want |= np.where((b[:, p] & 0x7F) == 0x7F, np.uint64(0x80) << np.uint64(8 * p), np.uint64(0))
    assert np.array_equal(flags, want)


SPLIT_HI = np.float32(402653184.0)   # 1.5 * 2^28: ulp 32
SPLIT_LO = np.float32(12582912.0)    # 1.5 * 2^23: ulp 1
FIX = np.float32(262144.0)           # 2^18


def exact_split(p):
    """The decode drain's split of a binary32 k-block partial p (a multiple
    of 2^-18 below 2^25 in magnitude): t = p + 1.5*2^28 rounds p to a multiple
    of 32; hi = bits(t) - bits(1.5*2^28) is that multiple over 32; the rest
    p - (t - 1.5*2^28) is exact, and u = rest * 2^18 + 1.5*2^23 gives
    lo = bits(u) - bits(1.5*2^23) = rest * 2^18.  Every step in binary32,
    round to nearest (numpy float32 arithmetic; fma as multiply then add is
    exact here because rest * 2^18 is an integer below 2^23)."""
    p = np.asarray(p, np.float32)
    t = (p + SPLIT_HI).astype(np.float32)
    rest = (p - (t - SPLIT_HI).astype(np.float32)).astype(np.float32)
    u = (rest * FIX + SPLIT_LO).astype(np.float32)
    hi = t.view(np.int32).astype(np.int64) - np.int64(SPLIT_HI.view(np.int32))
    lo = u.view(np.int32).astype(np.int64) - np.int64(SPLIT_LO.view(np.int32))
    return hi, lo


def test_exact_split_reconstructs_every_partial():
    """hi * 2^23 + lo (units of 2^-18) equals p * 2^18 exactly for binary32
    partials on the 2^-18 grid across the whole range the tensor core can
    produce from one 128-wide k-block of E4M3 products (|p| <= 128 * 448^2)."""
    g = np.random.default_rng(8200)
    mags = np.concatenate([
        g.integers(0, 2 ** 24, 100000),                     # small partials, every low bit live
        g.integers(0, 2 ** 43, 100000),                     # up to 2^25 in value
        np.array([0, 1, 2 ** 18, 2 ** 23 - 1, 2 ** 23, 2 ** 24 + 1, 128 * 448 * 448 * 2 ** 18]),
    ]).astype(np.int64)
    # a binary32 value on the 2^-18 grid: round the integer to 24 significant bits first
    vals = np.array([float(m) for m in mags], np.float64)
    p = (vals * 2.0 ** -18).astype(np.float32)
    p = np.concatenate([p, -p])
    keep = np.abs(p.astype(np.float64)) <= 128 * 448.0 ** 2
    p = p[keep]
    hi, lo = exact_split(p)
    exact = (p.astype(np.float64) * 2.0 ** 18)
    assert np.all(exact == np.round(exact))  # every p sits on the 2^-18 grid
    assert np.array_equal(hi * (1 << 23) + lo, exact.astype(np.int64))
    # the parts stay inside the ranges the drain's 32-bit accumulators assume
    assert np.all(np.abs(hi) < 2 ** 20) and np.all(np.abs(lo) <= 2 ** 22)


def test_exact_split_sums_are_order_free():
    """Adding the parts of many partials as integers gives the exact sum in
    any order (what makes the decode GEMM's result independent of how K is
    divided): against the binary64 sum, exact for these magnitudes."""
    g = np.random.default_rng(8300)
    p = (g.integers(-2 ** 40, 2 ** 40, 2048).astype(np.float64) * 2.0 ** -18).astype(np.float32)
    hi, lo = exact_split(p)
    total = int(np.sum(hi)) * (1 << 23) + int(np.sum(lo))
    want = sum(int(round(float(x) * 2.0 ** 18)) for x in p)
    assert total == want
    perm = g.permutation(len(p))
    hi2, lo2 = exact_split(p[perm])
    assert int(np.sum(hi2)) * (1 << 23) + int(np.sum(lo2)) == total


def two_sum_acc(hi, lo, v):
    """The blockwise paths' TwoSum accumulation (Knuth's error-free sum: s =
    hi + v and err with s + err == hi + v exactly, err folded into lo), every
    operation binary32 round to nearest."""
    f = np.float32
    s = f(hi + v)
    bv = f(s - hi)
    av = f(s - bv)
    err = f(f(hi - av) + f(v - bv))
    return s, f(lo + err)


def test_two_sum_is_error_free():
    """One step: s + err equals hi + v exactly (binary64 holds both sums
    exactly for exponents this close)."""
    g = np.random.default_rng(8400)
    a = (g.standard_normal(100000) * np.exp2(g.integers(-20, 20, 100000))).astype(np.float32)
    b = (g.standard_normal(100000) * np.exp2(g.integers(-20, 20, 100000))).astype(np.float32)
    for x, y in zip(a[:20000], b[:20000]):
        s, err = two_sum_acc(x, np.float32(0.0), y)
        assert float(s) + float(err) == float(x) + float(y)


def test_two_sum_accumulation_of_k_block_partials():
    """A tile's 40 scaled k-block partials (K 5120) folded into (hi, lo) and
    rounded once: within a few units of 2^-48 of the partials' absolute sum
    from the exact sum, where a plain binary32 sum is ~2^-24 away."""
    from fractions import Fraction
    g = np.random.default_rng(8500)
    worst_ts, worst_plain = 0.0, 0.0
    for _ in range(200):
        x = (g.standard_normal(40) * np.exp2(g.integers(-6, 6, 40))).astype(np.float32)
        hi, lo, plain = np.float32(0.0), np.float32(0.0), np.float32(0.0)
        for v in x:
            hi, lo = two_sum_acc(hi, lo, v)
            plain = np.float32(plain + v)
        exact = sum(Fraction(float(v)) for v in x)
        scale = float(sum(abs(Fraction(float(v))) for v in x))
        worst_ts = max(worst_ts, abs(float(Fraction(float(hi)) + Fraction(float(lo)) - exact)) / scale)
        worst_plain = max(worst_plain, abs(float(Fraction(float(plain)) - exact)) / scale)
    assert worst_ts <= 64 * 2.0 ** -48
    assert worst_plain > 2.0 ** -30  # the comparison has teeth: plain binary32 loses far more
