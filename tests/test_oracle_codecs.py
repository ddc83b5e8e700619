"""Pins for the oracle's E4M3 and bf16 codecs (CPU only).

Each check ties the oracle to something other than itself: the OCP FP8 table
of special values (golden file), torch's own float8_e4m3fn and bfloat16 casts
(library routines), exact rational arithmetic, and invariants that any correct
codec must satisfy.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_special_values():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_special_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, value = line.split()[:2]
            rows.append((int(code, 16), float(value)))
    return rows


def test_decode_matches_ocp_table(orc):
    rows = _golden_special_values()
    assert len(rows) == 10
    for code, value in rows:
        got = orc.e4m3_decode(np.array([code], np.uint8))[0]
        if math.isnan(value):
            assert math.isnan(got), hex(code)
        else:
            assert got == value and math.copysign(1, got) == math.copysign(1, value), hex(code)


def test_decode_matches_torch_for_all_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_decode_grid_invariants(orc):
    v = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    fin = v[~np.isnan(v)]
    scaled = fin * 512.0
    assert np.array_equal(scaled, np.round(scaled))          # multiples of 2^-9
    assert np.abs(scaled).max() == 229376                    # 448 * 2^9
    pos = v[:127]
    assert np.all(np.diff(pos) > 0)                          # codes monotone in value
    assert np.array_equal(v[128:255], -pos)                  # sign bit is a pure sign


def test_encode_roundtrip_all_codes(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = orc.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(vals), codes)


def test_encode_hand_cases(orc):
    cases = [
        (448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (float("inf"), 0x7E),
        (-float("inf"), 0xFE), (-500.0, 0xFE), (float("nan"), 0x7F),
        (2.0 ** -10, 0x00),            # half of the smallest subnormal: tie -> even (0)
        (-(2.0 ** -10), 0x80),         # sign of zero kept
        (3 * 2.0 ** -10, 0x02),        # tie between 2^-9 (0x01) and 2^-8 (0x02) -> even
        (1.0 + 1.0 / 16, 0x38),        # tie between 1.0 (0x38) and 1.125 (0x39) -> even
        (1.0 + 3.0 / 16, 0x3A),        # tie between 1.125 (0x39) and 1.25 (0x3A) -> even
        (432.0, 0x7E),                 # tie between 416 (0x7D) and 448 (0x7E) -> even (0x7E)
        (431.99, 0x7D),
        (-0.0, 0x80), (0.0, 0x00),
    ]
    vals = np.array([c[0] for c in cases], np.float32)
    got = orc.e4m3_encode(vals)
    for (v, want), g in zip(cases, got):
        assert g == want, (v, hex(int(g)), hex(want))


def _torch_encode_bits(start, count):
    bits = torch.arange(start, start + count, dtype=torch.int64).to(torch.int32)
    return bits.view(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encode_exhaustive_relevant_binades_vs_torch(orc):
    """Every binary32 value in [2^-12, 2^8) plus [2^8, 464], and two binades of
    negative values, against torch's RNE cast (torch does not saturate above
    464, so the comparison stops there)."""
    chunk = 1 << 23  # one binade
    lo_exp, hi_exp = 127 - 12, 127 + 8  # biased exponents of 2^-12 .. 2^7
    for e in range(lo_exp, hi_exp):
        start = e << 23
        assert np.array_equal(orc.e4m3_encode_bits_range(start, chunk), _torch_encode_bits(start, chunk)), e
    # [256, 464]: 464.0 is 0x43E80000
    start, stop = (127 + 8) << 23, 0x43E80000 + 1
    assert np.array_equal(orc.e4m3_encode_bits_range(start, stop - start), _torch_encode_bits(start, stop - start))
    # negative sign, two binades
    for e in (127 - 7, 127 + 2):
        start = (1 << 31) | (e << 23)
        assert np.array_equal(orc.e4m3_encode_bits_range(start, chunk), _torch_encode_bits(start, chunk)), e


def test_encode_outside_range(orc):
    """Below 2^-11 everything rounds to a signed zero; above 464 everything
    saturates (readings: round-to-nearest-even, saturating)."""
    rng = np.random.default_rng(1)
    tiny_bits = rng.integers(0, (127 - 11) << 23, size=100000, dtype=np.int64).astype(np.uint32)
    tiny = tiny_bits.view(np.float32)
    assert np.all(orc.e4m3_encode(tiny) == 0)
    assert np.all(orc.e4m3_encode(-tiny) == 0x80)
    big = rng.uniform(464.0001, 3e38, size=100000).astype(np.float32)
    assert np.all(orc.e4m3_encode(big) == 0x7E)
    assert np.all(orc.e4m3_encode(-big) == 0xFE)
    nan_bits = (np.uint32(0x7F800000) | rng.integers(1, 1 << 23, size=1000).astype(np.uint32))
    assert np.all(orc.e4m3_encode(nan_bits.view(np.float32)) == 0x7F)


def test_encode_monotone(orc):
    v = np.sort(np.random.default_rng(2).uniform(-500, 500, size=200000).astype(np.float32))
    dec = orc.e4m3_decode(orc.e4m3_encode(v))
    assert np.all(np.diff(dec) >= 0)


def test_encode_matches_exact_rational_nearest(orc):
    """Brute force with exact rationals: the nearest grid value, ties to the
    code with even mantissa, computed from scratch over the E4M3 grid."""
    grid = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            grid.append(Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7))
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.uniform(0, 448, 3000), np.exp2(rng.uniform(-12, 8.8, 3000))]).astype(np.float32)
    got = orc.e4m3_encode(vals)
    for v, g in zip(vals, got):
        fv = Fraction(float(v))
        if fv >= 448:
            want = 126
        else:
            dists = [abs(fv - q) for q in grid]
            best = min(dists)
            cands = [i for i, d in enumerate(dists) if d == best]
            want = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        assert g == want, (float(v), int(g), want)


def test_bf16_rne_from_f32_vs_torch(orc):
    """All 65536 bf16 neighbourhoods x the low-half patterns that decide rounding."""
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFF, 0x1234, 0x9ABC], np.uint32)
    bits = (hi[:, None] | lows[None, :]).ravel()
    v = bits.view(np.float32)
    ours = orc.bf16_rne(v)
    ref = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(v)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all((ours[nan] & 0x7F80) == 0x7F80) and np.all((ours[nan] & 0x7F) != 0)


def _bf16_exact_nearest(x: float) -> float:
    """Nearest bf16 to the binary64 x with exact rationals, ties to even significand."""
    if x == 0:
        return x
    fx = Fraction(x)
    a = abs(fx)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = Fraction(2) ** (e - 7)
    n = a / q
    f = math.floor(n)
    r = n - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        f += 1
    out = f * q
    if out >= Fraction(2) ** 128:
        return math.copysign(math.inf, x)
    return math.copysign(float(out), x)


def test_bf16_rne_from_f64_exact(orc):
    """The binary64 path rounds once (torch's double->bf16 rounds twice, so the
    check is against exact rationals)."""
    rng = np.random.default_rng(4)
    v = np.concatenate([
        rng.standard_normal(2000) * np.exp2(rng.integers(-130, 127, 2000)),
        1 + 2.0 ** -8 + np.array([2.0 ** -40, -(2.0 ** -40), 0.0]),    # just above / below / at a tie
        np.array([3.3895313892515355e38, 3.4e38, 1e-40, -1e-45, 2.0 ** -133, 3 * 2.0 ** -134]),
    ])
    ours = orc.bf16_to_f32(orc.bf16_rne(v.astype(np.float64)))
    for x, o in zip(v, ours):
        want = _bf16_exact_nearest(float(x))
        assert (o == want) or (math.isinf(o) and math.isinf(want) and (o > 0) == (want > 0)), (x, o, want)
