"""Constructed RMSNorm rows for the exact sum of squares (test inputs only; no
part of the method's arithmetic is shared with the oracle or the kernels).

A bf16 element with exponent field E (1 for subnormals) and integer
significand m (128 | mantissa for normals) is m * 2^(E - 134); its square is
m^2 * 2^(2E - 2) units of 2^-266, so a row's exact sum of squares is a Python
integer in those units.

`carry_row` builds a row whose sum, taken over the row's top 40 binades only
with the smaller squares reduced to a sticky bit, would round to binary32
one unit in the last place too low: the windowed integer has its guard bit 0
and a long run of one bits below it, and the squares under the window carry
through that run.  A probe element, a gamma and a static scale are then
chosen so that the one-ulp difference in the sum of squares reaches the E4M3
code of the probe.
"""
import math

import numpy as np


def split(b):
    b = int(b) & 0x7FFF
    e, mant = b >> 7, b & 0x7F
    return ((128 | mant) if e else mant), (e if e else 1)


def exact_units(row):
    """Exact sum of squares of a finite bf16 row, in units of 2^-266."""
    tot = 0
    for b in row:
        m, E = split(b)
        tot += (m * m) << (2 * E - 2)
    return tot


def round_units_f32(tot, q_min=117):
    """An integer number of 2^-266 units rounded once to binary32 (nearest,
    ties to even; 2^-149 = 2^117 units is the subnormal quantum)."""
    if tot == 0:
        return np.float32(0.0)
    top = tot.bit_length() - 1
    q = max(top - 23, q_min)
    keep, rem = tot >> q, tot & ((1 << q) - 1)
    half = 1 << (q - 1)
    if rem > half or (rem == half and keep & 1):
        keep += 1
    return np.float32(math.ldexp(keep, q - 266))


def window_f32(row):
    """The windowed rule alone: squares of binades >= emax - 39 exactly, any
    smaller nonzero square only as a sticky bit (no carry)."""
    emax = max(((int(b) >> 7) & 0xFF) for b in row)
    elo = max(emax - 39, 1)
    B, sticky = 0, False
    for b in row:
        m, E = split(b)
        if m == 0:
            continue
        if E >= elo:
            B += (m * m) << (2 * (E - elo))
        else:
            sticky = True
    # B in units of 2^(2 elo - 268) = 2^(2 elo - 2) units of 2^-266
    if B == 0:
        return np.float32(0.0)
    top = B.bit_length() - 1
    q = max(top - 23, 119 - 2 * elo)
    if q <= 0:
        return np.float32(math.ldexp(B, 2 * elo - 268))
    keep, rem = B >> q, B & ((1 << q) - 1)
    half = 1 << (q - 1)
    if (rem & half) and ((rem & (half - 1)) or sticky or keep & 1):
        keep += 1
    return np.float32(math.ldexp(keep, q + 2 * elo - 268))


def bf16_bits(E, m):
    return np.uint16((E << 7) | (m & 0x7F))


def _r_chain(ss, K, eps):
    mean = np.float32(ss) / np.float32(K)
    t = np.float32(mean + np.float32(eps))
    return np.float32(np.float32(1.0) / np.sqrt(t))


def _bf16_rne(f):
    u = np.asarray(f, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _bf16_to_f32(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32)


def carry_row(K=64, eps=1e-6, seed=0, max_tries=4000):
    """-> dict(row, gamma, s, probe, ss_exact, ss_window): the row (K bf16
    bits, rest zero), gamma (bf16 bits, 1.0 except at the probe), the static
    scale s (float32) and the probe's index."""
    assert K >= 64
    g = np.random.default_rng(seed)
    emax = 130
    elo = emax - 39
    for _ in range(max_tries):
        elems = [(emax, int(g.integers(128, 256)))]             # the largest binade
        probe_E, probe_m = emax - 2, int(g.integers(128, 256))
        elems.append((probe_E, probe_m))
        for _k in range(3):                                      # a few more large elements
            elems.append((int(g.integers(emax - 12, emax)), int(g.integers(128, 256))))
        big = sum((m * m) << (2 * (E - elo)) for E, m in elems)  # window units
        top = big.bit_length() - 1
        q = top - 23
        head = -(-big // (1 << q)) * (1 << q)                    # next multiple of 2^q
        delta = int(g.integers(1, 4096))
        R = head - big + (1 << (q - 1)) - delta                  # guard 0, ones below
        for j in range(38, -1, -1):                              # greedy fill, binades elo..elo+38
            while R >= (1 << 14) << (2 * j):
                m = min(255, math.isqrt(R >> (2 * j)))
                elems.append((elo + j, m))
                R -= (m * m) << (2 * j)
        d_eff = delta + R                                        # windowed sum = head + 2^(q-1) - d_eff
        n_small = d_eff // 4096 + 1                              # squares below: 4096 units each
        if len(elems) + n_small > K:
            continue
        row = np.zeros(K, np.uint16)
        for i, (E, m) in enumerate(elems):
            row[i] = bf16_bits(E, m)
        for i in range(n_small):
            row[len(elems) + i] = bf16_bits(elo - 1, 128)
        ss_exact = round_units_f32(exact_units(row))
        ss_win = window_f32(row)
        if ss_exact == ss_win:
            continue
        r_t, r_w = _r_chain(ss_exact, K, eps), _r_chain(ss_win, K, eps)
        if r_t == r_w:
            continue
        # a gamma for the probe whose bf16 product differs between the two r
        xp = _bf16_to_f32(bf16_bits(probe_E, probe_m))
        cand = np.arange(0x3F00, 0x4000, dtype=np.uint16)      # gamma in [0.5, 2)
        gam = _bf16_to_f32(cand)
        h_t = _bf16_rne(np.float32(xp * r_t) * gam)
        h_w = _bf16_rne(np.float32(xp * r_w) * gam)
        hit = np.nonzero(h_t != h_w)[0]
        if hit.size == 0:
            continue
        k = int(hit[0])
        ht, hw = _bf16_to_f32(h_t[k]), _bf16_to_f32(h_w[k])
        # a static scale that puts an E4M3 rounding boundary (1.0625, between
        # 1 and 1.125) between ht / s and hw / s
        s = np.float32((np.float64(ht) + np.float64(hw)) / 2.0 / 1.0625)
        lo, hi = sorted((float(np.float32(ht / s)), float(np.float32(hw / s))))
        if not (lo < 1.0625 < hi):
            continue
        gamma = np.full(K, 0x3F80, np.uint16)
        gamma[1] = cand[k]
        return {"row": row, "gamma": gamma, "s": float(s), "probe": 1, "eps": eps,
                "ss_exact": ss_exact, "ss_window": ss_win}
    raise RuntimeError("no carry row found")
