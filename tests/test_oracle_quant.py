"""Pins for the oracle's quantisers and RMSNorm producer (CPU only)."""
import math
from fractions import Fraction

import numpy as np
import sympy
import torch

import workloads


def _torch_e4m3(v32: np.ndarray) -> np.ndarray:
    """Library encoding: torch's RNE float8_e4m3fn cast after clamping to +-448
    (torch maps magnitudes above 464 to NaN instead of saturating)."""
    t = torch.from_numpy(np.ascontiguousarray(v32, np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _as_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def test_static_quant_vs_torch(orc):
    g = workloads.rng(10)
    x = workloads.bf16_normal(g, (16, 512), std=3.0)
    for s in (np.float32(1 / 56), np.float32(0.01), np.float32(0.37), np.float32(2.5e-3)):
        q = orc.quant_static(x, float(s))
        t = torch.from_numpy(_as_f32(x).copy()) / torch.tensor(s)      # IEEE binary32 division
        assert np.array_equal(q, _torch_e4m3(t.numpy()))


def test_static_quant_saturates(orc):
    x = np.array([[0x4400, 0xC400, 0x7F80, 0xFF80]], np.uint16)  # 512, -512, +inf, -inf
    q = orc.quant_static(x, 1.0)
    assert q.tolist() == [[0x7E, 0xFE, 0x7E, 0xFE]]


def test_quant_dequant_idempotent(orc):
    """enc(fp32(dec(q)*s)/s) == q for every finite code over a sweep of scales."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    dec = orc.e4m3_decode(codes)
    for s in np.exp2(np.linspace(-12, 6, 37)).astype(np.float32):
        v = (dec * float(s)).astype(np.float32)          # fp32(dec * s)
        back = (v / s).astype(np.float32)
        assert np.array_equal(orc.e4m3_encode(back), codes), s


def test_per_token_properties(orc):
    g = workloads.rng(11)
    x = workloads.bf16_normal_with_outliers(g, (64, 640))
    q, s = orc.quant_per_token(x)
    xf = _as_f32(x)
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
    # the amax element of each row encodes to +-448
    idx = np.abs(xf).argmax(axis=1)
    assert np.all((q[np.arange(64), idx] & 0x7F) == 0x7E)
    # same bytes as torch's encoder on x / s
    assert np.array_equal(q, _torch_e4m3(xf / s[:, None]))


def test_per_token_power_of_two_equivariance(orc):
    """Scaling a row by 2^k scales its scale by 2^k and leaves the codes alone."""
    g = workloads.rng(12)
    x = workloads.bf16_normal(g, (8, 256))
    q0, s0 = orc.quant_per_token(x)
    for k in (-5, 3, 9):
        xk = ((_as_f32(x) * np.float32(2.0 ** k)).view(np.uint32) >> 16).astype(np.uint16)  # exact
        qk, sk = orc.quant_per_token(xk)
        assert np.array_equal(qk, q0)
        assert np.array_equal(sk, (s0 * np.float32(2.0 ** k)).astype(np.float32))


def test_per_token_zero_row_and_single_row(orc):
    x = np.zeros((2, 32), np.uint16)
    x[1, 5] = 0x3F80  # 1.0
    q, s = orc.quant_per_token(x)
    assert s[0] == 1.0 and np.all(q[0] == 0)
    assert s[1] == np.float32(1.0) / np.float32(448.0)
    assert q[1, 5] == 0x7E and np.count_nonzero(q[1]) == 1


def test_per_token_of_flattened_tensor_is_static_amax_quant(orc):
    """One-row per-token quant of a flattened tensor == static quant with s = amax/448."""
    w = workloads.bf16_normal(workloads.rng(13), (64, 128), std=0.02)
    q1, s1 = orc.quant_per_token(w.reshape(1, -1))
    q2 = orc.quant_static(w, float(s1[0]))
    assert np.array_equal(q1.reshape(64, 128), q2)


def _rms_exact(xs, eps, gamma, k):
    """High-precision value of x_k * gamma_k / sqrt(mean(x^2) + eps)."""
    xs = [sympy.Rational(float(v)) for v in xs]
    mean = sum(v * v for v in xs) / len(xs)
    r = 1 / sympy.sqrt(mean + sympy.Rational(float(np.float32(eps))))
    return float(sympy.N(xs[k] * sympy.Rational(float(gamma)) * r, 40))


def test_rmsnorm_closed_forms(orc):
    """Constant rows and single-spike rows against a 40-digit evaluation: the
    oracle lands within one bf16 rounding of the exact value."""
    K = 64
    cases = []
    # 1.0, 3.0, -0.125, 2^-63 (rows whose mean square underflows binary32 are left
    # out: with eps = 0 the binary32 chain then divides by zero)
    for c in (0x3F80, 0x4040, 0xBE00, 0x2000):
        cases.append(np.full(K, c, np.uint16))
    spike = np.zeros(K, np.uint16)
    spike[7] = 0x40A0                                   # 5.0
    cases.append(spike)
    gamma = np.full(K, 0x3FC0, np.uint16)               # 1.5
    # 2^-126: the squares (2^-252) underflow binary32 and the sum of squares
    # rounds to zero; with eps > 0 the chain is defined and lands within one
    # bf16 rounding of the exact value, whose mean square is negligible next to eps
    tiny = np.full(K, 0x0080, np.uint16)
    for eps in (1e-6, 0.0, 0.25):
        for row in cases + ([tiny] if eps > 0 else []):
            h = orc.rmsnorm_bf16(row[None, :], gamma, eps)[0]
            hv = _as_f32(h)
            for k in (0, 7):
                want = _rms_exact(_as_f32(row), eps, 1.5, k)
                ulp = 2.0 ** (math.floor(math.log2(abs(want))) - 7) if want != 0 else 0.0
                assert abs(float(hv[k]) - want) <= ulp, (row[:2], eps, k, hv[k], want)
    assert orc.sum_squares_bf16(tiny) == 0.0


def test_rmsnorm_eps0_underflow_row(orc):
    """eps = 0 and a row whose mean square underflows binary32 (every element
    +-2^-126 or 0): the sum of squares rounds to 0, r = 1/sqrt(0) = +inf, so
    a nonzero element becomes +-inf and saturates to +-448 and a zero element
    becomes 0 * inf = NaN (the NaN code) -- IEEE semantics of the stated chain."""
    row = np.full((1, 64), 0x0080, np.uint16)
    row[0, 3] = 0x0000
    row[0, 5] = 0x8080
    gamma = np.full(64, 0x3FC0, np.uint16)
    q = orc.rmsnorm_quant(row, gamma, 0.0, float(np.float32(1 / 56)))[0]
    assert q[0] == 0x7E and q[5] == 0xFE and (q[3] & 0x7F) == 0x7F
    assert np.all(q[[1, 2, 4, 6, 63]] == 0x7E)


def test_rmsnorm_scale_invariance(orc):
    """With eps = 0, RMSNorm(2^j x) == RMSNorm(x) exactly (every step scales exactly)."""
    g = workloads.rng(14)
    x = workloads.bf16_normal(g, (4, 512))
    gamma = workloads.bf16_normal(g, (512,), mean=1.0, std=0.1)
    h0 = orc.rmsnorm_bf16(x, gamma, 0.0)
    for j in (-7, 4):
        xj = ((_as_f32(x) * np.float32(2.0 ** j)).view(np.uint32) >> 16).astype(np.uint16)
        assert np.array_equal(orc.rmsnorm_bf16(xj, gamma, 0.0), h0)


def _f32_nearest(fr: Fraction) -> np.float32:
    """Exact rational -> nearest binary32 (ties to even), normal range."""
    if fr == 0:
        return np.float32(0.0)
    a = abs(fr)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (e - 23)
    n = a / q
    f = math.floor(n)
    rem = n - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return np.float32(math.copysign(float(f * q), fr))


def test_sum_squares_exact_vs_rationals(orc):
    """The sum of squares is the exact rational sum rounded once to binary32,
    including rows whose terms span more binades than binary64 can hold."""
    g = np.random.default_rng(17)
    rows = [workloads.bf16_normal(g, (256,)), workloads.bf16_normal(g, (1000,), std=1e-3)]
    wide = workloads.bf16_normal(g, (64,))
    wide[::2] = (np.float32(2.0 ** -60) * _as_f32(wide[::2])).view(np.uint32) >> 16
    rows.append(wide.astype(np.uint16))                                # 2^-60 next to O(1): > 120 bits
    tie = np.array([0x3F80, 0x3F80, 0x3F80, 0x3380, 0x3380], np.uint16)  # 3 + 2*2^-48: a binary32 tie + sticky
    rows.append(tie)
    rows.append(np.array([0x0001, 0x0002, 0x0080], np.uint16))        # subnormal bf16 inputs
    for r in rows:
        exact = sum(Fraction(float(v)) ** 2 for v in _as_f32(r))
        assert orc.sum_squares_bf16(r) == _f32_nearest(exact) if exact >= Fraction(2) ** -126 else True
    # 1 + 2^-24 is a binary32 tie (rounds to even, 1.0); a 2^-80 term breaks the tie upwards
    assert orc.sum_squares_bf16(np.array([0x3F80, 0x3980], np.uint16)) == np.float32(1.0)
    assert orc.sum_squares_bf16(np.array([0x3F80, 0x3980, 0x2B80], np.uint16)) == np.nextafter(
        np.float32(1.0), np.float32(2.0))
    assert orc.sum_squares_bf16(np.zeros(8, np.uint16)) == 0.0
    assert np.isinf(orc.sum_squares_bf16(np.array([0x3F80, 0x7F80], np.uint16)))
    assert np.isnan(orc.sum_squares_bf16(np.array([0x7F80, 0x7FC1], np.uint16)))


def test_sum_squares_carry_rows(orc):
    """Constructed rows where the squares below the row's top 40 binades carry
    into the rounding (a run of one bits under a zero guard bit): the oracle's
    sum is the exact integer sum rounded once (Python integers), which here
    differs from the windowed sum with only a sticky bit for the small squares;
    and the probe element's E4M3 code follows the exact sum."""
    import norm_cases
    for K, seed in ((64, 0), (64, 1), (5120, 2), (64, 3)):
        d = norm_cases.carry_row(K=K, seed=seed)
        exact = norm_cases.round_units_f32(norm_cases.exact_units(d["row"]))
        assert orc.sum_squares_bf16(d["row"]) == exact == d["ss_exact"]
        assert exact != norm_cases.window_f32(d["row"])
        frac = sum(Fraction(float(v)) ** 2 for v in _as_f32(d["row"]))
        assert exact == _f32_nearest(frac)
        q = orc.rmsnorm_quant(d["row"][None, :], d["gamma"], d["eps"], d["s"])[0]
        assert q[d["probe"]] == 0x38        # 1.0: the boundary 1.0625 lies between the exact and windowed h / s


def test_rmsnorm_vs_numpy_restatement(orc):
    """The pinned arithmetic restated with numpy's vectorised ops (binary64 sum
    of the exact squares, then the binary32 chain) gives the same bf16 bits."""
    g = workloads.rng(15)
    x = workloads.bf16_normal(g, (32, 5120))
    gamma = workloads.bf16_normal(g, (5120,), mean=1.0, std=0.1)
    h = orc.rmsnorm_bf16(x, gamma, 1e-6)
    xf = _as_f32(x)
    ss = np.sum(xf.astype(np.float64) ** 2, axis=1).astype(np.float32)
    t = (ss / np.float32(5120)).astype(np.float32) + np.float32(1e-6)
    r = (np.float32(1.0) / np.sqrt(t.astype(np.float32))).astype(np.float32)
    u = (xf * r[:, None]).astype(np.float32) * _as_f32(gamma)[None, :]
    ref = torch.from_numpy(u.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(h, ref)


def test_rmsnorm_quant_is_norm_then_static_quant(orc):
    g = workloads.rng(16)
    x = workloads.bf16_normal(g, (8, 1024))
    gamma = workloads.bf16_normal(g, (1024,), mean=1.0, std=0.1)
    s = float(np.float32(1 / 56))
    assert np.array_equal(orc.rmsnorm_quant(x, gamma, 1e-6, s), orc.quant_static(orc.rmsnorm_bf16(x, gamma, 1e-6), s))
    # zero rows: eps keeps the root finite and every code is zero
    z = np.zeros((2, 1024), np.uint16)
    assert np.all(orc.rmsnorm_quant(z, gamma, 1e-6, s) == 0)


# --------------------------------------------------------------------------- residual add (R18)

def _bf16_bits_of_f32(v32):
    """float32 -> bf16 bits by torch's round-to-nearest-even cast (a library
    primitive, pinned separately against exact rationals)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_residual_add_is_f32_sum_then_bf16(orc):
    """h = bf16(fp32(x) + fp32(r)): against numpy's IEEE binary32 addition
    followed by torch's RNE cast, on random pairs with every exponent gap
    (exact fp32 sums and rounded ones), both signs, zeros and subnormals."""
    g = np.random.default_rng(70)
    x = workloads.bf16_normal(g, (4096,), std=1.0)
    r = workloads.bf16_normal(g, (4096,), std=1.0)
    scale = (2.0 ** g.integers(-40, 40, 4096)).astype(np.float32)
    r = (((r.astype(np.uint32) << 16).view(np.float32) * scale).view(np.uint32) >> 16).astype(np.uint16)
    r[:16] = [0, 0x8000, 0x0001, 0x8001, 0x7F7F, 0xFF7F, 0x3F80, 0xBF80] * 2
    x[:16] = [0, 0, 0x0001, 0x0001, 0x7F7F, 0x7F7F, 0xBF80, 0x3F80] + [0x4000] * 8
    with np.errstate(over="ignore"):
        want = _bf16_bits_of_f32((x.astype(np.uint32) << 16).view(np.float32)
                                 + (r.astype(np.uint32) << 16).view(np.float32))
    h = orc.residual_add_bf16(x, r)
    assert np.array_equal(h, want)
    assert np.array_equal(orc.residual_add_bf16(r, x), h)          # commutative
    assert h[4] == 0x7F80                                          # max + max overflows to +inf
    assert h[6] == 0x0000                                          # -1 + 1 = +0 (round to nearest)


def test_residual_add_exact_rationals(orc):
    """Where the binary32 sum is exact (exponent gap <= 16), h is the exact
    rational sum rounded once to bf16 (ties to even), computed with fractions."""
    from fractions import Fraction
    g = np.random.default_rng(71)
    xs = workloads.bf16_normal(g, (300,))
    rs = workloads.bf16_normal(g, (300,), std=0.05)
    h = orc.residual_add_bf16(xs, rs)

    def val(b):
        return Fraction(float((np.uint32(b) << np.uint32(16)).view(np.float32)))

    def bf16_rne(q):
        if q == 0:
            return 0.0
        sgn = -1 if q < 0 else 1
        a = abs(q)
        e = 0
        while a >= 2:
            a /= 2
            e += 1
        while a < 1:
            a *= 2
            e -= 1
        unit = Fraction(1, 128)
        k = a / unit
        lo = int(k)
        rem = k - lo
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
            lo += 1
        return sgn * float(lo * unit * Fraction(2) ** e)

    checked = 0
    for a, b, got in zip(xs, rs, h):
        fa, fb = val(a), val(b)
        if fa == 0 or fb == 0:
            continue
        ea = int(np.floor(np.log2(abs(float(fa)))))
        eb = int(np.floor(np.log2(abs(float(fb)))))
        if abs(ea - eb) > 16:
            continue
        want = bf16_rne(fa + fb)
        assert float((np.uint32(got) << np.uint32(16)).view(np.float32)) == want
        checked += 1
    assert checked > 200


def test_add_rmsnorm_quant_composition(orc):
    """The fused producer is residual add, then the pinned RMSNorm -> quant;
    a zero residual gives exactly rmsnorm_quant(x) (x has no negative zeros,
    which the add would turn into +0)."""
    d = workloads.decode_fused(seed=7)
    g = np.random.default_rng(72)
    r = workloads.bf16_normal(g, d["x"].shape, std=0.5)
    s = float(d["s_a"])
    q, h = orc.add_rmsnorm_quant(d["x"], r, d["gamma"], d["eps"], s)
    assert np.array_equal(h, orc.residual_add_bf16(d["x"], r))
    assert np.array_equal(q, orc.rmsnorm_quant(h, d["gamma"], d["eps"], s))
    z = np.zeros_like(d["x"])
    q0, h0 = orc.add_rmsnorm_quant(d["x"], z, d["gamma"], d["eps"], s)
    assert np.array_equal(q0, orc.rmsnorm_quant(d["x"], d["gamma"], d["eps"], s))


# --------------------------------------------------------------------------- SiLU * up -> per-token quant (R19)

def test_exp_f32_within_two_ulp_of_binary64(orc):
    y = np.linspace(-87.0, 88.0, 400001).astype(np.float32)
    e = orc.exp_f32(y).astype(np.float64)
    t = np.exp(y.astype(np.float64))
    ulp = np.spacing(t.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(e - t) / ulp) <= 2.0
    assert np.all(np.diff(e) >= 0)                       # monotone on the sweep
    assert orc.exp_f32(np.float32(0.0))[0] == 1.0
    assert orc.exp_f32(np.float32(1.0))[0] == np.float32(np.e)
    sp = orc.exp_f32(np.array([np.nan, -100.0, -87.5, 100.0, np.inf, -np.inf], np.float32))
    assert np.isnan(sp[0]) and sp[1] == 0.0 and sp[2] == 0.0 and np.isinf(sp[3]) and np.isinf(sp[4])
    assert sp[5] == 0.0


def test_silu_against_binary64(orc):
    """silu(g) = g / (1 + e(-g)) within 4 ulp of the binary64 value
    g / (1 + exp(-g)) over [-80, 80], exact special cases."""
    g = np.linspace(-80.0, 80.0, 200001).astype(np.float32)
    got = orc.silu_f32(g).astype(np.float64)
    ref = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64)))
    ulp = np.maximum(np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64), 1e-45)
    assert np.max(np.abs(got - ref) / ulp) <= 4.0
    sp = orc.silu_f32(np.array([0.0, np.inf, -100.0, np.nan], np.float32))
    assert sp[0] == 0.0 and sp[1] == np.inf
    assert sp[2] == 0.0 and np.signbit(sp[2])            # -100 / inf = -0
    assert np.isnan(sp[3])


def test_silu_mul_bf16_definition(orc):
    """a = bf16(silu(g) * u): the binary32 product of the pinned silu and u,
    rounded by torch's RNE cast; gate is the first half of each row."""
    import torch
    g = np.random.default_rng(73)
    gu = workloads.bf16_normal(g, (3, 2 * 64), std=3.0)
    a = orc.silu_mul_bf16(gu)
    gate = (gu[:, :64].astype(np.uint32) << 16).view(np.float32)
    up = (gu[:, 64:].astype(np.uint32) << 16).view(np.float32)
    s = orc.silu_f32(gate).reshape(gate.shape)
    want = torch.from_numpy(s * up).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(a, want)


def test_silu_mul_quant_composition(orc):
    """The fused producer equals the per-token quantisation of the bf16
    intermediate; its amax element maps to +-448."""
    g = np.random.default_rng(74)
    gu = workloads.bf16_normal_with_outliers(g, (4, 2 * 256))
    gu[1] = 0
    q, s = orc.silu_mul_quant_per_token(gu)
    a = orc.silu_mul_bf16(gu)
    q2, s2 = orc.quant_per_token(a)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
    assert s[1] == 1.0 and np.all(q[1] == 0)
    for m in (0, 2, 3):
        assert np.max(q[m] & 0x7F) == 0x7E


# --------------------------------------------------------------------------- shard requantisation (R20)

ALL_CODES = np.arange(256, dtype=np.uint8)
NAN_CODES = (ALL_CODES & 0x7F) == 0x7F


def test_requant_identity_and_powers_of_two(orc):
    """Same scale: every code maps to itself.  Twice the scale: every code
    maps to the code of half its value (exact in E4M3 down to the smallest
    normals; subnormal halves round to nearest even)."""
    for s in (1.0, 3.7e-3, 2.0 ** -20, 123.0):
        s = float(np.float32(s))
        q = orc.requant(ALL_CODES, s, s)
        assert np.array_equal(q[~NAN_CODES], ALL_CODES[~NAN_CODES])
        assert np.all((q[NAN_CODES] & 0x7F) == 0x7F)
    dec = orc.e4m3_decode(ALL_CODES)
    half = orc.requant(ALL_CODES, 0.5, 1.0)
    want = orc.e4m3_encode((dec / 2).astype(np.float32))
    assert np.array_equal(half[~NAN_CODES], want[~NAN_CODES])
    exact = (~NAN_CODES) & ((ALL_CODES & 0x78) >= 0x10)          # exponent field >= 2: halving stays normal
    assert np.array_equal(orc.e4m3_decode(half[exact]), dec[exact] / 2)


def test_requant_to_max_scale_is_monotone_and_close(orc):
    """Requantising to a larger scale keeps the order of the values and each
    result is the nearest E4M3 value to dec(q) * s_in / s_out (brute force
    over the 254 finite values)."""
    s_in, s_out = float(np.float32(1.3e-3)), float(np.float32(2.9e-3))
    q = orc.requant(ALL_CODES, s_in, s_out)
    dec = orc.e4m3_decode(ALL_CODES)
    fin = ~NAN_CODES
    order = np.argsort(dec[fin], kind="stable")
    got = orc.e4m3_decode(q[fin])[order]
    assert np.all(np.diff(got) >= 0)
    grid = np.unique(orc.e4m3_decode(ALL_CODES[fin]))
    target = (np.float32(dec[fin]) * np.float32(s_in)) / np.float32(s_out)
    nearest = np.abs(grid[None, :] - target.astype(np.float64)[:, None]).min(axis=1)
    assert np.all(np.abs(orc.e4m3_decode(q[fin]) - target) <= nearest + 1e-12)
