"""Pins for the oracle's weight-only FP8 GEMM (W8A16) and its large-M weight
dequantisation (CPU only).  Independent references: torch's bf16 and
float8_e4m3fn decoders and its RNE float32 -> bf16 conversion, numpy's float64
matmul, exact integer and rational arithmetic, and the W8A8 oracle on
activations that are themselves E4M3 values."""
from fractions import Fraction

import numpy as np
import torch

import workloads


def _dec_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _dec_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()


def _operands(seed, M, N, K, per_channel=True):
    g = workloads.rng(seed)
    x = workloads.bf16_normal_with_outliers(g, (M, K))
    W = workloads.e4m3_codes(g, (N, K))
    sb = workloads.uniform_f32(g, (N if per_channel else 1,), 0.5, 2.0) * np.float32(1e-3)
    return x, W, sb.astype(np.float32)


def test_w8a16_matches_library_matmul(orc):
    """numpy float64 matmul of torch-decoded operands: the same sum in another
    order, so equal to within a few ulps of sum |x w|."""
    for per_channel in (True, False):
        x, W, sb = _operands(31, 5, 67, 1040, per_channel)
        y64, _ = orc.w8a16_mm(x, W, sb, per_channel)
        ref = (_dec_bf16(x) @ _dec_e4m3(W).T) * (sb.astype(np.float64)[None, :] if per_channel else float(sb[0]))
        mag = (np.abs(_dec_bf16(x)) @ np.abs(_dec_e4m3(W)).T) * np.max(sb)
        assert np.all(np.abs(y64 - ref) <= 1e-13 * mag + 1e-300)


def test_w8a16_integer_operands_exact(orc):
    """Integer-valued activations and weights: the sum is an exact integer."""
    g = np.random.default_rng(32)
    M, N, K = 3, 11, 4096
    xi = g.integers(-16, 17, (M, K))
    wi = g.integers(-16, 17, (N, K))
    x = torch.from_numpy(xi.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    W = torch.from_numpy(wi.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(_dec_e4m3(W), wi) and np.array_equal(_dec_bf16(x), xi)
    y64, yb = orc.w8a16_mm(x, W, np.array([1.0], np.float32), False)
    assert np.array_equal(y64, (xi @ wi.T).astype(np.float64))
    # the bf16 output is the RNE rounding of that integer
    ref_b = torch.from_numpy((xi @ wi.T).astype(np.float64)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(yb, ref_b.view(np.uint16))


def test_w8a16_brute_force_rationals_tiny(orc):
    g = np.random.default_rng(33)
    for (M, N, K) in ((1, 1, 1), (2, 3, 7), (3, 4, 33)):
        x, W, sb = _operands(int(g.integers(1 << 30)), M, N, K)
        y64, _ = orc.w8a16_mm(x, W, sb, True)
        xv, wv = _dec_bf16(x), _dec_e4m3(W)
        for m in range(M):
            for n in range(N):
                s = sum(Fraction(float(xv[m, k])) * Fraction(float(wv[n, k])) for k in range(K))
                assert abs(Fraction(float(y64[m, n])) - s * Fraction(float(sb[n]))) <= \
                    Fraction(2) ** -50 * abs(s * Fraction(float(sb[n]))) + Fraction(2) ** -1000


def test_w8a16_equals_w8a8_on_e4m3_activations(orc):
    """Activations that are E4M3 values (bf16 holds every E4M3 value exactly):
    the weight-only GEMM is the W8A8 GEMM with activation scale 1."""
    d = workloads.random_gemm(34, 6, 45, 2064, 1)
    A, W, sb = d["A"], d["B"], d["sb"]
    x = torch.from_numpy(_dec_e4m3(A).astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y16, yb16 = orc.w8a16_mm(x, W, sb, True)
    y8, yb8 = orc.scaled_mm(A, W, np.array([1.0], np.float32), sb, 1)
    assert np.array_equal(y16, y8) and np.array_equal(yb16, yb8)


def test_w8a16_points_match_full(orc):
    x, W, sb = _operands(35, 9, 300, 528)
    y64, _ = orc.w8a16_mm(x, W, sb, True)
    g = np.random.default_rng(36)
    rows, cols = g.integers(0, 9, 200), g.integers(0, 300, 200)
    assert np.array_equal(orc.w8a16_points(x, W, sb, True, rows, cols), y64[rows, cols])


def test_w8a16_nan_weight_code_gives_nan(orc):
    x, W, sb = _operands(37, 2, 4, 64)
    W[1, 5] = 0x7F
    y64, yb = orc.w8a16_mm(x, W, sb, True)
    assert np.all(np.isnan(y64[:, 1])) and not np.any(np.isnan(y64[:, [0, 2, 3]]))
    assert np.all((yb[:, 1] & 0x7F80) == 0x7F80) and np.all((yb[:, 1] & 0x7F) != 0)


def test_dequant_weight_bf16(orc):
    """bf16_rne(fp32(dec(w) * s)): against torch's float32 multiply and RNE
    bf16 conversion; with s = 1 it is the exact E4M3 value."""
    g = np.random.default_rng(38)
    W = workloads.e4m3_codes(g, (37, 96))
    sb = (g.uniform(0.25, 4.0, 37) * 1e-3).astype(np.float32)
    out = orc.dequant_weight_bf16(W, sb, True)
    ref = (torch.from_numpy(_dec_e4m3(W).astype(np.float32)) * torch.from_numpy(sb)[:, None]).to(torch.bfloat16)
    assert np.array_equal(out, ref.view(torch.int16).numpy().view(np.uint16))
    one = orc.dequant_weight_bf16(W, np.array([1.0], np.float32), False)
    assert np.array_equal(_dec_bf16(one), _dec_e4m3(W))
