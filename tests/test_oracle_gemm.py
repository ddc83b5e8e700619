"""Pins for the oracle's scaled GEMM (CPU only)."""
import os
from fractions import Fraction

import numpy as np
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_acc_f64_equals_int64_twin(orc):
    for (M, N, K) in ((3, 5, 17408), (7, 9, 5120), (1, 1, 1)):
        d = workloads.random_gemm(20 + K, M, N, K, 0)
        A, B = d["A"], d["B"]
        A[0, :8] = 0x7E
        B[0, :8] = 0xFE
        acc = orc.gemm_acc_f64(A, B)
        acc_i = orc.gemm_acc_i64(A, B)
        assert np.array_equal(acc, acc_i.astype(np.float64) * 2.0 ** -18)
        assert np.all(np.abs(acc_i) < 2 ** 53)


def test_acc_equals_library_matmul_of_decoded(orc):
    """numpy's float64 matmul of the torch-decoded operands is exact here, so it
    must agree bit for bit."""
    d = workloads.random_gemm(21, 13, 37, 1024, 0)
    acc = orc.gemm_acc_f64(d["A"], d["B"])
    ref = _torch_decode(d["A"]) @ _torch_decode(d["B"]).T
    assert np.array_equal(acc, ref)


def test_acc_brute_force_rationals_tiny(orc):
    rng = np.random.default_rng(22)
    for (M, N, K) in ((1, 1, 1), (2, 3, 5), (4, 8, 32)):
        d = workloads.random_gemm(int(rng.integers(1 << 30)), M, N, K, 0)
        acc = orc.gemm_acc_f64(d["A"], d["B"])
        a = _torch_decode(d["A"])
        b = _torch_decode(d["B"])
        for m in range(M):
            for n in range(N):
                want = sum(Fraction(float(a[m, k])) * Fraction(float(b[n, k])) for k in range(K))
                assert Fraction(float(acc[m, n])) == want


def test_acc_hand_cases(orc):
    K = 96
    one = np.full((1, K), 0x38, np.uint8)
    big = np.full((1, K), 0x7E, np.uint8)
    assert orc.gemm_acc_f64(one, one)[0, 0] == K
    assert orc.gemm_acc_f64(big, big)[0, 0] == 200704 * K
    assert orc.gemm_acc_f64(big, big[:, ::1] | 0x80)[0, 0] == -200704 * K
    a = np.array([[0x40]], np.uint8)   # 2.0
    b = np.array([[0x2C]], np.uint8)   # 0.375 = 1.5 * 2^-2
    assert orc.gemm_acc_f64(a, b)[0, 0] == 0.75


def test_scale_granularities_agree(orc):
    M, N, K = 6, 10, 64
    d = workloads.random_gemm(23, M, N, K, 0)
    A, B = d["A"], d["B"]
    sa = np.float32(0.0123)
    sb = np.float32(0.00456)
    y0, b0 = orc.scaled_mm(A, B, [sa], [sb], 0)
    y1, b1 = orc.scaled_mm(A, B, [sa], np.full(N, sb, np.float32), 1)
    y2, b2 = orc.scaled_mm(A, B, np.full(M, sa, np.float32), np.full(N, sb, np.float32), 2)
    y3, b3 = orc.scaled_mm(A, B, np.full(M, sa, np.float32), [sb], 3)
    for y, b in ((y1, b1), (y2, b2), (y3, b3)):
        assert np.array_equal(y, y0) and np.array_equal(b, b0)
    # y64 = acc * (double(sa) * double(sb))
    acc = orc.gemm_acc_f64(A, B)
    assert np.array_equal(y0, acc * (float(sa) * float(sb)))


def test_per_token_is_transposed_per_channel(orc):
    """Swapping the operands swaps the roles of token and channel scales."""
    M, N, K = 5, 7, 128
    d = workloads.random_gemm(24, M, N, K, 2)
    sa = d["sa"]
    sb0 = d["sb"][:1]
    y_tok, b_tok = orc.scaled_mm(d["A"], d["B"], sa, sb0, 3)
    y_ch, b_ch = orc.scaled_mm(d["B"], d["A"], sb0, sa, 1)
    assert np.array_equal(y_tok, y_ch.T) and np.array_equal(b_tok, b_ch.T)
    # per-token x channel with one vector constant reduces to the other two
    y2, _ = orc.scaled_mm(d["A"], d["B"], sa, np.full(N, sb0[0], np.float32), 2)
    assert np.array_equal(y2, y_tok)


def test_scaled_mm_bf16_is_rne_of_y64(orc):
    d = workloads.random_gemm(25, 9, 33, 256, 2)
    y64, yb = orc.scaled_mm(d["A"], d["B"], d["sa"], d["sb"], 2)
    # the bf16 result is within half a bf16 ulp of the exact binary64 value
    yv = orc.bf16_to_f32(yb).astype(np.float64)
    nz = y64 != 0
    ulp = np.exp2(np.floor(np.log2(np.abs(y64[nz]))) - 7)
    assert np.all(np.abs(yv[nz] - y64[nz]) <= ulp / 2)


def test_points_match_full(orc):
    d = workloads.random_gemm(26, 17, 41, 320, 2)
    y64, _ = orc.scaled_mm(d["A"], d["B"], d["sa"], d["sb"], 2)
    rows = np.array([0, 16, 5, 9], np.int64)
    cols = np.array([40, 0, 7, 33], np.int64)
    assert np.array_equal(orc.scaled_mm_points(d["A"], d["B"], d["sa"], d["sb"], 2, rows, cols), y64[rows, cols])


def test_nan_codes_propagate(orc):
    A = np.full((1, 32), 0x38, np.uint8)
    B = np.full((2, 32), 0x38, np.uint8)
    B[1, 3] = 0x7F
    y64, yb = orc.scaled_mm(A, B, [1.0], [1.0], 0)
    assert y64[0, 0] == 32 and np.isnan(y64[0, 1])
    assert (yb[0, 1] & 0x7F80) == 0x7F80 and (yb[0, 1] & 0x7F) != 0
    assert orc.has_nan_code(B) and not orc.has_nan_code(A)


def test_pages_weight_stream_accounting():
    """The benchmark counts N*K bytes of E4M3 weight per GEMM launch; with the
    launch counts and times printed on the pages this reproduces their GiB/s."""
    rows, totals = [], []
    with open(os.path.join(GOLDEN, "pages_weight_stream_rates.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if len(line) == 5:
                rows.append(tuple(map(float, line)))
            elif len(line) == 2:
                totals.append(tuple(map(float, line)))
    assert len(rows) == 2 and len(totals) == 1
    for N, K, launches, ms, gibs in rows:
        rate = N * K * launches / (ms * 1e-3) / 2 ** 30
        # the printed ms and GiB/s carry 3-4 significant digits: agree to 0.1%
        assert abs(rate - gibs) <= 1e-3 * gibs, (rate, gibs)
    total_b, gib = totals[0]
    assert abs(total_b / 2 ** 30 - gib) < 5e-5


# --------------------------------------------------------------------------- blockwise scaling (R21)

def _dec(orc, codes):
    return orc.e4m3_decode(codes).astype(np.float64)


def test_block_gemm_matches_groupwise_numpy(orc):
    """The blockwise GEMM against numpy's float64 matmul of the decoded
    operands, one 128-wide K group at a time, each group's product scaled by
    sa[m, g] * sb[n // 128, g] (ragged K and N, distinct scales per block)."""
    g = np.random.default_rng(120)
    M, N, K = 5, 300, 400
    A = workloads.e4m3_codes(g, (M, K))
    B = workloads.e4m3_codes(g, (N, K))
    KB, NB = -(-K // 128), -(-N // 128)
    sa = g.uniform(0.5, 2.0, (M, KB)).astype(np.float32)
    sb = g.uniform(0.5, 2.0, (NB, KB)).astype(np.float32)
    Ad, Bd = _dec(orc, A), _dec(orc, B)
    want = np.zeros((M, N))
    for gi in range(KB):
        k0, k1 = gi * 128, min(K, gi * 128 + 128)
        part = Ad[:, k0:k1] @ Bd[:, k0:k1].T
        want += part * (sa[:, gi].astype(np.float64)[:, None] * sb[np.arange(N) // 128, gi].astype(np.float64)[None, :])
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    got = orc.scaled_mm_block_points(A, B, sa, sb, rows.ravel(), cols.ravel()).reshape(M, N)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-9)


def test_block_gemm_with_uniform_scales_is_token_channel(orc):
    """Scales constant along K reduce the blockwise GEMM to the per-token x
    per-channel one (gran 2) of the same operands."""
    g = np.random.default_rng(121)
    M, N, K = 3, 256, 512
    A = workloads.e4m3_codes(g, (M, K))
    B = workloads.e4m3_codes(g, (N, K))
    a = g.uniform(0.5, 2.0, M).astype(np.float32)
    b = g.uniform(0.5, 2.0, 2).astype(np.float32)
    sa = np.repeat(a[:, None], 4, axis=1)
    sb = np.repeat(b[:, None], 4, axis=1)
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    got = orc.scaled_mm_block_points(A, B, sa, sb, rows.ravel(), cols.ravel())
    want = orc.scaled_mm_points(A, B, a, np.repeat(b, 128), 2, rows.ravel(), cols.ravel())
    assert np.allclose(got, want, rtol=1e-13, atol=0)


def test_per_token_group_quant_is_per_token_on_groups(orc):
    """Each 128-wide group quantised exactly like a per-token row of its own
    (the rows reshaped so that each group is a row), ragged last group."""
    g = np.random.default_rng(122)
    x = workloads.bf16_normal_with_outliers(g, (4, 512))
    q, s = orc.quant_per_token_group(x)
    q2, s2 = orc.quant_per_token(x.reshape(16, 128))
    assert np.array_equal(q, q2.reshape(4, 512)) and np.array_equal(s, s2.reshape(4, 4))
    x3 = workloads.bf16_normal(g, (2, 400))
    q3, s3 = orc.quant_per_token_group(x3)
    assert s3.shape == (2, 4)
    qt, st = orc.quant_per_token(x3[:, 384:])
    assert np.array_equal(q3[:, 384:], qt) and np.array_equal(s3[:, 3], st)


def test_weight_block_quant(orc):
    """Block scales from numpy's per-block amax / 448 in binary32, codes the
    static quantisation of each block by its scale; the amax element of every
    block maps to +-448; an all-zero block gets scale 1 and zero codes."""
    g = np.random.default_rng(123)
    w = workloads.bf16_normal(g, (256, 384), std=0.02)
    w[:128, 128:256] = 0
    q, s = orc.quant_weight_block(w)
    wf = (w.astype(np.uint32) << 16).view(np.float32)
    amax = np.abs(wf).reshape(2, 128, 3, 128).max(axis=(1, 3))
    want_s = np.where(amax == 0, np.float32(1.0), amax / np.float32(448.0)).astype(np.float32)
    assert np.array_equal(s, want_s)
    for nb in range(2):
        for gb in range(3):
            blk = w[nb * 128:(nb + 1) * 128, gb * 128:(gb + 1) * 128]
            assert np.array_equal(q[nb * 128:(nb + 1) * 128, gb * 128:(gb + 1) * 128],
                                  orc.quant_static(blk, float(s[nb, gb])))
            if amax[nb, gb] > 0:
                assert np.max(q[nb * 128:(nb + 1) * 128, gb * 128:(gb + 1) * 128] & 0x7F) == 0x7E
    assert s[0, 1] == 1.0 and np.all(q[:128, 128:256] == 0)
