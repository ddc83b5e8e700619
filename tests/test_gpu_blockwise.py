"""GPU parity of blockwise FP8 scaling (128 x 128 weight blocks, 128-wide token
groups) against the CPU oracle: the two quantisers byte-exact, and the GEMM
with FP8_GRAN_BLOCK_128 on both kernels (decode M <= 32, tile M >= 33) within
the acceptance bound, every output of the small cases and sampled outputs of
the workload-sized ones."""
import numpy as np
import pytest
import torch

import workloads
from helpers import Guarded, bf16_bits_to_f64, host_bits, to_dev_bf16, to_dev_e4m3, to_dev_f32

pytestmark = pytest.mark.gpu

BLOCK = 128
GRAN_BLOCK = 4


@pytest.fixture(scope="module")
def fp8():
    import fp8_w8a8_scaled_gb300 as f
    f.clear_device_error()
    yield f
    assert f.get_device_error() == 0


def dev_scales(s):
    return torch.from_numpy(np.ascontiguousarray(s, np.float32)).cuda()


def run_block_mm(fp8, A, B, sa, sb):
    """Device operands and scales; returns the bf16 output bits (guard bands
    around the output checked)."""
    M, N = A.shape[0], B.shape[0]
    buf = Guarded(M * N * 2)
    out = buf.view(torch.bfloat16, (M, N))
    fp8.fp8_scaled_mm(A, B, sa, sb, GRAN_BLOCK, out=out)
    torch.cuda.synchronize()
    assert buf.intact(), "write outside the output buffer"
    return host_bits(out)


def block_check(orc, A, B, sa, sb, y_bits, what, rows=None, cols=None):
    """Outputs (all, or the listed points) against the oracle's blockwise GEMM.

    Bound: 1e-2 |ref| + 1e-3 sqrt(K) max_g(sa[m,g] sb[n/128,g]) -- the
    acceptance bound with the largest scale product of the output standing in
    for the single one -- plus the binary32 accumulation bound of the kernels'
    arithmetic: each k-block's sum comes from the tensor core (at most
    ceil(K/32) + 1 roundings of a partial sum in all), and each scaled
    k-block sum is rounded once more when it is added, so
    |error| <= (ceil(K/32) + ceil(K/128) + 1) 2^-23 sum_g s_g sum_k |a_k b_k|.
    Returns the largest err / acceptance bound."""
    M, K = A.shape
    N = B.shape[0]
    KB = -(-K // BLOCK)
    if rows is None:
        rr, cc = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        rows, cols = rr.ravel(), cc.ravel()
    rows = np.asarray(rows, np.int64)
    cols = np.asarray(cols, np.int64)
    y64 = orc.scaled_mm_block_points(A, B, sa, sb, rows, cols)
    abs_sum = orc.scaled_mm_block_points(np.asarray(A) & 0x7F, np.asarray(B) & 0x7F, np.abs(sa), np.abs(sb),
                                         rows, cols)
    sa64 = np.asarray(sa, np.float64).reshape(M, KB)
    sb64 = np.asarray(sb, np.float64).reshape(-(-N // BLOCK), KB)
    smax = np.max(np.abs(sa64[rows] * sb64[cols // BLOCK]), axis=1)
    bound = 1e-2 * np.abs(y64) + 1e-3 * np.sqrt(K) * smax
    acc = (-(-K // 32) + KB + 1) * 2.0 ** -23 * abs_sum
    y = bf16_bits_to_f64(np.asarray(y_bits).reshape(M, N)[rows, cols])
    assert not np.any(np.isnan(y)), f"{what}: NaN in GPU output"
    err = np.abs(y - y64)
    bad = ~(err <= bound + acc)
    ratio = float(np.max(err / np.where(bound > 0, bound, np.inf))) if err.size else 0.0
    assert int(bad.sum()) == 0, f"{what}: {int(bad.sum())} of {err.size} outputs outside the bound"
    print(f"{what}: max err/bound {ratio:.4f}")
    return ratio


# ------------------------------------------------------------------ quantisers

GROUP_SHAPES = [(1, 128), (3, 5120), (5, 272), (17, 400), (64, 17408), (2, 16)]


@pytest.mark.parametrize("M,K", GROUP_SHAPES)
def test_group_quant_matches_oracle(fp8, orc, M, K):
    x = workloads.bf16_normal_with_outliers(workloads.rng(7000 + M + K), (M, K))
    q, s = fp8.quant_per_token_group(to_dev_bf16(x))
    torch.cuda.synchronize()
    wq, ws = orc.quant_per_token_group(x)
    assert s.shape == (M, -(-K // BLOCK))
    assert np.array_equal(host_bits(s), ws)
    assert np.array_equal(host_bits(q), wq)


def test_group_quant_special_groups(fp8, orc):
    """A zero group (scale 1), a group with a NaN (left out of the max), a group
    with an infinity (scale inf): each touches only its own group."""
    M, K = 2, 512
    x = workloads.bf16_normal(workloads.rng(7100), (M, K))
    x[0, 0:128] = 0
    x[0, 130] = 0x7FC0
    x[1, 300] = 0x7F80
    q, s = fp8.quant_per_token_group(to_dev_bf16(x))
    torch.cuda.synchronize()
    wq, ws = orc.quant_per_token_group(x)
    qh, sh = host_bits(q), host_bits(s)
    assert sh[0, 0] == 1.0 and np.isinf(sh[1, 2])
    assert np.array_equal(sh, ws)
    nan_w = (wq & 0x7F) == 0x7F
    assert np.array_equal(qh[~nan_w], wq[~nan_w])
    assert np.all((qh[nan_w] & 0x7F) == 0x7F)
    assert np.array_equal(qh[1, :256], wq[1, :256]) and np.array_equal(qh[1, 384:], wq[1, 384:])


BLOCK_SHAPES = [(128, 128), (300, 400), (8, 16), (1032, 5120), (10240, 5120)]


@pytest.mark.parametrize("N,K", BLOCK_SHAPES)
def test_weight_block_quant_matches_oracle(fp8, orc, N, K):
    w = workloads.bf16_normal(workloads.rng(7200 + N + K), (N, K), std=0.02)
    if N >= 256 and K >= 256:
        w[128:256, 128:256] = 0  # an all-zero block: scale 1.0
    q, s = fp8.quant_weight_block(to_dev_bf16(w))
    torch.cuda.synchronize()
    wq, ws = orc.quant_weight_block(w)
    assert s.shape == (-(-N // BLOCK), -(-K // BLOCK))
    assert np.array_equal(host_bits(s), ws)
    assert np.array_equal(host_bits(q), wq)


def test_quantisers_empty(fp8):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s = fp8.quant_per_token_group(x)
    qw, sw = fp8.quant_weight_block(x)
    torch.cuda.synchronize()
    assert q.shape == (0, 256) and s.shape == (0, 2) and qw.shape == (0, 256) and sw.shape == (0, 2)


# ------------------------------------------------------------------ GEMM, random codes

SHAPES = [(1, 136, 400), (3, 8, 16), (5, 1032, 5120), (16, 264, 272), (16, 128, 128),
          (17, 264, 400), (32, 10240, 1040), (33, 1000, 272), (129, 520, 1040), (200, 8, 4096), (300, 1032, 2064),
          (1100, 4504, 400)]  # the last: a short last round split into 128-channel half tiles


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_block_gemm_random_codes(fp8, orc, M, N, K):
    c = workloads.random_gemm(8000 + M * 7 + N * 3 + K, M, N, K, GRAN_BLOCK)
    want = fp8.KERNEL_DECODE_SPLITK if M <= 32 else fp8.KERNEL_PREFILL
    assert fp8.describe_dispatch(M, N, K, GRAN_BLOCK) == want
    y = run_block_mm(fp8, to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"]), dev_scales(c["sa"]), dev_scales(c["sb"]))
    block_check(orc, c["A"], c["B"], c["sa"], c["sb"], y, f"{M}x{N}x{K} blockwise")


@pytest.mark.parametrize("M,N,K,S", [(1, 34816, 1040, 1), (16, 10240, 256, 1), (16, 12800, 400, 2),
                                     (16, 10232, 5136, 3), (2, 7168, 4096, 4), (16, 6144, 1040, 5),
                                     (5, 5120, 8192, 6), (4, 4096, 2064, 7), (11, 3840, 1552, 8),
                                     (1, 128, 5120, 0), (9, 1032, 17408, 0), (32, 10240, 5120, 3),
                                     (17, 5120, 8192, 6), (20, 1032, 4096, 0)])
def test_block_decode_modes(fp8, orc, M, N, K, S):
    """The blockwise decode kernel's modes on a 152-SM GB300 -- clusters of S
    CTAs per 128-channel tile for every S from 1 to 8 (rows split unevenly
    among the S CTAs for S = 3, 5, 6, 7; ragged last tiles; K ranges split
    unevenly) and the stream-K grid (S = 0) -- every output against the
    oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert fp8.decode_split(M, N, K, sms, granularity=GRAN_BLOCK) == S
    assert fp8.decode_exact(M, N, K, granularity=GRAN_BLOCK) == 0
    c = workloads.random_gemm(8600 + M + N + K, M, N, K, GRAN_BLOCK)
    y = run_block_mm(fp8, to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"]), dev_scales(c["sa"]), dev_scales(c["sb"]))
    block_check(orc, c["A"], c["B"], c["sa"], c["sb"], y, f"{M}x{N}x{K} blockwise split {S}")


def test_block_gemm_scales_select_blocks(fp8, orc):
    """Scales zero everywhere but one (token, k-group) and one (weight block,
    k-group): only that group's products survive, in that block's outputs."""
    M, N, K = 4, 384, 512
    c = workloads.random_gemm(8100, M, N, K, GRAN_BLOCK)
    sa = np.zeros((M, 4), np.float32)
    sb = np.zeros((3, 4), np.float32)
    sa[2, 1] = 0.5
    sb[1, 1] = 0.25
    for m_rows in (M, 24, 40):  # decode kernel (16- and 32-token tiles), then tile kernel
        A = np.resize(c["A"], (m_rows, K))
        sam = np.zeros((m_rows, 4), np.float32)
        sam[2, 1] = 0.5
        y = run_block_mm(fp8, to_dev_e4m3(A), to_dev_e4m3(c["B"]), dev_scales(sam), dev_scales(sb))
        yf = bf16_bits_to_f64(y)
        assert np.all(yf[np.arange(m_rows) != 2] == 0)
        assert np.all(yf[2, :128] == 0) and np.all(yf[2, 256:] == 0)
        block_check(orc, A, c["B"], sam, sb, y, f"M={m_rows} one live group")


def test_block_gemm_rerun_is_bitwise_identical(fp8):
    M, N, K = 8, 2048, 5120
    c = workloads.random_gemm(8200, M, N, K, GRAN_BLOCK)
    A, B = to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"])
    sa, sb = dev_scales(c["sa"]), dev_scales(c["sb"])
    y0 = run_block_mm(fp8, A, B, sa, sb)
    for _ in range(3):
        assert np.array_equal(run_block_mm(fp8, A, B, sa, sb), y0)


# ------------------------------------------------------------------ end to end, workload shapes

def quantised_block_operands(fp8, orc, M, N, K, seed):
    """bf16 activations with outliers and N(0, 0.02) weights, quantised on the
    GPU per token group / per weight block and checked byte-exact against the
    oracle's quantisers."""
    g = workloads.rng(seed)
    x = workloads.bf16_normal_with_outliers(g, (M, K))
    w = workloads.bf16_normal(g, (N, K), std=0.02)
    qa, sa = fp8.quant_per_token_group(to_dev_bf16(x))
    qb, sb = fp8.quant_weight_block(to_dev_bf16(w))
    wa, wsa = orc.quant_per_token_group(x)
    wb, wsb = orc.quant_weight_block(w)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(qa), wa) and np.array_equal(host_bits(sa), wsa)
    assert np.array_equal(host_bits(qb), wb) and np.array_equal(host_bits(sb), wsb)
    return qa, qb, sa, sb, wa, wb, wsa, wsb


@pytest.mark.parametrize("M", [1, 8, 16, 32])
def test_block_qkv_decode(fp8, orc, M):
    """Merged QKV (N 10240, K 5120) at decode M, every output."""
    qa, qb, sa, sb, wa, wb, wsa, wsb = quantised_block_operands(fp8, orc, M, 10240, 5120, 8300 + M)
    y = run_block_mm(fp8, qa, qb, sa, sb)
    block_check(orc, wa, wb, wsa, wsb, y, f"QKV M={M} blockwise")


@pytest.mark.parametrize("M,N,K", [(64, 34816, 5120), (2048, 10240, 5120)])
def test_block_prefill_sampled(fp8, orc, M, N, K):
    """gate|up at M 64 and a 2048-token prefill chunk of QKV: 20000 sampled
    outputs, plus every output of the first and last 128 x 128 blocks."""
    qa, qb, sa, sb, wa, wb, wsa, wsb = quantised_block_operands(fp8, orc, M, N, K, 8400 + M)
    y = run_block_mm(fp8, qa, qb, sa, sb)
    g = workloads.rng(8500 + M)
    rows = g.integers(0, M, 20000)
    cols = g.integers(0, N, 20000)
    corner = np.array([(r, cc) for r in list(range(min(M, 128))) + list(range(max(0, M - 128), M))
                       for cc in list(range(128)) + list(range(N - 128, N))], np.int64)
    rows = np.concatenate([rows, corner[:, 0]])
    cols = np.concatenate([cols, corner[:, 1]])
    block_check(orc, wa, wb, wsa, wsb, y, f"{M}x{N}x{K} blockwise", rows, cols)
