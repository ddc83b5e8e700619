"""GPU parity of the weight-only FP8 GEMM (W8A16: bf16 activations, E4M3
weights) against the CPU oracle: the CUDA-core GEMV (M <= 4, every output),
the widen-on-chip decode kernel (M <= 32, every output), the weight widening
entry point (byte-exact), the large-M
tile kernel (ragged shapes, every output; a 2048 x 10240 x 5120 prefill
chunk, sampled outputs), and the invariants (determinism, dispatch, NaN
codes)."""
import numpy as np
import pytest
import torch

import workloads
from helpers import Guarded, bf16_bits_to_f64, host_bits, to_dev_bf16, to_dev_e4m3, to_dev_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    import fp8_w8a8_scaled_gb300 as f
    f.clear_device_error()
    yield f
    assert f.get_device_error() == 0


def run_w16(fp8, x, W, sb, gran, flags=0):
    M, N = x.shape[0], W.shape[0]
    buf = Guarded(M * N * 2)
    out = buf.view(torch.bfloat16, (M, N))
    fp8.w8a16_mm(x, W, sb, gran, out=out, flags=flags)
    torch.cuda.synchronize()
    assert buf.intact(), "write outside the output buffer"
    return host_bits(out)


def _dec_bf16(bits):
    return bf16_bits_to_f64(bits)


def w16_bound(x_bits, W_codes, sb, per_channel, y64, orc, K, mma_k):
    """Acceptance bound of the weight-only GEMM: 1e-2 |ref| + 1e-3 sa sb sqrt(K)
    with sa = max_k |x[m,k]| / 448 (the scale a per-token quantisation of the
    row would take), plus the binary32 accumulation bound of the tensor core's
    sums of mma_k-wide chunks (ceil(K/mma_k) + 1) 2^-23 sb sum_k |x w|."""
    xa = np.abs(_dec_bf16(x_bits))
    sa = xa.max(axis=1) / 448.0
    sbv = np.asarray(sb, np.float64).reshape(-1)
    sbn = sbv if per_channel else np.full(W_codes.shape[0], sbv[0])
    wabs = np.abs(orc.e4m3_decode(W_codes))
    abs_sum = (xa @ wabs.T) * sbn[None, :]
    acc = (-(-K // mma_k) + 1) * 2.0 ** -23 * abs_sum
    return 1e-2 * np.abs(y64) + 1e-3 * sa[:, None] * sbn[None, :] * np.sqrt(K), acc


def operands(seed, M, N, K, per_channel=True, weights="codes"):
    g = workloads.rng(seed)
    x = workloads.bf16_normal_with_outliers(g, (M, K))
    if weights == "codes":
        W = workloads.e4m3_codes(g, (N, K))
        sb = workloads.uniform_f32(g, (N if per_channel else 1,), 0.5, 2.0) * np.float32(1e-3)
    else:  # N(0, 0.02) weights quantised per channel by the oracle (amax / 448)
        import oracle
        w = workloads.bf16_normal(g, (N, K), std=0.02)
        W, sb = oracle.quant_per_token(w if per_channel else w.reshape(1, -1))
        W = W.reshape(N, K)
    return x, W, np.asarray(sb, np.float32)


def check(fp8, orc, x, W, sb, per_channel, what, flags=0):
    M, K = x.shape
    y = run_w16(fp8, to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb), 1 if per_channel else 0, flags)
    y64, _ = orc.w8a16_mm(x, W, sb, per_channel)
    bound, acc = w16_bound(x, W, sb, per_channel, y64, orc, K, 16)
    yf = bf16_bits_to_f64(y)
    err = np.abs(yf - y64)
    assert not np.any(np.isnan(yf)), f"{what}: NaN"
    bad = ~(err <= bound + acc)
    ratio = float(np.max(err / np.where(bound > 0, bound, np.inf)))
    assert int(bad.sum()) == 0, f"{what}: {int(bad.sum())} of {err.size} outside the bound (max {ratio:.3g})"
    print(f"{what}: max err/bound {ratio:.4f}")
    return y


# ------------------------------------------------------------------ decode kernel (M <= 32)

SHAPES = [(1, 8, 16), (3, 136, 272), (16, 128, 128), (5, 1032, 5120), (16, 264, 1040), (17, 136, 400),
          (32, 1032, 2064), (24, 520, 1552)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("per_channel", [True, False])
def test_w16_decode_random_codes(fp8, orc, M, N, K, per_channel):
    # M <= 4 runs the GEMV, the others the decode kernel
    want = fp8.KERNEL_W16_GEMV if M <= 4 else fp8.KERNEL_W16_DECODE
    assert fp8.w8a16_describe_dispatch(M, N, K) == want
    x, W, sb = operands(9000 + M + N + K, M, N, K, per_channel)
    check(fp8, orc, x, W, sb, per_channel, f"w16 {M}x{N}x{K} pc={per_channel}")


# (M, N, K) with 29 to 100 output tiles (tiles shared by 3 to 10 CTAs of the
# persistent grid), one with a ragged last tile and a ragged k-block
TILE_COUNT_SHAPES = [(3, 12800, 512), (5, 6400, 640), (8, 5632, 768), (2, 4608, 1024), (16, 4104, 1040),
                     (1, 3712, 1024)]


@pytest.mark.parametrize("M,N,K", TILE_COUNT_SHAPES)
def test_w16_decode_tile_counts(fp8, orc, M, N, K):
    """Every output against the oracle, and a rerun bitwise."""
    x, W, sb = operands(9050 + N, M, N, K, True)
    y = check(fp8, orc, x, W, sb, True, f"w16 {M}x{N}x{K}")
    assert np.array_equal(run_w16(fp8, to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb), 1), y)


@pytest.mark.parametrize("M", [1, 4, 8, 16, 32])
def test_w16_decode_qkv(fp8, orc, M):
    """Merged QKV (N 10240, K 5120), per-channel quantised N(0, 0.02) weights,
    every output."""
    x, W, sb = operands(9100 + M, M, 10240, 5120, True, weights="quant")
    check(fp8, orc, x, W, sb, True, f"w16 QKV M={M}", flags=fp8.FLAG_WEIGHTS_STATIC)


def test_w16_decode_rerun_bitwise(fp8):
    x, W, sb = operands(9200, 8, 2048, 5120)
    xd, Wd, sbd = to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb)
    y0 = run_w16(fp8, xd, Wd, sbd, 1)
    for _ in range(3):
        assert np.array_equal(run_w16(fp8, xd, Wd, sbd, 1), y0)


def test_w16_rows_independent(fp8):
    """Row m of an M=16 call against the same row in a 5-token call: same
    16-token tile of the decode kernel, same K division, so bitwise."""
    x, W, sb = operands(9300, 16, 1032, 2064)
    xd, Wd, sbd = to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb)
    full = run_w16(fp8, xd, Wd, sbd, 1)
    for m in (0, 9, 11):
        assert fp8.w8a16_describe_dispatch(5, 1032, 2064) == fp8.KERNEL_W16_DECODE
        assert np.array_equal(run_w16(fp8, xd[m:m + 5].contiguous(), Wd, sbd, 1)[0], full[m])


def test_w16_gemv_rows_independent(fp8):
    """The GEMV: each token's sum runs in its own registers in a fixed order,
    so a row alone, in a pair and among four gives the same bits."""
    x, W, sb = operands(9310, 4, 2056, 5120)
    xd, Wd, sbd = to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb)
    assert fp8.w8a16_describe_dispatch(4, 2056, 5120) == fp8.KERNEL_W16_GEMV
    full = run_w16(fp8, xd, Wd, sbd, 1)
    for m in range(4):
        assert np.array_equal(run_w16(fp8, xd[m:m + 1].contiguous(), Wd, sbd, 1)[0], full[m])
    assert np.array_equal(run_w16(fp8, xd[1:3].contiguous(), Wd, sbd, 1), full[1:3])


# (M, N, K) for the GEMV: one 16-byte vector per row (K 16), rows fewer than
# the CTAs (N 8, 24), 512-byte segments with a ragged last one (K 4112, 272),
# the largest K for one and for four tokens (the bf16 token copy at its 40 KB
# limit), a long K (the down projection), warps with one to several rows
# (N 20000: 132 rows per CTA, 5 or 6 per warp)
GEMV_SHAPES = [(1, 8, 16), (2, 24, 4112), (3, 1032, 5120), (4, 2056, 5120), (1, 5120, 17408), (1, 600, 20480),
               (4, 304, 272), (2, 20000, 1024)]


@pytest.mark.parametrize("M,N,K", GEMV_SHAPES)
@pytest.mark.parametrize("per_channel", [True, False])
def test_w16_gemv(fp8, orc, M, N, K, per_channel):
    """Every output of the GEMV against the oracle at the acceptance bound
    (its binary32 sums are well inside the tensor-core accumulation allowance
    the bound carries), and a rerun bitwise."""
    assert fp8.w8a16_describe_dispatch(M, N, K) == fp8.KERNEL_W16_GEMV
    x, W, sb = operands(9320 + M + N + K, M, N, K, per_channel, weights="codes" if K <= 5120 else "quant")
    y = check(fp8, orc, x, W, sb, per_channel, f"w16 gemv {M}x{N}x{K} pc={per_channel}")
    assert np.array_equal(run_w16(fp8, to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb), 1 if per_channel else 0), y)


@pytest.mark.parametrize("M", [4, 8])
def test_w16_nan_weight_code(fp8, orc, M):
    """A NaN weight code: that output channel is NaN for every token, the
    others finite (M 4: the GEMV; M 8: the decode kernel)."""
    x, W, sb = operands(9400, M, 136, 272)
    W[7, 100] = 0x7F
    y = run_w16(fp8, to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb), 1)
    assert np.all(np.isnan(bf16_bits_to_f64(y[:, 7])))
    assert not np.any(np.isnan(bf16_bits_to_f64(np.delete(y, 7, axis=1))))


@pytest.mark.parametrize("M", [4, 32, 256])
@pytest.mark.parametrize("per_channel", [True, False])
def test_w16_every_code_exact(fp8, orc, M, per_channel):
    """Every non-NaN E4M3 weight code through the on-chip widening, exactly:
    token m is one-hot at k = m, so y[m, n] = bf16(dec(W[n, m]) * 1) is the
    decoded code itself (subnormal codes and signed zeros included); over the
    256 rows n the codes (n + 8 m) mod 256 cover all 254 non-NaN codes for
    every m.  M 4 runs the GEMV, M 32 the decode kernel, M 256 the tile
    kernel."""
    N, K = 256, 256
    x = np.zeros((M, K), np.uint16)
    x[np.arange(M), np.arange(M)] = 0x3F80  # bf16 1.0
    n, k = np.meshgrid(np.arange(N), np.arange(K), indexing="ij")
    W = ((n + 8 * k) % 256).astype(np.uint8)
    W[(W & 0x7F) == 0x7F] = 0x00  # NaN codes would turn a whole row into NaN
    sb = np.ones(N if per_channel else 1, np.float32)
    y = _dec_bf16(run_w16(fp8, to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb), 1 if per_channel else 0))
    want = orc.e4m3_decode(W[:, :M]).T
    assert np.array_equal(y, want)
    y64, _ = orc.w8a16_mm(x, W, sb, per_channel)
    assert np.array_equal(y64, want)


def test_w16_nan_weight_code_tile_kernel(fp8, orc):
    """A NaN weight code through the tile kernel's widening: that output
    channel is NaN for every token, the others finite."""
    x, W, sb = operands(9410, 40, 296, 528)
    W[7, 100] = 0x7F
    W[290, 517] = 0xFF
    assert fp8.w8a16_describe_dispatch(40, 296, 528) == fp8.KERNEL_W16_DENSE
    y = _dec_bf16(run_w16(fp8, to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb), 1))
    assert np.all(np.isnan(y[:, [7, 290]]))
    assert not np.any(np.isnan(np.delete(y, [7, 290], axis=1)))


def test_w16_m_zero(fp8):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((64, 64), dtype=torch.float8_e4m3fn, device="cuda")
    y = fp8.w8a16_mm(x, W, to_dev_f32([1.0]), 0)
    assert y.shape == (0, 64)


# ------------------------------------------------------------------ large-M branch

@pytest.mark.parametrize("per_channel", [True, False])
def test_widen_weight_bitexact(fp8, orc, per_channel):
    g = workloads.rng(9500)
    W = workloads.e4m3_codes(g, (300, 400))
    W[3, 5] = 0x7F
    W[4, 6] = 0xFF
    sb = (g.uniform(0.25, 4.0, 300 if per_channel else 1) * 1e-3).astype(np.float32)
    out = fp8.widen_weight(to_dev_e4m3(W), to_dev_f32(sb), 1 if per_channel else 0)
    torch.cuda.synchronize()
    want = orc.dequant_weight_bf16(W, sb, per_channel)
    got = host_bits(out)
    nan_w = (want & 0x7F80) == 0x7F80
    assert np.array_equal(got[~nan_w], want[~nan_w])
    assert np.all((got[nan_w] & 0x7F80) == 0x7F80) and np.all((got[nan_w] & 0x7F) != 0)


@pytest.mark.parametrize("M,N,K", [(33, 136, 272), (64, 1032, 2064), (300, 520, 1040), (129, 8, 5136),
                                   (1100, 4504, 272), (200, 392, 400)])
@pytest.mark.parametrize("per_channel", [True, False])
def test_w16_dense_branch(fp8, orc, M, N, K, per_channel):
    """Large M: the tile kernel (weight widened on chip, bf16 MMAs with fp32
    accumulation over the whole K in tensor memory, the scale in binary32
    before the one bf16 rounding) against the method's exact result: the
    acceptance bound plus the binary32 accumulation bound of the tensor
    core's 16-wide chunks; ragged M, N and K.  1100 x 4504 has more tiles
    than SMs and a short last round, which runs as half tiles; 300 x 520 ends
    in a weight tile of one half, 200 x 392 in one whose second half has 8 rows."""
    assert fp8.w8a16_describe_dispatch(M, N, K) == fp8.KERNEL_W16_DENSE
    x, W, sb = operands(9600 + M, M, N, K, per_channel, weights="quant")
    y = bf16_bits_to_f64(run_w16(fp8, to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb), 1 if per_channel else 0))
    y64, _ = orc.w8a16_mm(x, W, sb, per_channel)
    bound, acc = w16_bound(x, W, sb, per_channel, y64, orc, K, 16)
    err = np.abs(y - y64)
    assert np.all(err <= bound + acc)
    print(f"w16 dense {M}x{N}x{K} pc={per_channel}: max err/acceptance bound {float(np.max(err / bound)):.4f}")


def test_w16_dense_qkv_m2048(fp8, orc):
    """The large-M branch at a prefill chunk of the merged QKV projection
    (M 2048, N 10240, K 5120; activations N(0,1) with 1% outliers, weights
    N(0, 0.02) quantised per channel): 20000 sampled outputs plus the first
    and last 128 x 128 corner of the output, against the oracle at the same
    bound (no allowance beyond the tensor core's accumulation)."""
    M, N, K = 2048, 10240, 5120
    x, W, sb = operands(9700, M, N, K, True, weights="quant")
    y = run_w16(fp8, to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb), 1)
    g = workloads.rng(9701)
    rows = g.integers(0, M, 20000)
    cols = g.integers(0, N, 20000)
    corner = np.array([(r, c) for r in list(range(128)) + list(range(M - 128, M))
                       for c in list(range(128)) + list(range(N - 128, N))], np.int64)
    rows = np.concatenate([rows, corner[:, 0]])
    cols = np.concatenate([cols, corner[:, 1]])
    y64 = orc.w8a16_points(x, W, sb, True, rows, cols)
    xa = np.abs(_dec_bf16(x))
    wa = np.abs(orc.e4m3_decode(W))
    abs_sum = np.concatenate([np.einsum("ij,ij->i", xa[rows[i:i + 4096]], wa[cols[i:i + 4096]])
                              for i in range(0, rows.size, 4096)]) * sb[cols].astype(np.float64)
    sa = xa.max(axis=1)[rows] / 448.0
    bound = 1e-2 * np.abs(y64) + 1e-3 * sa * sb[cols].astype(np.float64) * np.sqrt(K)
    acc = (-(-K // 16) + 1) * 2.0 ** -23 * abs_sum
    yf = bf16_bits_to_f64(y[rows, cols])
    err = np.abs(yf - y64)
    assert not np.any(np.isnan(yf))
    assert np.all(err <= bound + acc), int(np.sum(err > bound + acc))
    print(f"w16 dense 2048x10240x5120: max err/acceptance bound {float(np.max(err / bound)):.4f}")
