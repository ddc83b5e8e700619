"""GPU parity of the activation quantisers against the CPU oracle: the E4M3
bytes and the per-token scales must be bit-exact."""
import numpy as np
import pytest
import torch

import workloads
from helpers import Guarded, host_bits, to_dev_bf16, to_dev_e4m3, to_dev_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    import fp8_w8a8_scaled_gb300 as f
    f.clear_device_error()
    yield f
    assert f.get_device_error() == 0


ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(4096, 16)
NAN_MASK = ((ALL_BF16 & 0x7F80) == 0x7F80) & ((ALL_BF16 & 0x7F) != 0)


@pytest.mark.parametrize("s", [1.0, 1 / 56, 0.37, 3.3e-3, 2.0 ** -10, 7.5, 1e-30, 1e30, 2.0 ** -130])
def test_static_quant_every_bf16_value(fp8, orc, s):
    """Every bf16 bit pattern through q = e4m3(x / s) for a sweep of scales."""
    s = float(np.float32(s))
    x = to_dev_bf16(ALL_BF16)
    q = host_bits(fp8.quant_fp8_static(x, to_dev_f32(s)))
    want = orc.quant_static(ALL_BF16, s)
    ok = ~NAN_MASK
    assert np.array_equal(q[ok], want[ok]), np.argwhere((q != want) & ok)[:10]
    # NaN inputs: a NaN code (the oracle's reading is 0x7F; record what the hardware emits)
    assert np.all((q[NAN_MASK] & 0x7F) == 0x7F)


def test_static_quant_near_midpoints(fp8, orc):
    """Quotients x / s within a few binary32 units of an E4M3 rounding midpoint
    (where a reciprocal multiply could pick the other code): for 64 bf16 x and
    midpoints across the whole range (the subnormal steps, 2^-10 next to zero,
    the normal binades up to 432 below the saturation at 448), s is chosen so
    that x0 / s lands 0, +-1, +-2 or +-4 units from the midpoint; every x of
    the vector, the ones near midpoints and the others, bit-exact."""
    g = workloads.rng(33)
    xs = workloads.bf16_normal(g, (1, 64))
    xs[0, :4] = [0x3F80, 0x4140, 0xBF80, 0x3C23]      # 1, 12, -1, ~0.01
    e4 = orc.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8))   # 0 .. 448, ascending
    mids = (e4[:-1] + e4[1:]) / 2.0
    pick = np.unique(np.concatenate([mids[:10], mids[10::7], mids[-3:]]))
    dev_x = to_dev_bf16(xs)
    x_f = orc.bf16_to_f32(xs[0])
    checked = 0
    for j, m in enumerate(pick):
        x0 = float(x_f[j % 4])
        base = np.float32(abs(x0) / m)
        for k in (0, 1, -1, 2, -2, 4, -4):
            s = base
            for _ in range(abs(k)):
                s = np.nextafter(s, np.float32(np.inf) if k > 0 else np.float32(0), dtype=np.float32)
            q = host_bits(fp8.quant_fp8_static(dev_x, to_dev_f32(float(s))))
            assert np.array_equal(q, orc.quant_static(xs, float(s))), (m, k, float(s))
            checked += 1
    assert checked == 7 * len(pick)


def test_static_quant_nan_encoding(fp8):
    """The hardware conversion's NaN code for a positive and a negative NaN."""
    x = np.zeros((1, 16), np.uint16)
    x[0, 0] = 0x7FC0
    x[0, 1] = 0xFFC0
    q = host_bits(fp8.quant_fp8_static(to_dev_bf16(x), to_dev_f32(1.0)))
    print("NaN codes:", hex(int(q[0, 0])), hex(int(q[0, 1])))
    assert (q[0, 0] & 0x7F) == 0x7F and (q[0, 1] & 0x7F) == 0x7F


def test_static_quant_large_and_guarded(fp8, orc):
    g = workloads.rng(30)
    x = workloads.bf16_normal(g, (64, 5120))
    s = float(workloads.STATIC_INPUT_SCALE)
    buf = Guarded(64 * 5120)
    out = buf.view(torch.float8_e4m3fn, (64, 5120))
    fp8.quant_fp8_static(to_dev_bf16(x), to_dev_f32(s), out=out)
    assert np.array_equal(host_bits(out), orc.quant_static(x, s))
    assert buf.intact()


@pytest.mark.parametrize("M,K", [(1, 16), (3, 48), (7, 5120), (64, 5120), (33, 8192), (5, 8208), (700, 8192), (999, 48),
                                 (9, 17408), (2, 32768), (3, 40000), (2, 65536), (1, 65552), (1, 131072)])
def test_per_token_shapes(fp8, orc, M, K):
    """Covers every kernel variant: 128x8, 256x16 and 512x16 register-resident
    rows and the two-pass path for rows beyond 65536."""
    g = workloads.rng(31 + M + K)
    x = workloads.bf16_normal_with_outliers(g, (M, K))
    x[0, : min(K, 16)] = 0           # a partly-zero row
    if M > 2:
        x[2] = 0                     # an all-zero row: scale 1.0, codes 0
    buf = Guarded(M * K)
    out = buf.view(torch.float8_e4m3fn, (M, K))
    q, s = fp8.quant_fp8_per_token(to_dev_bf16(x), out=out)
    wq, ws = orc.quant_per_token(x)
    assert np.array_equal(host_bits(s), ws)
    assert np.array_equal(host_bits(q), wq)
    assert buf.intact()


def test_per_token_prefill_activations(fp8, orc):
    """Prefill activations: M=2048, K=5120, N(0,1) with 1% outliers x20."""
    d = workloads.prefill(seed=0, m=2048, n=16)
    q, s = fp8.quant_fp8_per_token(to_dev_bf16(d["x"]))
    wq, ws = orc.quant_per_token(d["x"])
    assert np.array_equal(host_bits(s), ws)
    assert np.array_equal(host_bits(q), wq)


def test_per_channel_weight_quant_gate_up(fp8, orc):
    """Per-output-channel weight quantisation of the merged gate_up weight
    [34816, 5120] (quant_fp8_per_token applied to the weight rows)."""
    d = workloads.gate_up_decode(seed=0)
    q, s = fp8.quant_fp8_per_token(to_dev_bf16(d["w"]))
    wq, ws = orc.quant_per_token(d["w"])
    assert np.array_equal(host_bits(s), ws)
    assert np.array_equal(host_bits(q), wq)


def test_per_token_special_values(fp8, orc):
    x = np.zeros((4, 32), np.uint16)
    x[0, :4] = [0x7F80, 0x3F80, 0xBF80, 0x0001]   # +inf in the row: scale inf
    x[1, :4] = [0x7FC0, 0x4000, 0xC100, 0x0000]   # NaN does not take part in the max
    x[2, :2] = [0x0001, 0x8002]                   # subnormal-only row
    x[3, :] = 0x8000                              # negative zeros
    q, s = fp8.quant_fp8_per_token(to_dev_bf16(x))
    wq, ws = orc.quant_per_token(x)
    assert np.array_equal(host_bits(s), ws)
    qh = host_bits(q)
    nan_in = ((x & 0x7F80) == 0x7F80) & ((x & 0x7F) != 0)
    inf_in = (x & 0x7FFF) == 0x7F80
    ok = ~(nan_in | inf_in)
    assert np.array_equal(qh[ok], wq[ok])
    assert np.all((qh[~ok] & 0x7F) == 0x7F)   # inf/inf and NaN/s are NaN


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32])
def test_rmsnorm_quant_decode_fused(fp8, orc, M):
    """Decode fused path producer: rows 0..M-1 of x [32, 5120], gamma =
    1 + N(0, 0.1), eps 1e-6, the static activation scale."""
    d = workloads.decode_fused(seed=0)
    x = d["x"][:M]
    buf = Guarded(M * 5120)
    out = buf.view(torch.float8_e4m3fn, (M, 5120))
    q = fp8.rmsnorm_quant_fp8(to_dev_bf16(x), to_dev_bf16(d["gamma"]), d["eps"], to_dev_f32(d["s_a"]), out=out)
    assert np.array_equal(host_bits(q), orc.rmsnorm_quant(x, d["gamma"], d["eps"], float(d["s_a"])))
    assert buf.intact()


@pytest.mark.parametrize("M,K,eps,s", [(32, 5120, 1e-6, 1 / 112), (5, 16, 1e-6, 1 / 56), (3, 17408, 1e-5, 0.02),
                                       (2, 65536, 0.0, 0.01), (4, 8192, 1e-6, 1 / 56), (300, 5120, 1e-6, 1 / 56),
                                       (1000, 5120, 1e-6, 1 / 56), (640, 8192, 1e-5, 0.02)])
def test_rmsnorm_quant_shapes(fp8, orc, M, K, eps, s):
    g = workloads.rng(40 + K)
    x = workloads.bf16_normal(g, (M, K))
    gamma = workloads.bf16_normal(g, (K,), mean=1.0, std=0.1)
    x[0] = 0          # all-zero row: eps keeps the root finite (eps == 0 gives inf * 0 = NaN codes)
    s = float(np.float32(s))
    q = host_bits(fp8.rmsnorm_quant_fp8(to_dev_bf16(x), to_dev_bf16(gamma), eps, to_dev_f32(s)))
    want = orc.rmsnorm_quant(x, gamma, eps, s)
    if eps == 0.0:
        assert np.all((q[0] & 0x7F) == 0x7F) and np.all((want[0] & 0x7F) == 0x7F)
        q, want = q[1:], want[1:]
    assert np.array_equal(q, want)


def test_rmsnorm_eps0_underflow_row(fp8, orc):
    """eps = 0 and rows whose mean square underflows binary32 (elements +-2^-126
    or 0, at two row lengths): r = inf, nonzero elements saturate to +-448
    and zero elements give a NaN code, as in the oracle (any NaN code for
    NaN)."""
    for K in (64, 5120):
        rows = np.full((2, K), 0x0080, np.uint16)
        rows[0, 3] = 0x0000
        rows[1, 5::7] = 0x8080
        gamma = np.full(K, 0x3FC0, np.uint16)
        q = host_bits(fp8.rmsnorm_quant_fp8(to_dev_bf16(rows), to_dev_bf16(gamma), 0.0, to_dev_f32(1 / 56)))
        want = orc.rmsnorm_quant(rows, gamma, 0.0, float(np.float32(1 / 56)))
        nan = (want & 0x7F) == 0x7F
        assert np.array_equal(q[~nan], want[~nan]) and np.all((q[nan] & 0x7F) == 0x7F)


def test_rmsnorm_fused_equals_unfused(fp8, orc):
    """Fused norm-quant == static quant of the bf16 norm output, byte for byte
    (the norm output comes from the oracle; the quant runs on the GPU)."""
    d = workloads.decode_fused(seed=1)
    h = orc.rmsnorm_bf16(d["x"], d["gamma"], d["eps"])
    s = to_dev_f32(d["s_a"])
    unfused = host_bits(fp8.quant_fp8_static(to_dev_bf16(h), s))
    fused = host_bits(fp8.rmsnorm_quant_fp8(to_dev_bf16(d["x"]), to_dev_bf16(d["gamma"]), d["eps"], s))
    assert np.array_equal(fused, unfused)


def test_per_token_flattened_equals_static_amax(fp8):
    """Per-token quant of a tensor viewed as one row == static quant with that
    row's scale (the tiny workload's per-tensor quantisation)."""
    d = workloads.tiny_gemm(seed=0)
    x = to_dev_bf16(d["x"])
    q1, s1 = fp8.quant_fp8_per_token(x.view(1, -1))
    q2 = fp8.quant_fp8_static(x, s1)
    assert np.array_equal(host_bits(q1).reshape(4, 256), host_bits(q2))


def test_rmsnorm_exact_sum_edge_rows(fp8, orc):
    """Rows that exercise the exact sum of squares: a binary32 tie broken by a
    term 80 binades down (below the 40-binade window: the sticky bit), terms
    spanning more than 120 bits, subnormal inputs, NaN / Inf, constant rows."""
    K = 64
    rows = np.zeros((10, K), np.uint16)
    rows[0, :2] = [0x3F80, 0x3980]                    # 1 + 2^-24: a tie
    rows[1, :3] = [0x3F80, 0x3980, 0x2B80]            # ... broken upwards by 2^-80
    g = workloads.rng(44)
    rows[2] = workloads.bf16_normal(g, (K,))
    rows[2, ::3] = 0x1F80                             # 2^-64 next to O(1) values
    rows[3, :5] = [0x0001, 0x0003, 0x8005, 0x007F, 0x0080]   # subnormals and the smallest normal
    rows[4, :2] = [0x7FC0, 0x3F80]                    # NaN
    rows[5, :2] = [0x7F80, 0x3F80]                    # +Inf
    rows[6, :3] = [0x7F80, 0x7FC0, 0x3F80]            # Inf and NaN: NaN
    rows[7] = 0x4040                                  # constant 3.0
    rows[8] = workloads.bf16_normal(g, (K,), std=1e6)
    rows[9] = 0x5F00                                  # 2^63: squares overflow binary32 -> Inf
    gamma = workloads.bf16_normal(g, (K,), mean=1.0, std=0.1)
    for eps in (1e-6, 0.0):
        q = host_bits(fp8.rmsnorm_quant_fp8(to_dev_bf16(rows), to_dev_bf16(gamma), eps, to_dev_f32(1 / 56)))
        want = orc.rmsnorm_quant(rows, gamma, eps, float(np.float32(1 / 56)))
        nan_w = (want & 0x7F) == 0x7F
        assert np.array_equal(q[~nan_w], want[~nan_w]), eps
        assert np.all((q[nan_w] & 0x7F) == 0x7F), eps


def test_rmsnorm_warp_windows(fp8, orc):
    """Rows of 5120 (20 warps of one vector per thread) whose warps see very
    different largest binades, so that aligning the warps' window sums to the
    row's window shifts bits out: large values in one warp's elements only,
    tiny ones elsewhere (squares below the row's window, some of them exact
    multiples of its unit), an Inf or a NaN in a single warp, subnormals around
    one normal value."""
    K = 5120
    g = workloads.rng(77)
    rows = np.zeros((8, K), np.uint16)
    big = workloads.bf16_normal(g, (K,))
    tiny = workloads.bf16_normal(g, (K,), std=2.0 ** -50)
    rows[0] = tiny
    rows[0, :256] = big[:256]                          # warp 0 large, the rest 2^-50
    rows[1] = tiny
    rows[1, 4000:4256] = big[4000:4256]                # a late warp large
    rows[2] = 0x2000                                   # 2^-63: squares exact in the row's unit
    rows[2, 300] = 0x4000                              # one 2.0
    rows[3] = big
    rows[3, 2000] = 0x7F80                             # Inf in one warp
    rows[4] = big
    rows[4, 5119] = 0x7FC1                             # NaN in the last warp
    rows[5] = g.integers(1, 128, K).astype(np.uint16)  # subnormals ...
    rows[5, 4321] = 0x0080                             # ... and the smallest normal
    rows[6] = tiny
    rows[6, ::640] = 0x4B00                            # a few 2^23 values, every other warp
    rows[7] = big
    rows[7, 1:K:7] = 0x0001                            # a subnormal every 7th element
    gamma = workloads.bf16_normal(g, (K,), mean=1.0, std=0.1)
    for eps in (1e-6, 0.0):
        s = float(np.float32(1 / 56))
        q = host_bits(fp8.rmsnorm_quant_fp8(to_dev_bf16(rows), to_dev_bf16(gamma), eps, to_dev_f32(s)))
        want = orc.rmsnorm_quant(rows, gamma, eps, s)
        nan_w = (want & 0x7F) == 0x7F
        assert np.array_equal(q[~nan_w], want[~nan_w]), eps
        assert np.all((q[nan_w] & 0x7F) == 0x7F), eps


@pytest.mark.parametrize("K", [64, 5120])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_rmsnorm_carry_rows(fp8, orc, K, seed):
    """Rows whose squares below the 40-binade window carry into the rounding
    of the windowed sum (constructed: guard bit 0, a run of ones below it):
    the windowed rule alone rounds the sum of squares one ulp low and the
    probe's E4M3 code one step high; the kernel must detect the case and sum
    the row exactly.  Between two ordinary rows; also through the residual
    path, the row arriving as the residual (x = 0) so that the exact sum must
    read the summed row."""
    import norm_cases
    d = norm_cases.carry_row(K=K, seed=seed)
    assert d["ss_exact"] != d["ss_window"]
    g = workloads.rng(70 + seed)
    rows = workloads.bf16_normal(g, (4, K))
    rows[1] = d["row"]
    # the same elements scattered over the row (other warps, other windows);
    # the probe stays where its gamma is
    perm = np.concatenate([[d["probe"]], g.permutation(np.delete(np.arange(K), d["probe"]))])
    rows[3] = 0
    rows[3][perm] = d["row"][np.concatenate([[d["probe"]], np.delete(np.arange(K), d["probe"])])]
    s = float(np.float32(d["s"]))
    want = orc.rmsnorm_quant(rows, d["gamma"], d["eps"], s)
    q = host_bits(fp8.rmsnorm_quant_fp8(to_dev_bf16(rows), to_dev_bf16(d["gamma"]), d["eps"], to_dev_f32(s)))
    assert np.array_equal(q, want)
    zeros = np.zeros_like(rows)
    want_q, want_h = orc.add_rmsnorm_quant(zeros, rows, d["gamma"], d["eps"], s)
    assert np.array_equal(want_q, want)
    rd = to_dev_bf16(rows)
    q2 = host_bits(fp8.add_rmsnorm_quant_fp8(to_dev_bf16(zeros), rd, to_dev_bf16(d["gamma"]), d["eps"],
                                             to_dev_f32(s)))
    assert np.array_equal(q2, want) and np.array_equal(host_bits(rd), want_h)


@pytest.mark.parametrize("M,K", [(1, 5120), (8, 5120), (32, 5120), (3, 17408), (1000, 5120), (5, 16)])
def test_add_rmsnorm_quant(fp8, orc, M, K):
    """Residual add -> RMSNorm -> static quant: the E4M3 bytes and the updated
    residual (in place) bit-exact against the oracle, including residual
    values that overflow the sum and signed zeros."""
    g = workloads.rng(80 + M + K)
    x = workloads.bf16_normal(g, (M, K))
    r = workloads.bf16_normal(g, (M, K), std=4.0)
    gamma = workloads.bf16_normal(g, (K,), mean=1.0, std=0.1)
    r[0, :4] = [0x8000, 0x0000, 0x7F7F, 0xFF7F]
    x[0, :4] = [0x8000, 0x8000, 0x7F7F, 0x3F80]
    s = float(np.float32(1 / 56))
    want_q, want_h = orc.add_rmsnorm_quant(x, r, gamma, 1e-6, s)
    rd = to_dev_bf16(r)
    q = fp8.add_rmsnorm_quant_fp8(to_dev_bf16(x), rd, to_dev_bf16(gamma), 1e-6, to_dev_f32(s))
    assert np.array_equal(host_bits(rd), want_h)
    qh = host_bits(q)
    nan_w = (want_q & 0x7F) == 0x7F
    assert np.array_equal(qh[~nan_w], want_q[~nan_w])
    assert np.all((qh[nan_w] & 0x7F) == 0x7F)


def test_add_rmsnorm_equals_add_then_norm(fp8, orc):
    """Fused == the residual sum materialised, then rmsnorm_quant_fp8 on it."""
    d = workloads.decode_fused(seed=9)
    g = workloads.rng(90)
    r = workloads.bf16_normal(g, d["x"].shape, std=0.5)
    s = to_dev_f32(d["s_a"])
    rd = to_dev_bf16(r)
    q = host_bits(fp8.add_rmsnorm_quant_fp8(to_dev_bf16(d["x"]), rd, to_dev_bf16(d["gamma"]), d["eps"], s))
    h = orc.residual_add_bf16(d["x"], r)
    q2 = host_bits(fp8.rmsnorm_quant_fp8(to_dev_bf16(h), to_dev_bf16(d["gamma"]), d["eps"], s))
    assert np.array_equal(q, q2)
    assert np.array_equal(host_bits(rd), h)


@pytest.mark.parametrize("M,I", [(1, 17408), (8, 17408), (3, 16), (1000, 1024), (5, 2064), (2, 65536)])
def test_silu_mul_quant_per_token(fp8, orc, M, I):
    """SiLU(gate) * up -> per-token quant, bit-exact (codes and scales) against
    the oracle on MLP-like rows ([gate | up], N(0,1) with 1% outliers x20),
    including all-zero rows and large negative gates."""
    g = workloads.rng(100 + M + I)
    gu = workloads.bf16_normal_with_outliers(g, (M, 2 * I))
    if M > 2:
        gu[2] = 0
    gu[0, :8] = [0xC2C8, 0x42C8, 0xFF80, 0x7F80, 0x0001, 0x8001, 0x3F80, 0xBF80]   # -100, 100, -inf, inf, ...
    q, s = fp8.silu_mul_quant_per_token(to_dev_bf16(gu))
    wq, ws = orc.silu_mul_quant_per_token(gu)
    sh, qh = host_bits(s), host_bits(q)
    ok_rows = np.isfinite(ws)
    assert np.array_equal(sh[ok_rows], ws[ok_rows])
    assert np.all(np.isnan(sh[~ok_rows]) | np.isinf(sh[~ok_rows]))
    nan_w = (wq & 0x7F) == 0x7F
    assert np.array_equal(qh[ok_rows][~nan_w[ok_rows]], wq[ok_rows][~nan_w[ok_rows]])


def test_silu_mul_quant_equals_unfused(fp8, orc):
    """Fused == the bf16 intermediate materialised (oracle), then the GPU's
    per-token quantiser on it."""
    g = workloads.rng(101)
    gu = workloads.bf16_normal(g, (16, 2 * 4096), std=2.0)
    q, s = fp8.silu_mul_quant_per_token(to_dev_bf16(gu))
    a = orc.silu_mul_bf16(gu)
    q2, s2 = fp8.quant_fp8_per_token(to_dev_bf16(a))
    assert np.array_equal(host_bits(q), host_bits(q2)) and np.array_equal(host_bits(s), host_bits(s2))


def test_requant_merge_qkv_shards(fp8, orc):
    """Three shards (q 8192, k 1024, v 1024 rows of K 512) with different
    per-tensor scales merged at the largest: codes bit-exact against the
    oracle (NaN codes stay NaN codes), the scale is the maximum."""
    g = workloads.rng(110)
    K = 512
    rows = (workloads.Q_WIDTH, workloads.KV_WIDTH, workloads.KV_WIDTH)
    shards = [workloads.e4m3_codes(g, (r, K)) for r in rows]
    shards[1][0, :4] = [0x7F, 0xFF, 0x7E, 0xFE]
    scales = [np.float32(2.1e-3), np.float32(3.3e-3), np.float32(1.7e-3)]
    merged, s = fp8.requant_merge([to_dev_e4m3(w) for w in shards], [to_dev_f32(x) for x in scales])
    smax = max(scales)
    assert host_bits(s)[0] == smax
    want = np.concatenate([orc.requant(w, float(x), float(smax)) for w, x in zip(shards, scales)])
    got = host_bits(merged)
    nan_w = (want & 0x7F) == 0x7F
    assert np.array_equal(got[~nan_w], want[~nan_w])
    assert np.all((got[nan_w] & 0x7F) == 0x7F)
    # the shard at the largest scale is unchanged
    assert np.array_equal(got[rows[0]:rows[0] + rows[1]][~nan_w[rows[0]:rows[0] + rows[1]]],
                          shards[1][~nan_w[rows[0]:rows[0] + rows[1]]])
