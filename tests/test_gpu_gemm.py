"""GPU parity of the FP8 W8A8 scaled GEMM against the CPU oracle, on the
workload shapes and on ragged random shapes, plus the invariants the method
guarantees (determinism, graph == eager, merged == split, batch invariance)."""
import numpy as np
import pytest
import torch

import workloads
from helpers import Guarded, check_gemm, check_gemm_tc, host_bits, scale_product, to_dev_bf16, to_dev_e4m3, to_dev_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    import fp8_w8a8_scaled_gb300 as f
    f.clear_device_error()
    yield f
    assert f.get_device_error() == 0


def run_mm(fp8, A, B, sa, sb, gran):
    """A, B: device E4M3 tensors; returns the bf16 output bits, checking the
    guard bands around the output."""
    M, N = A.shape[0], B.shape[0]
    buf = Guarded(M * N * 2)
    out = buf.view(torch.bfloat16, (M, N))
    fp8.fp8_scaled_mm(A, B, sa, sb, gran, out=out)
    torch.cuda.synchronize()
    assert buf.intact(), "write outside the output buffer"
    return host_bits(out)


def full_check(orc, A_codes, B_codes, sa, sb, gran, y_bits, what, tc_bound=False):
    """Every output against the oracle.  With tc_bound (stress inputs:
    uniformly random codes, or outlier-free data on the large-M kernel's long
    accumulation groups) the binary32 accumulation bound is added to the
    acceptance bound; the ratio to the acceptance bound alone is still
    reported."""
    y64, _ = orc.scaled_mm(A_codes, B_codes, sa, sb, gran)
    M, N = y64.shape
    rows = np.arange(M)[:, None]
    cols = np.arange(N)[None, :]
    sab = scale_product(sa, sb, gran, rows, cols)
    K = A_codes.shape[1]
    if tc_bound:
        abs_sum = orc.gemm_acc_f64(np.asarray(A_codes) & 0x7F, np.asarray(B_codes) & 0x7F)
        r_acc, r_tot = check_gemm_tc(y_bits, y64, sab, K, abs_sum, what)
        print(f"{what}: max err/bound {r_acc:.4f} (with accumulation bound {r_tot:.4f})")
        return r_acc, y64.size
    return check_gemm(y_bits, y64, sab, K, what)


# ----------------------------------------------------------------------------- workloads

def test_tiny_gemm_per_tensor(fp8, orc):
    """M=4, K=256, N=512; A and B quantised per tensor with scale amax/448."""
    d = workloads.tiny_gemm(seed=0)
    qa, sa = fp8.quant_fp8_per_token(to_dev_bf16(d["x"]).view(1, -1))
    qb, sb = fp8.quant_fp8_per_token(to_dev_bf16(d["w"]).view(1, -1))
    wa, wsa = orc.quant_per_token(d["x"].reshape(1, -1))
    wb, wsb = orc.quant_per_token(d["w"].reshape(1, -1))
    assert np.array_equal(host_bits(qa).ravel(), wa.ravel()) and np.array_equal(host_bits(sa), wsa)
    assert np.array_equal(host_bits(qb).ravel(), wb.ravel()) and np.array_equal(host_bits(sb), wsb)
    A = qa.view(4, 256)
    B = qb.view(512, 256)
    y = run_mm(fp8, A, B, sa, sb, 0)
    full_check(orc, wa.reshape(4, 256), wb.reshape(512, 256), wsa, wsb, 0, y, "tiny")


@pytest.fixture(scope="module")
def decode_fused_case(orc):
    d = workloads.decode_fused(seed=0)
    A_all = orc.rmsnorm_quant(d["x"], d["gamma"], d["eps"], float(d["s_a"]))
    y64, _ = orc.scaled_mm(A_all, d["B"], d["s_a"], d["sb"], 1)
    return d, A_all, y64


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32])
def test_decode_fused_qkv(fp8, decode_fused_case, M):
    """RMSNorm -> static quant -> merged QKV GEMM (N=10240, K=5120), per-channel
    weight scales; rows 0..M-1 of one [32, 5120] batch."""
    d, A_all, y64 = decode_fused_case
    s_a = to_dev_f32(d["s_a"])
    A = fp8.rmsnorm_quant_fp8(to_dev_bf16(d["x"][:M]), to_dev_bf16(d["gamma"]), d["eps"], s_a)
    assert np.array_equal(host_bits(A), A_all[:M])
    want = fp8.KERNEL_DECODE_SPLITK if M <= 32 else fp8.KERNEL_PREFILL
    assert fp8.describe_dispatch(M, 10240, 5120, 1) == want
    y = run_mm(fp8, A, to_dev_e4m3(d["B"]), s_a, to_dev_f32(d["sb"]), 1)
    sab = scale_product(d["s_a"], d["sb"], 1, np.arange(M)[:, None], np.arange(10240)[None, :])
    worst, _ = check_gemm(y, y64[:M], sab, 5120, f"decode fused M={M}")
    print(f"M={M} max err/bound {worst:.4f}")


@pytest.fixture(scope="module")
def gate_up_case(fp8, orc):
    d = workloads.gate_up_decode(seed=0)
    qb, sb = fp8.quant_fp8_per_token(to_dev_bf16(d["w"]))
    wb, wsb = orc.quant_per_token(d["w"])
    assert np.array_equal(host_bits(qb), wb) and np.array_equal(host_bits(sb), wsb)
    s_a = float(d["s_a"])
    qa = fp8.quant_fp8_static(to_dev_bf16(d["x"]), to_dev_f32(s_a))
    wa = orc.quant_static(d["x"], s_a)
    assert np.array_equal(host_bits(qa), wa)
    y64, _ = orc.scaled_mm(wa, wb, [s_a], wsb, 1)
    return d, qa, qb, sb, wsb, y64


@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_gate_up_decode(fp8, gate_up_case, M):
    """Merged gate_up decode GEMM: N=34816, K=5120, per-channel weight scales,
    per-tensor static activation scale."""
    d, qa, qb, sb, wsb, y64 = gate_up_case
    y = run_mm(fp8, qa[:M].contiguous(), qb, to_dev_f32(d["s_a"]), sb, 1)
    sab = scale_product([d["s_a"]], wsb, 1, np.arange(M)[:, None], np.arange(34816)[None, :])
    worst, _ = check_gemm(y, y64[:M], sab, 5120, f"gate_up M={M}")
    print(f"M={M} max err/bound {worst:.4f}")


@pytest.mark.parametrize("M,N", [(2048, 10240)])
def test_prefill_chunk_qkv_full(fp8, orc, M, N):
    """Prefill chunk: per-token activation quant (1% outliers x20), per-channel
    weights, M=2048, N=10240, K=5120; every output against the oracle."""
    d = workloads.prefill(seed=0, m=M, n=N)
    qa, sa = fp8.quant_fp8_per_token(to_dev_bf16(d["x"]))
    qb, sb = fp8.quant_fp8_per_token(to_dev_bf16(d["w"]))
    wa, wsa = orc.quant_per_token(d["x"])
    wb, wsb = orc.quant_per_token(d["w"])
    assert np.array_equal(host_bits(qa), wa) and np.array_equal(host_bits(sa), wsa)
    assert np.array_equal(host_bits(qb), wb) and np.array_equal(host_bits(sb), wsb)
    assert fp8.describe_dispatch(M, N, 5120, 2) == fp8.KERNEL_PREFILL
    y = run_mm(fp8, qa, qb, sa, sb, 2)
    worst, _ = full_check(orc, wa, wb, wsa, wsb, 2, y, f"prefill {M}x{N}")
    print(f"prefill {M}x{N} max err/bound {worst:.4f}")


def test_down_projection_long_k(fp8, orc):
    """The decode step's down projection: N=5120, K=17408, M=8."""
    qa, qb, sa, sb, wa, wb, wsa, wsb = quantised_operands(fp8, orc, 8, 5120, 17408, 2, 50)
    y = run_mm(fp8, qa, qb, sa, sb, 2)
    worst, _ = full_check(orc, wa, wb, wsa, wsb, 2, y, "down 8x5120x17408")
    print(f"down max err/bound {worst:.4f}")


# ----------------------------------------------------------------------------- decode modes

# (M, N, K, S): the decode kernel's mode for the shape on a 152-SM GB300 --
# clusters of S CTAs per 128-channel tile (every S from 1 to 8, rows split
# unevenly among the S CTAs for S = 3, 5, 6, 7; a ragged last tile; K ranges
# split unevenly), or 0 for the persistent stream-K grid.
DECODE_MODES = [(1, 34816, 1040, 1), (16, 10240, 256, 1), (16, 12800, 400, 2), (3, 13312, 2064, 2), (16, 10232, 5136, 3),
                (7, 8192, 1552, 3), (2, 7168, 4096, 4), (16, 6144, 1040, 5), (5, 5120, 8192, 6),
                (4, 4096, 2064, 7), (11, 3840, 1552, 8),
                (1, 128, 5120, 0), (16, 2048, 5120, 0), (9, 1032, 17408, 0),
                # the 32-token tile (17 <= M <= 32)
                (32, 10240, 5120, 3), (24, 34816, 1040, 1), (17, 5120, 8192, 6), (32, 2048, 5120, 0),
                (20, 1032, 4096, 0)]


@pytest.mark.parametrize("M,N,K,S", DECODE_MODES)
def test_decode_modes(fp8, orc, M, N, K, S):
    """Every output of both decode modes against the oracle, per-token x
    per-channel scales (exact k-block sums).  Uniformly random codes are
    stress inputs: their 128-wide k-block sums are large next to the
    acceptance bound's absolute term, and the tensor core's binary32
    accumulation inside a k-block is allowed its own bound (as on the tile
    kernel)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert fp8.decode_split(M, N, K, sms, granularity=2) == S
    assert fp8.decode_exact(M, N, K, granularity=2) == 1
    c = workloads.random_gemm(7000 + M + N + K, M, N, K, 2)
    y = run_mm(fp8, to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"]), to_dev_f32(c["sa"]), to_dev_f32(c["sb"]), 2)
    worst, _ = full_check(orc, c["A"], c["B"], c["sa"], c["sb"], 2, y, f"{M}x{N}x{K} split {S}", tc_bound=True)
    print(f"{M}x{N}x{K} split {fp8.decode_split(M, N, K, granularity=2)}: max err/bound {worst:.4f}")


# ----------------------------------------------------------------------------- ragged shapes

# Uniformly random E4M3 codes: every code value, with a heavier magnitude tail
# than quantised activations/weights; used where K is short.
SHAPES_CODES = [(1, 8, 16), (3, 136, 48), (17, 264, 400), (33, 1000, 272), (65, 520, 1040), (127, 392, 784),
                (129, 256, 512), (16, 128, 128)]


@pytest.mark.parametrize("M,N,K", SHAPES_CODES)
@pytest.mark.parametrize("gran", [0, 1, 2, 3])
def test_random_codes(fp8, orc, M, N, K, gran):
    c = workloads.random_gemm(1000 + M * 7 + N * 3 + K + gran, M, N, K, gran)
    y = run_mm(fp8, to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"]), to_dev_f32(c["sa"]), to_dev_f32(c["sb"]), gran)
    full_check(orc, c["A"], c["B"], c["sa"], c["sb"], gran, y, f"{M}x{N}x{K} gran {gran}", tc_bound=True)


def quantised_operands(fp8, orc, M, N, K, gran, seed):
    """Workload-like operands: N(0,1) activations and N(0,0.02) weights in bf16,
    quantised on the GPU (per token / per tensor for A, per channel / per
    tensor for B as the granularity asks) and checked byte-exact against the
    oracle's quantisers first."""
    g = workloads.rng(seed)
    x = workloads.bf16_normal(g, (M, K))
    w = workloads.bf16_normal(g, (N, K), std=0.02)
    tok = gran in (2, 3)
    ch = gran in (1, 2)
    qa, sa = fp8.quant_fp8_per_token(to_dev_bf16(x) if tok else to_dev_bf16(x).view(1, -1))
    qb, sb = fp8.quant_fp8_per_token(to_dev_bf16(w) if ch else to_dev_bf16(w).view(1, -1))
    wa, wsa = orc.quant_per_token(x if tok else x.reshape(1, -1))
    wb, wsb = orc.quant_per_token(w if ch else w.reshape(1, -1))
    assert np.array_equal(host_bits(qa).ravel(), wa.ravel()) and np.array_equal(host_bits(sa), wsa)
    assert np.array_equal(host_bits(qb).ravel(), wb.ravel()) and np.array_equal(host_bits(sb), wsb)
    return qa.view(M, K), qb.view(N, K), sa, sb, wa.reshape(M, K), wb.reshape(N, K), wsa, wsb


SHAPES_QUANT = [(64, 1032, 2064), (200, 8, 4096), (31, 2056, 3088), (5, 264, 8208), (48, 640, 17408)]


@pytest.mark.parametrize("M,N,K", SHAPES_QUANT)
@pytest.mark.parametrize("gran", [0, 1, 2, 3])
def test_quantised_operands_long_k(fp8, orc, M, N, K, gran):
    qa, qb, sa, sb, wa, wb, wsa, wsb = quantised_operands(fp8, orc, M, N, K, gran, 3000 + M + N + K + gran)
    y = run_mm(fp8, qa, qb, sa, sb, gran)
    full_check(orc, wa, wb, wsa, wsb, gran, y, f"{M}x{N}x{K} gran {gran}")


def test_extreme_codes(fp8, orc):
    """All-448 operands (largest products), all-ones, and a mix with zeros."""
    M, N, K = 5, 256, 1024
    A = np.full((M, K), 0x7E, np.uint8)
    B = np.full((N, K), 0x7E, np.uint8)
    B[1::2] = 0xFE
    A[1] = 0x38
    A[2] = 0x00
    y = run_mm(fp8, to_dev_e4m3(A), to_dev_e4m3(B), to_dev_f32([1e-3]), to_dev_f32([2e-3]), 0)
    full_check(orc, A, B, [1e-3], [2e-3], 0, y, "extreme")


def test_nan_code_propagates(fp8):
    M, N, K = 2, 16, 256
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((N, K), 0x38, np.uint8)
    B[3, 100] = 0x7F
    y = run_mm(fp8, to_dev_e4m3(A), to_dev_e4m3(B), to_dev_f32([1.0]), to_dev_f32([1.0]), 0)
    v = (y.astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.isnan(v[:, 3]))
    assert np.all(v[:, [0, 1, 2, 4]] == 256.0)


# ----------------------------------------------------------------------------- invariants

def test_rerun_is_bitwise_identical(fp8):
    for (M, N, K) in ((32, 10240, 5120), (3, 1000, 272)):
        c = workloads.random_gemm(60, M, N, K, 2)
        args = (to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"]), to_dev_f32(c["sa"]), to_dev_f32(c["sb"]), 2)
        y1 = run_mm(fp8, *args)
        y2 = run_mm(fp8, *args)
        assert np.array_equal(y1, y2)


def test_graph_replay_equals_eager(fp8):
    M, N, K = 8, 10240, 5120
    c = workloads.random_gemm(61, M, N, K, 1)
    A, B = to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"])
    sa, sb = to_dev_f32(c["sa"]), to_dev_f32(c["sb"])
    eager = run_mm(fp8, A, B, sa, sb, 1)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fp8.fp8_scaled_mm(A, B, sa, sb, 1, out=out)   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fp8.fp8_scaled_mm(A, B, sa, sb, 1, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out), eager)


def test_merged_equals_split(fp8, orc):
    """QKV as one GEMM over [Wq; Wk; Wv] against three GEMMs: bitwise equal
    (the decode kernel sums each tile's k-block partials exactly, so how the
    K ranges are divided among CTAs -- different for the three shapes -- does
    not change a bit), and both within the bound of the oracle."""
    M, K = 8, 5120
    d = workloads.decode_fused(seed=2)
    B = d["B"]
    A = orc.rmsnorm_quant(d["x"][:M], d["gamma"], d["eps"], float(d["s_a"]))
    sa = to_dev_f32(d["s_a"])
    Ad = to_dev_e4m3(A)
    merged = run_mm(fp8, Ad, to_dev_e4m3(B), sa, to_dev_f32(d["sb"]), 1)
    parts, lo = [], 0
    for w in (workloads.Q_WIDTH, workloads.KV_WIDTH, workloads.KV_WIDTH):
        parts.append(run_mm(fp8, Ad, to_dev_e4m3(B[lo:lo + w]), sa, to_dev_f32(d["sb"][lo:lo + w]), 1))
        lo += w
    split = np.concatenate(parts, axis=1)
    y64, _ = orc.scaled_mm(A, B, d["s_a"], d["sb"], 1)
    sab = scale_product(d["s_a"], d["sb"], 1, np.arange(M)[:, None], np.arange(10240)[None, :])
    assert fp8.decode_split(M, 10240, K) != fp8.decode_split(M, workloads.KV_WIDTH, K)
    assert np.array_equal(merged, split)
    check_gemm(merged, y64, sab, K, "merged")


def test_batch_rows_independent(fp8):
    """Row m of an M=16 call against the same row alone (M=1): both use the
    16-token tile and the same division of the K ranges, so bitwise."""
    N, K = 10240, 5120
    c = workloads.random_gemm(62, 16, N, K, 1)
    A = to_dev_e4m3(c["A"])
    B = to_dev_e4m3(c["B"])
    sa, sb = to_dev_f32(c["sa"]), to_dev_f32(c["sb"])
    full = run_mm(fp8, A, B, sa, sb, 1)
    for m in (0, 7, 15):
        one = run_mm(fp8, A[m:m + 1].contiguous(), B, sa, sb, 1)
        assert fp8.decode_ctas(1, N, K) == fp8.decode_ctas(16, N, K)
        assert np.array_equal(one[0], full[m])


def test_batch_rows_independent_across_token_tiles(fp8):
    """Row m of an M=32 call (32-token tile) against the same row alone (M=1,
    16-token tile): the k-block partials come from MMAs of different widths
    but the same operands, and the exact sum makes the division of K
    irrelevant, so the decode kernel is batch-invariant over M <= 32."""
    N, K = 10240, 5120
    c = workloads.random_gemm(64, 32, N, K, 2)
    A = to_dev_e4m3(c["A"])
    B = to_dev_e4m3(c["B"])
    sa, sb = to_dev_f32(c["sa"]), to_dev_f32(c["sb"])
    full = run_mm(fp8, A, B, sa, sb, 2)
    for m in (0, 16, 31):
        one = run_mm(fp8, A[m:m + 1].contiguous(), B, sa[m:m + 1].contiguous(), sb, 2)
        assert np.array_equal(one[0], full[m]), m


def test_stream_k_on_two_streams(fp8):
    """Stream-K launches (few 128-row tiles with a long K: the mode that uses
    scratch) issued back to back on two streams at once: each stream has its
    own scratch, so every result equals the serial one bit for bit."""
    cases = []
    for i, (M, N, K) in enumerate([(16, 2048, 5120), (9, 1032, 17408)]):
        assert fp8.decode_split(M, N, K, granularity=2) == 0
        c = workloads.random_gemm(65 + i, M, N, K, 2)
        args = (to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"]), to_dev_f32(c["sa"]), to_dev_f32(c["sb"]), 2)
        cases.append((args, run_mm(fp8, *args)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = [[], []]
    for _ in range(8):
        for j, s in enumerate(streams):
            with torch.cuda.stream(s):
                outs[j].append(fp8.fp8_scaled_mm(*cases[j][0]))
    torch.cuda.synchronize()
    for j in range(2):
        for o in outs[j]:
            assert np.array_equal(host_bits(o), cases[j][1]), j


def test_stream_k_first_call_inside_graph_capture(fp8):
    """A stream whose first stream-K call is made while it is captured into a
    CUDA graph: the scratch is allocated during the capture, the graph's
    replays and a later eager call on the same stream all give the serial
    result bit for bit."""
    M, N, K = 16, 2048, 5120
    assert fp8.decode_split(M, N, K, granularity=2) == 0
    c = workloads.random_gemm(67, M, N, K, 2)
    args = (to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"]), to_dev_f32(c["sa"]), to_dev_f32(c["sb"]), 2)
    ref = run_mm(fp8, *args)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fp8.fp8_scaled_mm(*args, out=out)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(out), ref)
    with torch.cuda.stream(s):
        eager = fp8.fp8_scaled_mm(*args)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(eager), ref)
    assert fp8.get_device_error() == 0


def test_m_zero_is_noop(fp8):
    A = torch.empty((0, 64), dtype=torch.float8_e4m3fn, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.float8_e4m3fn, device="cuda")
    out = fp8.fp8_scaled_mm(A, B, to_dev_f32([1.0]), to_dev_f32([1.0]), 0)
    assert out.shape == (0, 64)


def test_launch_flags_do_not_change_results(fp8):
    """Weights-static prefetch and launches without programmatic dependent
    launch give the same bytes as the default."""
    M, N, K = 16, 10240, 5120
    c = workloads.random_gemm(63, M, N, K, 1)
    A, B = to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"])
    sa, sb = to_dev_f32(c["sa"]), to_dev_f32(c["sb"])
    ref = run_mm(fp8, A, B, sa, sb, 1)
    for flags in (fp8.FLAG_WEIGHTS_STATIC, fp8.FLAG_NO_PDL, fp8.FLAG_WEIGHTS_STATIC | fp8.FLAG_NO_PDL):
        out = fp8.fp8_scaled_mm(A, B, sa, sb, 1, flags=flags)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(out), ref), flags


def test_chained_producer_consumer_with_pdl(fp8, orc):
    """A per-channel weight quantisation immediately followed by the GEMM that
    reads it (the default launch must wait for the producer)."""
    d = workloads.gate_up_decode(seed=3, rows=8, n=2048, k=1024)
    w = to_dev_bf16(d["w"])
    x = to_dev_bf16(d["x"])
    s_a = to_dev_f32(d["s_a"])
    for _ in range(3):
        qb, sb = fp8.quant_fp8_per_token(w)
        qa = fp8.quant_fp8_static(x, s_a)
        y = fp8.fp8_scaled_mm(qa, qb, s_a, sb, 1)
    torch.cuda.synchronize()
    wb, wsb = orc.quant_per_token(d["w"])
    wa = orc.quant_static(d["x"], float(d["s_a"]))
    y64, _ = orc.scaled_mm(wa, wb, [d["s_a"]], wsb, 1)
    sab = scale_product([d["s_a"]], wsb, 1, np.arange(8)[:, None], np.arange(2048)[None, :])
    check_gemm(host_bits(y), y64, sab, 1024, "chained")
