"""Seeded random-shape sweeps through every dispatch region of both GEMMs,
every output against the CPU oracle: the W8A8 scaled GEMM (decode kernel in
cluster and stream-K modes, the tile kernel on single CTAs and on CTA pairs,
all five granularities) and the weight-only GEMM (decode and tile kernels).
Shapes are drawn from a fixed generator: M over the decode range, the
single-CTA tile range and the paired range, N a multiple of 8, K a multiple
of 16, both ragged against the 128-wide tiles and k-blocks.  Operands are
uniformly random E4M3 codes, so the binary32 accumulation bound is added to
the acceptance bound (as for every random-code test)."""
import numpy as np
import pytest
import torch

import workloads
from helpers import to_dev_bf16, to_dev_e4m3, to_dev_f32
from test_gpu_blockwise import block_check, dev_scales, run_block_mm
from test_gpu_gemm import full_check, run_mm
from test_gpu_w8a16 import run_w16, w16_bound

pytestmark = pytest.mark.gpu

GRAN_BLOCK = 4
MAX_MACS = 4e8  # keeps each oracle call to about a second


def _shape(g, m_lo, m_hi):
    while True:
        M = int(g.integers(m_lo, m_hi + 1))
        N = 8 * int(g.integers(1, 513))
        K = 16 * int(g.integers(1, 261))
        if M * N * K <= MAX_MACS:
            return M, N, K


@pytest.fixture(scope="module")
def fp8():
    import fp8_w8a8_scaled_gb300 as f
    f.clear_device_error()
    yield f
    assert f.get_device_error() == 0


# (seed, M range): decode, single-CTA tile, CTA-pair tile
SCALED_CASES = [(s, (1, 32)) for s in range(6)] + [(s, (33, 128)) for s in range(6, 10)] + \
               [(s, (129, 700)) for s in range(10, 16)]


@pytest.mark.parametrize("seed,m_range", SCALED_CASES)
def test_scaled_mm_random_shape(fp8, orc, seed, m_range):
    g = np.random.default_rng(9000 + seed)
    M, N, K = _shape(g, *m_range)
    gran = int(g.integers(0, 5))
    c = workloads.random_gemm(9100 + seed, M, N, K, gran)
    A, B = to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"])
    what = f"sweep {M}x{N}x{K} gran {gran} (dispatch {fp8.describe_dispatch(M, N, K, gran)})"
    if gran == GRAN_BLOCK:
        y = run_block_mm(fp8, A, B, dev_scales(c["sa"]), dev_scales(c["sb"]))
        worst = block_check(orc, c["A"], c["B"], c["sa"], c["sb"], y, what)
        print(f"{what}: max err/bound {worst:.4f}")
    else:
        y = run_mm(fp8, A, B, to_dev_f32(c["sa"]), to_dev_f32(c["sb"]), gran)
        full_check(orc, c["A"], c["B"], c["sa"], c["sb"], gran, y, what, tc_bound=True)
    assert fp8.get_device_error() == 0


W16_CASES = [(s, (1, 32)) for s in range(4)] + [(s, (33, 600)) for s in range(4, 10)]


@pytest.mark.parametrize("seed,m_range", W16_CASES)
def test_w8a16_random_shape(fp8, orc, seed, m_range):
    g = np.random.default_rng(9200 + seed)
    M, N, K = _shape(g, *m_range)
    per_channel = bool(g.integers(0, 2))
    x = workloads.bf16_normal_with_outliers(g, (M, K))
    W = workloads.e4m3_codes(g, (N, K))
    sb = (workloads.uniform_f32(g, (N if per_channel else 1,), 0.5, 2.0) * np.float32(1e-3)).astype(np.float32)
    y = run_w16(fp8, to_dev_bf16(x), to_dev_e4m3(W), to_dev_f32(sb), 1 if per_channel else 0)
    y64, _ = orc.w8a16_mm(x, W, sb, per_channel)
    bound, acc = w16_bound(x, W, sb, per_channel, y64, orc, K, 16)
    from helpers import bf16_bits_to_f64
    err = np.abs(bf16_bits_to_f64(y) - y64)
    what = f"w16 sweep {M}x{N}x{K} pc={per_channel} (dispatch {fp8.w8a16_describe_dispatch(M, N, K)})"
    assert np.all(err <= bound + acc), what
    print(f"{what}: max err/acceptance bound {float(np.max(err / bound)):.4f}")
    assert fp8.get_device_error() == 0
