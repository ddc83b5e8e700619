"""One layer of the synthetic decode step (the benchmark's own step function,
the same launches with the same flags), run eagerly through the C ABI at
M in {1, 4, 8} on realistic weights: bf16 N(0, 0.02) quantised per output
channel on the GPU (checked byte-exact against the oracle's quantiser).  The
chain is RMSNorm -> static quant -> QKV; per-token quant of the attention
output stub -> O; gate_up on the normalised input; SiLU(gate) * up ->
per-token quant -> down.  Every quantised byte and scale is compared bit for
bit with the oracle's producer on the same input, and every GEMM output
element by element at the acceptance bound against the oracle's GEMM on the
oracle's own operands; the SiLU producer's input is the GPU gate_up output
(checked just before)."""
import os
import sys

import numpy as np
import pytest
import torch

import workloads
from helpers import check_gemm, host_bits, scale_product, to_dev_bf16

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fp8():
    import fp8_w8a8_scaled_gb300 as f
    f.clear_device_error()
    yield f
    assert f.get_device_error() == 0


@pytest.fixture(scope="module")
def layer(fp8, orc):
    """One layer's four weights, quantised per output channel on the GPU and
    by the oracle (the bytes and scales must agree)."""
    shapes = workloads.LayerShapes()
    g = workloads.rng(77)
    dev, host = [], []
    for (n, k) in (shapes.qkv, shapes.o, shapes.gate_up, shapes.down):
        w = workloads.bf16_normal(g, (n, k), std=0.02)
        q, sb = fp8.quant_fp8_per_token(to_dev_bf16(w))
        wq, wsb = orc.quant_per_token(w)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(q), wq) and np.array_equal(host_bits(sb), wsb)
        dev.append((q, sb))
        host.append((wq, wsb))
    return dev, host


def _gemm_check(orc, A, B, sa, sb, gran, y_bits, what):
    y64, _ = orc.scaled_mm(A, B, sa, sb, gran)
    M, N = y64.shape
    sab = scale_product(sa, sb, gran, np.arange(M)[:, None], np.arange(N)[None, :])
    worst, _ = check_gemm(y_bits, y64, sab, A.shape[1], what)
    print(f"{what}: max err/bound {worst:.4f}")


@pytest.mark.parametrize("M", [1, 4, 8])
def test_decode_step_layer_chain(fp8, orc, layer, M):
    sys.path.insert(0, ROOT)
    import bench
    dev, host = layer
    buf = {}
    step = bench.decode_step_fn(torch, fp8, torch.device("cuda", 0), [dev], M, buffers=buf)
    step(0)
    torch.cuda.synchronize()
    (wqkv, sqkv), (wo, so), (wgu, sgu), (wdn, sdn) = host
    x, gamma, o_in = host_bits(buf["x"]), host_bits(buf["gamma"]), host_bits(buf["o_in"])
    s_a = float(host_bits(buf["s_a"])[0])
    y_qkv, y_o, y_gu, y_dn = (host_bits(t) for t in buf["y"])
    # RMSNorm -> static quant, then QKV (per-tensor activation scale, per-channel weights)
    a = orc.rmsnorm_quant(x, gamma, workloads.RMS_EPS, s_a)
    assert np.array_equal(host_bits(buf["a"]), a)
    _gemm_check(orc, a, wqkv, [s_a], sqkv, 1, y_qkv, f"QKV M={M}")
    # attention-output stub -> per-token quant -> O (per-token x per-channel)
    a_o, s_o = orc.quant_per_token(o_in)
    assert np.array_equal(host_bits(buf["a_o"]), a_o) and np.array_equal(host_bits(buf["s_o"]), s_o)
    _gemm_check(orc, a_o, wo, s_o, so, 2, y_o, f"O M={M}")
    # gate_up on the same normalised input
    _gemm_check(orc, a, wgu, [s_a], sgu, 1, y_gu, f"gate_up M={M}")
    # SiLU(gate) * up -> per-token quant of the GPU gate_up output, then down
    a_d, s_d = orc.silu_mul_quant_per_token(y_gu)
    assert np.array_equal(host_bits(buf["a_d"]), a_d) and np.array_equal(host_bits(buf["s_d"]), s_d)
    _gemm_check(orc, a_d, wdn, s_d, sdn, 2, y_dn, f"down M={M}")
