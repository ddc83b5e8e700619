"""GPU tests of fp8_rmsnorm_quant_scaled_mm, the RMSNorm -> static quant ->
GEMM call: its E4M3 activations are byte-identical to rmsnorm_quant_fp8 (and
so to the oracle's), its GEMM output is byte-identical to fp8_scaled_mm on
those activations (and within the acceptance bound of the oracle), on the
decode and the tile kernel, across repeated calls and CUDA-graph replays."""
import numpy as np
import pytest
import torch

import workloads
from helpers import check_gemm, host_bits, scale_product, to_dev_bf16, to_dev_e4m3, to_dev_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    import fp8_w8a8_scaled_gb300 as f
    f.clear_device_error()
    yield f
    assert f.get_device_error() == 0


@pytest.fixture(scope="module")
def case(orc):
    d = workloads.decode_fused(seed=5)
    A_all = orc.rmsnorm_quant(d["x"], d["gamma"], d["eps"], float(d["s_a"]))
    y64, _ = orc.scaled_mm(A_all, d["B"], d["s_a"], d["sb"], 1)
    dev = dict(x=to_dev_bf16(d["x"]), gamma=to_dev_bf16(d["gamma"]), sa=to_dev_f32(d["s_a"]),
               B=to_dev_e4m3(d["B"]), sb=to_dev_f32(d["sb"]))
    return d, A_all, y64, dev


@pytest.mark.parametrize("M", [1, 2, 3, 8, 16, 17, 32])
def test_fused_matches_norm_then_gemm(fp8, case, M):
    d, A_all, y64, dev = case
    a, y = fp8.rmsnorm_quant_scaled_mm(dev["x"][:M], dev["gamma"], d["eps"], dev["sa"], dev["B"], dev["sb"], 1,
                                       flags=fp8.FLAG_WEIGHTS_STATIC)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(a), A_all[:M])
    ref = fp8.fp8_scaled_mm(a, dev["B"], dev["sa"], dev["sb"], 1)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(y), host_bits(ref))
    sab = scale_product(d["s_a"], d["sb"], 1, np.arange(M)[:, None], np.arange(10240)[None, :])
    worst, _ = check_gemm(host_bits(y), y64[:M], sab, 5120, f"fused M={M}")
    print(f"fused M={M}: max err/bound {worst:.4f}")


@pytest.mark.parametrize("M,N,K,gran", [(33, 1032, 2064, 1), (64, 2048, 5120, 0), (8, 520, 17408, 1),
                                        (5, 264, 400, 0), (16, 128, 128, 1)])
def test_fused_other_paths(fp8, orc, M, N, K, gran):
    """Tile-kernel M, a long row, small ragged decode shapes, per-tensor or
    per-channel weight scales."""
    g = workloads.rng(6000 + M + N + K)
    x = workloads.bf16_normal(g, (M, K))
    gamma = workloads.bf16_normal(g, (K,), mean=1.0, std=0.1)
    B = workloads.e4m3_codes(g, (N, K))
    sb = (workloads.uniform_f32(g, (N if gran == 1 else 1,), 0.5, 2.0) * np.float32(1e-3)).astype(np.float32)
    s_a = float(workloads.STATIC_INPUT_SCALE)
    a, y = fp8.rmsnorm_quant_scaled_mm(to_dev_bf16(x), to_dev_bf16(gamma), 1e-6, to_dev_f32(s_a), to_dev_e4m3(B),
                                       to_dev_f32(sb), gran)
    torch.cuda.synchronize()
    want_a = orc.rmsnorm_quant(x, gamma, 1e-6, s_a)
    assert np.array_equal(host_bits(a), want_a)
    ref = fp8.fp8_scaled_mm(a, to_dev_e4m3(B), to_dev_f32(s_a), to_dev_f32(sb), gran)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(y), host_bits(ref))


def test_fused_repeated_and_graph(fp8, case, orc):
    """Back-to-back calls on different rows, then a graph of three calls
    replayed three times: every result right."""
    d, A_all, y64, dev = case
    outs = []
    for m in (4, 1, 32, 16, 4):
        outs.append((m, fp8.rmsnorm_quant_scaled_mm(dev["x"][:m], dev["gamma"], d["eps"], dev["sa"], dev["B"],
                                                    dev["sb"], 1)))
    torch.cuda.synchronize()
    for m, (a, y) in outs:
        assert np.array_equal(host_bits(a), A_all[:m])
        ref = fp8.fp8_scaled_mm(a, dev["B"], dev["sa"], dev["sb"], 1)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(y), host_bits(ref))
    ms = (1, 8, 32)
    a_bufs = [torch.empty((m, 5120), dtype=torch.float8_e4m3fn, device="cuda") for m in ms]
    y_bufs = [torch.empty((m, 10240), dtype=torch.bfloat16, device="cuda") for m in ms]

    def run():
        for m, a, y in zip(ms, a_bufs, y_bufs):
            fp8.rmsnorm_quant_scaled_mm(dev["x"][:m], dev["gamma"], d["eps"], dev["sa"], dev["B"], dev["sb"], 1,
                                        a_out=a, out=y, flags=fp8.FLAG_WEIGHTS_STATIC)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [host_bits(y) for y in y_bufs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(3):
        for a, y in zip(a_bufs, y_bufs):
            a.view(torch.uint8).zero_()
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for m, a, y, e in zip(ms, a_bufs, y_bufs, eager):
            assert np.array_equal(host_bits(a), A_all[:m])
            assert np.array_equal(host_bits(y), e)
