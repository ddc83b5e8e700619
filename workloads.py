"""Seeded synthetic inputs for the FP8 W8A8 scaled-GEMM workloads.

Shared by the tests (both the CUDA side and the CPU oracle side) and by the
benchmark.  It holds none of the method's arithmetic: no quantisation, no
rounding to bf16, no scaling.  It only draws random numbers and lays them out:

* bf16 inputs are drawn as binary32 values and *truncated* to their upper 16
  bits, which is a way of drawing random bf16 numbers, not the round-to-nearest
  conversion the method specifies;
* E4M3 operands that the workloads do not derive by quantisation are drawn as
  uniformly random codes, skipping the two NaN codes 0x7F and 0xFF;
* scales are drawn as binary32 numbers.

Every array is a pure function of (seed, shape); the numpy generator is
``default_rng(seed)`` consumed in a fixed call order.
"""
from dataclasses import dataclass

import numpy as np

# --- workload shapes ---------------------------------------------------------------

HIDDEN = 5120          # model width K of the QKV / gate_up projections
QKV_N = 10240          # merged q|k|v output width (q 8192, k 1024, v 1024)
Q_WIDTH, KV_WIDTH = 8192, 1024
O_K = 8192             # O projection input width
GATE_UP_N = 34816      # merged gate|up output width (17408 + 17408)
DOWN_K = 17408         # down projection input width
RMS_EPS = 1e-6
# Static activation scale of the decode workloads: a fixed, checkpoint-style
# `input_scale`.  1/56 maps |h| <= 8 into the E4M3 range (8 / (1/56) = 448).
STATIC_INPUT_SCALE = np.float32(1.0 / 56.0)

TINY = dict(M=4, K=256, N=512)
DECODE_FUSED_MS = (1, 2, 4, 8, 16, 32)
GATE_UP_MS = (1, 8, 32, 64)
PREFILL_MS = (2048, 8192)
PREFILL_NS = (QKV_N, GATE_UP_N)
STEP_MS = (1, 4, 8)
STEP_LAYERS = 64


@dataclass(frozen=True)
class LayerShapes:
    """The four projections of one synthetic decoder layer: (N, K) each."""
    qkv: tuple = (QKV_N, HIDDEN)
    o: tuple = (HIDDEN, O_K)
    gate_up: tuple = (GATE_UP_N, HIDDEN)
    down: tuple = (HIDDEN, DOWN_K)

    def weight_bytes(self) -> int:
        return sum(n * k for n, k in (self.qkv, self.o, self.gate_up, self.down))


# --- primitive draws -----------------------------------------------------------------

def rng(seed: int = 0) -> np.random.Generator:
    return np.random.default_rng(seed)


def _truncate_to_bf16_bits(v32: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(v32, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_normal(g: np.random.Generator, shape, mean=0.0, std=1.0) -> np.ndarray:
    """Random bf16 bit patterns (uint16) drawn around N(mean, std^2)."""
    v = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    if mean != 0.0:
        v += np.float32(mean)
    return _truncate_to_bf16_bits(v)


def bf16_normal_with_outliers(g, shape, p=0.01, factor=20.0) -> np.ndarray:
    """N(0,1) bf16 with each element independently (probability p) multiplied by factor."""
    v = g.standard_normal(size=shape, dtype=np.float32)
    mask = g.random(size=shape, dtype=np.float32) < np.float32(p)
    v[mask] *= np.float32(factor)
    return _truncate_to_bf16_bits(v)


_NON_NAN_CODES = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


def e4m3_codes(g: np.random.Generator, shape) -> np.ndarray:
    """Uniformly random non-NaN E4M3 codes (uint8)."""
    idx = g.integers(0, _NON_NAN_CODES.size, size=shape, dtype=np.int64)
    return _NON_NAN_CODES[idx]


def uniform_f32(g: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return g.uniform(lo, hi, size=shape).astype(np.float32)


# --- the workloads ---------------------------------------------------------------------

def tiny_gemm(seed: int = 0):
    """Tiny GEMM, M=4, K=256, N=512: bf16 activations N(0,1) and bf16 weights
    N(0, 0.02); both are quantised per-tensor (scale = amax/448) by the side
    under test."""
    g = rng(seed)
    M, K, N = TINY["M"], TINY["K"], TINY["N"]
    x = bf16_normal(g, (M, K))
    w = bf16_normal(g, (N, K), std=0.02)
    return dict(x=x, w=w, M=M, K=K, N=N)


def decode_fused(seed: int = 0, n: int = QKV_N, k: int = HIDDEN, rows: int = 32):
    """Decode fused path: x bf16 [32,K] N(0,1) (the M-row cases use rows 0..M-1),
    gamma = 1 + N(0, 0.1) in bf16, eps 1e-6, a static activation scale, and a
    merged-QKV weight of random E4M3 codes [N,K] with per-output-channel scales
    drawn U(0.5, 2) * 1e-3."""
    g = rng(seed)
    x = bf16_normal(g, (rows, k))
    gamma = bf16_normal(g, (k,), mean=1.0, std=0.1)
    B = e4m3_codes(g, (n, k))
    sb = (uniform_f32(g, (n,), 0.5, 2.0) * np.float32(1e-3)).astype(np.float32)
    return dict(x=x, gamma=gamma, B=B, sb=sb, eps=RMS_EPS, s_a=STATIC_INPUT_SCALE, N=n, K=k)


def gate_up_decode(seed: int = 0, rows: int = 64, n: int = GATE_UP_N, k: int = HIDDEN):
    """Merged gate_up decode GEMM: bf16 weights N(0, 0.02) [N,K] (quantised
    per output channel by the side under test) and bf16 activations N(0,1)
    [rows,K] quantised with the static activation scale."""
    g = rng(seed)
    w = bf16_normal(g, (n, k), std=0.02)
    x = bf16_normal(g, (rows, k))
    return dict(w=w, x=x, s_a=STATIC_INPUT_SCALE, N=n, K=k)


def prefill(seed: int = 0, m: int = 2048, n: int = QKV_N, k: int = HIDDEN):
    """Prefill chunk: activations N(0,1) with 1% outliers x20 (quantised per
    token by the side under test) and bf16 weights N(0, 0.02) (quantised per
    output channel)."""
    g = rng(seed)
    x = bf16_normal_with_outliers(g, (m, k))
    w = bf16_normal(g, (n, k), std=0.02)
    return dict(x=x, w=w, M=m, N=n, K=k)


def random_gemm(seed: int, M: int, N: int, K: int, gran: int):
    """Random E4M3 operands and positive scales for a GEMM of the given shape
    and granularity (0 per-tensor, 1 per-channel, 2 per-token x channel,
    3 per-token, 4 blockwise: sa [M, ceil(K/128)], sb [ceil(N/128), ceil(K/128)])."""
    g = rng(seed)
    A = e4m3_codes(g, (M, K))
    B = e4m3_codes(g, (N, K))
    if gran == 4:
        na = (M, -(-K // 128))
        nb = (-(-N // 128), -(-K // 128))
    else:
        na = (M if gran in (2, 3) else 1,)
        nb = (N if gran in (1, 2) else 1,)
    sa = uniform_f32(g, na, 0.25, 4.0) * np.float32(1e-2)
    sb = uniform_f32(g, nb, 0.25, 4.0) * np.float32(1e-3)
    return dict(A=A, B=B, sa=sa.astype(np.float32), sb=sb.astype(np.float32))


# --- device-side draws for the workloads too large to draw on the host -------------------

def device_e4m3_codes(torch, shape, seed: int, device):
    """Uniform non-NaN E4M3 codes drawn with torch's seeded device generator."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    idx = torch.randint(0, _NON_NAN_CODES.size, shape, generator=gen, device=device, dtype=torch.int32)
    table = torch.as_tensor(_NON_NAN_CODES, device=device)
    return table[idx]


def device_uniform_f32(torch, shape, lo: float, hi: float, seed: int, device):
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.empty(shape, dtype=torch.float32, device=device).uniform_(lo, hi, generator=gen)


def device_bf16_normal(torch, shape, seed: int, device, std: float = 1.0, mean: float = 0.0):
    """Random bf16 values drawn around N(mean, std^2) on the device (truncated draws)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    if mean != 0.0:
        v.add_(mean)
    return (v.view(torch.int32) >> 16).to(torch.int16).view(torch.bfloat16)
