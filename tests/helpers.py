"""Shared test helpers: host <-> device conversion of bit patterns, the GEMM
acceptance bound, and guard-band canaries around output buffers."""
import numpy as np
import torch

GUARD = 256          # bytes of canary before and after an output buffer
CANARY = 0xA5


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 on cuda:0 (bit-preserving)."""
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev_e4m3(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).cuda()


def to_dev_f32(v) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.atleast_1d(v), np.float32)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> its raw bytes reinterpreted as an unsigned numpy array."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return t.view(torch.uint8).numpy()
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def scale_product(sa, sb, gran, rows, cols):
    """sa*sb (binary64) for the (rows, cols) outputs under a granularity."""
    sa = np.atleast_1d(np.asarray(sa, np.float32)).astype(np.float64)
    sb = np.atleast_1d(np.asarray(sb, np.float32)).astype(np.float64)
    a = sa[rows] if gran in (2, 3) else sa[0]
    b = sb[cols] if gran in (1, 2) else sb[0]
    return a * b


def gemm_bound(y64: np.ndarray, sab: np.ndarray, K: int) -> np.ndarray:
    """Acceptance bound of the scaled GEMM, element-wise:
    |y - ref| <= 1e-2 * |ref| + 1e-3 * (scale_a * scale_b) * sqrt(K)."""
    return 1e-2 * np.abs(y64) + 1e-3 * np.abs(sab) * np.sqrt(K)


def check_gemm(y_bits: np.ndarray, y64: np.ndarray, sab: np.ndarray, K: int, what: str = ""):
    """Asserts every output is within the bound; returns (max err/bound, count)."""
    y = bf16_bits_to_f64(y_bits)
    err = np.abs(y - y64)
    bound = gemm_bound(y64, sab, K)
    ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1), np.where(err > 0, np.inf, 0.0))
    bad = ~(err <= bound)
    worst = float(np.nanmax(ratio)) if ratio.size else 0.0
    assert not np.any(np.isnan(y[~np.isnan(y64)])), f"{what}: NaN in GPU output"
    assert int(bad.sum()) == 0, (f"{what}: {int(bad.sum())} of {bad.size} outputs outside the bound; "
                                 f"max err/bound {worst:.3g}")
    return worst, int(bad.size)


def tc_accumulation_bound(abs_sum: np.ndarray, sab: np.ndarray, K: int) -> np.ndarray:
    """Worst-case error of accumulating the K exact E4M3 products in binary32
    on the tensor core, from the arithmetic alone: the sum is formed as
    ceil(K/32) chunk sums added one after another into a binary32 accumulator,
    each step (including the chunk's own reduction) off by at most one unit
    in the last place of a partial sum whose magnitude is at most
    sum_k |a_k * b_k|; so |error| <= (ceil(K/32) + 1) * 2^-23 * sum_k |a_k * b_k|,
    times the scales.  `abs_sum` is sum_k |a_k * b_k| in code units."""
    steps = -(-K // 32) + 1
    return steps * 2.0 ** -23 * np.abs(sab) * abs_sum


def check_gemm_tc(y_bits, y64, sab, K, abs_sum, what=""):
    """For outputs of the large-M kernel on stress inputs (uniformly random
    codes, outlier-free activations) whose partial sums are large next to the
    acceptance bound's absolute term: asserts |y - ref| <= bound + the binary32
    accumulation bound above.  Returns (max err / acceptance bound,
    max err / (bound + accumulation bound))."""
    y = bf16_bits_to_f64(y_bits)
    err = np.abs(y - y64)
    bound = gemm_bound(y64, sab, K)
    total = bound + tc_accumulation_bound(abs_sum, sab, K)
    assert not np.any(np.isnan(y[~np.isnan(y64)])), f"{what}: NaN in GPU output"
    bad = ~(err <= total)
    r_acc = float(np.max(err / np.where(bound > 0, bound, np.inf))) if err.size else 0.0
    r_tot = float(np.max(err / np.where(total > 0, total, np.inf))) if err.size else 0.0
    assert int(bad.sum()) == 0, f"{what}: {int(bad.sum())} outputs outside bound + accumulation bound ({r_tot:.3g})"
    return r_acc, r_tot


class Guarded:
    """A device buffer of `nbytes` with canary bands on both sides."""

    def __init__(self, nbytes: int):
        self.nbytes = nbytes
        self.raw = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        return self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        head = self.raw[:GUARD].cpu().numpy()
        tail = self.raw[GUARD + self.nbytes:].cpu().numpy()
        return bool(np.all(head == CANARY) and np.all(tail == CANARY))
