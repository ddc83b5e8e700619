"""fp8_scaled_mm_noalloc, the entry point for callers that cannot allocate
device memory (code that runs inside a memory pool or arena that must own
every allocation, or while its allocator is locked).  It is called here
through the C ABI, twice in a row per case: both results must equal
fp8_scaled_mm's bit for bit (same kernel, same plan) and lie within the
acceptance bound of the oracle.  A fresh process checks that it allocates no
device memory.  This file is collected last on purpose."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import workloads
from helpers import bf16_bits_to_f64, check_gemm_tc, host_bits, scale_product, to_dev_e4m3, to_dev_f32

pytestmark = pytest.mark.gpu

FP8_OK = 0
FP8_ERR_TOO_LARGE = 6
GRAN_BLOCK = 4
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _noalloc():
    import fp8_w8a8_scaled_gb300 as fp8
    fn = fp8.lib().fp8_scaled_mm_noalloc
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [P, P, P, P, I32, I32, I64, I64, I64, P, P]
    fn.restype = I32
    return fp8, fn


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _oracle_check(orc, c, gran, y_bits, what):
    """Every output against the oracle: uniformly random codes, so the tensor
    core's binary32 accumulation inside a k-block gets its own bound beside
    the acceptance bound (blockwise: the largest scale product of the output
    stands in for the single one, and each scaled k-block sum is rounded once
    more)."""
    A, B, sa, sb = c["A"], c["B"], c["sa"], c["sb"]
    M, K = A.shape
    N = B.shape[0]
    if gran != GRAN_BLOCK:
        y64, _ = orc.scaled_mm(A, B, sa, sb, gran)
        sab = scale_product(sa, sb, gran, np.arange(M)[:, None], np.arange(N)[None, :])
        abs_sum = orc.gemm_acc_f64(np.asarray(A) & 0x7F, np.asarray(B) & 0x7F)
        check_gemm_tc(y_bits, y64, sab, K, abs_sum, what)
        return
    rr, cc = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    rows, cols = rr.ravel(), cc.ravel()
    y64 = orc.scaled_mm_block_points(A, B, sa, sb, rows, cols)
    abs_sum = orc.scaled_mm_block_points(np.asarray(A) & 0x7F, np.asarray(B) & 0x7F, np.abs(sa), np.abs(sb),
                                         rows, cols)
    kb = -(-K // 128)
    smax = np.max(np.abs(np.asarray(sa, np.float64).reshape(M, kb)[rows] *
                         np.asarray(sb, np.float64).reshape(-(-N // 128), kb)[cols // 128]), axis=1)
    bound = 1e-2 * np.abs(y64) + 1e-3 * np.sqrt(K) * smax + (-(-K // 32) + kb + 1) * 2.0 ** -23 * abs_sum
    y = bf16_bits_to_f64(np.asarray(y_bits).reshape(M, N)[rows, cols])
    assert np.all(np.abs(y - y64) <= bound), what


# (M, N, K, gran): the decode kernel's cluster mode (no scratch) and its
# stream-K mode (the fixed scratch), exact sums and blockwise TwoSum parts
CASES = [(1, 10240, 5120, 1), (16, 2048, 5120, 2), (5, 520, 1040, 3), (9, 1032, 4096, 0),
         (16, 2048, 5120, GRAN_BLOCK), (3, 6144, 1040, GRAN_BLOCK)]


@pytest.mark.parametrize("M,N,K,gran", CASES)
def test_noalloc_matches_scaled_mm_twice(orc, M, N, K, gran):
    """Two calls in a row: bitwise equal to fp8_scaled_mm and within the
    oracle's bound."""
    fp8, fn = _noalloc()
    c = workloads.random_gemm(7100 + M + N + K + gran, M, N, K, gran)
    A, B = to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"])
    sa, sb = to_dev_f32(c["sa"].ravel()), to_dev_f32(c["sb"].ravel())
    ref = host_bits(fp8.fp8_scaled_mm(A, B, sa, sb, gran))
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = fn(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), gran, 0, M, N, K, _ptr(out), stream)
        assert st == FP8_OK, fp8.status_string(st)
        torch.cuda.synchronize()
        y = host_bits(out)
        assert np.array_equal(y, ref)
        _oracle_check(orc, c, gran, y, f"noalloc {M}x{N}x{K} gran {gran}")
    assert fp8.get_device_error() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    fp8, fn = _noalloc()
    A = torch.zeros((17, 64), dtype=torch.float8_e4m3fn, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.float8_e4m3fn, device="cuda")
    s = torch.ones(1, device="cuda")
    out = torch.empty((17, 64), dtype=torch.bfloat16, device="cuda")
    st = fn(_ptr(A), _ptr(B), _ptr(s), _ptr(s), 0, 0, 17, 64, 64, _ptr(out),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == FP8_ERR_TOO_LARGE


_FRESH = r"""
import ctypes, sys
sys.path.insert(0, %r)
import numpy as np, torch
import fp8_w8a8_scaled_gb300 as fp8
import workloads
fn = fp8.lib().fp8_scaled_mm_noalloc
P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
fn.argtypes = [P, P, P, P, I32, I32, I64, I64, I64, P, P]
fn.restype = I32
def mem_free():
    f, _ = torch.cuda.mem_get_info()
    return f
ops = []
for M, N, K, gran in ((16, 2048, 5120, 2), (1, 10240, 5120, 1), (16, 2048, 5120, 4)):
    c = workloads.random_gemm(7200 + M + N, M, N, K, gran)
    A = torch.from_numpy(c["A"]).view(torch.float8_e4m3fn).cuda()
    B = torch.from_numpy(c["B"]).view(torch.float8_e4m3fn).cuda()
    sa = torch.from_numpy(np.ascontiguousarray(c["sa"].ravel())).cuda()
    sb = torch.from_numpy(np.ascontiguousarray(c["sb"].ravel())).cuda()
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ops.append((A, B, sa, sb, gran, M, N, K, out))
s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
def run_all():
    for A, B, sa, sb, gran, M, N, K, out in ops:
        st = fn(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()), ctypes.c_void_p(sa.data_ptr()),
                ctypes.c_void_p(sb.data_ptr()), gran, 0, M, N, K, ctypes.c_void_p(out.data_ptr()), s)
        assert st == 0, fp8.status_string(st)
    torch.cuda.synchronize()
# the first calls load the library's kernels (module loading reserves device
# memory for code and the fixed scratch array); after that, calls of every
# kind must leave the free device memory unchanged
run_all()
before = mem_free()
for _ in range(3):
    run_all()
after = mem_free()
assert before == after, (before, after)
assert fp8.get_device_error() == 0
print("noalloc-fresh-ok", before - after)
""" % ROOT


def test_noalloc_allocates_nothing_in_a_fresh_process():
    """In a new process whose first library GEMM calls are fp8_scaled_mm_noalloc
    (so fp8_scaled_mm's per-stream scratch was never made): repeated calls of
    the cluster and stream-K modes, exact and blockwise, leave the free device
    memory exactly unchanged."""
    r = subprocess.run([sys.executable, "-c", _FRESH], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "noalloc-fresh-ok 0" in r.stdout
