"""fp8_scaled_mm_noalloc, the entry point for callers that cannot allocate
device memory (code that runs inside a memory pool or arena that must own
every allocation, or while its allocator is locked).  It is called here
through the C ABI, twice in a row, and must agree with fp8_scaled_mm within
the GEMM acceptance bound.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from helpers import bf16_bits_to_f64, gemm_bound, host_bits, scale_product, to_dev_e4m3, to_dev_f32

pytestmark = pytest.mark.gpu

FP8_OK = 0
FP8_ERR_TOO_LARGE = 6


def _noalloc():
    import fp8_w8a8_scaled_gb300 as fp8
    fn = fp8.lib().fp8_scaled_mm_noalloc
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [P, P, P, P, I32, I32, I64, I64, I64, P, P]
    fn.restype = I32
    return fp8, fn


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("M,N,K,gran", [(1, 10240, 5120, 1), (16, 2056, 3088, 2), (5, 520, 1040, 3)])
def test_noalloc_matches_scaled_mm_twice(M, N, K, gran):
    fp8, fn = _noalloc()
    c = workloads.random_gemm(7000 + M + N + K, M, N, K, gran)
    A, B = to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"])
    sa, sb = to_dev_f32(c["sa"]), to_dev_f32(c["sb"])
    ref = fp8.fp8_scaled_mm(A, B, sa, sb, gran)
    torch.cuda.synchronize()
    y_ref = bf16_bits_to_f64(host_bits(ref))
    bound = gemm_bound(y_ref, scale_product(c["sa"], c["sb"], gran, np.arange(M)[:, None], np.arange(N)[None, :]), K)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = fn(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), gran, 0, M, N, K, _ptr(out), stream)
        assert st == FP8_OK, fp8.status_string(st)
        torch.cuda.synchronize()
        y = bf16_bits_to_f64(host_bits(out))
        assert np.all(np.abs(y - y_ref) <= bound)
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
