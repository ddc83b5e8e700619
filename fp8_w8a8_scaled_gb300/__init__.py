"""Python binding of the GB300 FP8 (E4M3) W8A8 scaled-GEMM library.

Argument marshalling only: every function here checks torch tensor dtypes,
shapes, contiguity and devices, then calls the C ABI of ``libfp8w8a8``
(``include/fp8w8a8.h``) with raw device pointers and the current torch CUDA
stream.  All arithmetic happens in the library's CUDA kernels; there is no
fallback of any kind -- if the library is missing or a call fails, an
exception is raised.

Functions carry the C names: ``fp8_scaled_mm``, ``rmsnorm_quant_fp8``,
``quant_fp8_per_token``, ``quant_fp8_static``, and the blockwise-scaling
quantisers ``quant_per_token_group`` / ``quant_weight_block``.
"""
import ctypes
import os
import platform

import torch

HERE = os.path.dirname(os.path.abspath(__file__))

FP8_OK = 0
FP8_ERR_INVALID_ARG = 1
FP8_ERR_ALIGNMENT = 2
FP8_ERR_UNSUPPORTED = 3
FP8_ERR_CUDA = 4
FP8_ERR_DEVICE = 5

GRAN_PER_TENSOR = 0
GRAN_PER_CHANNEL = 1
GRAN_PER_TOKEN_CHANNEL = 2
GRAN_PER_TOKEN = 3
GRAN_BLOCK_128 = 4
BLOCK = 128

OUT_BF16 = 0

FLAG_WEIGHTS_STATIC = 1
FLAG_NO_PDL = 2

KERNEL_NONE = 0
KERNEL_DECODE_SPLITK = 1
KERNEL_PREFILL = 2
KERNEL_W16_DECODE = 3
KERNEL_W16_DENSE = 4
KERNEL_W16_GEMV = 5

E4M3 = torch.float8_e4m3fn

_lib = None
_current_device = None


class Fp8Error(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def lib_path() -> str:
    return os.path.join(HERE, "_build", f"libfp8w8a8_{platform.machine()}.so")


def lib():
    """The loaded C library (ctypes.CDLL) with argument types declared."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libfp8w8a8 is not built ({path} missing): run __graft_entry__.build() "
                           "or python fp8_w8a8_scaled_gb300/build.py")
    L = ctypes.CDLL(path)
    P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    L.fp8_scaled_mm.argtypes = [P, P, P, P, I32, I32, I64, I64, I64, P, P]
    L.fp8_scaled_mm.restype = I32
    L.fp8_scaled_mm_ex.argtypes = [P, P, P, P, I32, I32, I64, I64, I64, P, P, ctypes.c_uint]
    L.fp8_scaled_mm_ex.restype = I32
    L.fp8_rmsnorm_quant_scaled_mm.argtypes = [P, P, F32, P, P, P, I32, I32, I64, I64, I64, P, P, P, ctypes.c_uint]
    L.fp8_rmsnorm_quant_scaled_mm.restype = I32
    L.fp8_requant_merge.argtypes = [P, P, P, I32, I64, P, P, P]
    L.fp8_requant_merge.restype = I32
    L.fp8_silu_mul_quant_per_token.argtypes = [P, P, P, I64, I64, P]
    L.fp8_silu_mul_quant_per_token.restype = I32
    L.fp8_add_rmsnorm_quant.argtypes = [P, P, P, F32, P, P, I64, I64, P]
    L.fp8_add_rmsnorm_quant.restype = I32
    L.rmsnorm_quant_fp8.argtypes = [P, P, F32, P, P, I64, I64, P]
    L.rmsnorm_quant_fp8.restype = I32
    L.quant_fp8_per_token.argtypes = [P, P, P, I64, I64, P]
    L.quant_fp8_per_token.restype = I32
    L.fp8_w8a16_mm.argtypes = [P, P, P, I32, I32, I64, I64, I64, P, P]
    L.fp8_w8a16_mm.restype = I32
    L.fp8_w8a16_mm_ex.argtypes = [P, P, P, I32, I32, I64, I64, I64, P, P, ctypes.c_uint]
    L.fp8_w8a16_mm_ex.restype = I32
    L.fp8_w8a16_describe_dispatch.argtypes = [I64, I64, I64]
    L.fp8_w8a16_describe_dispatch.restype = I32
    L.fp8_widen_weight.argtypes = [P, P, I32, I64, I64, P, P]
    L.fp8_widen_weight.restype = I32
    L.fp8_quant_per_token_group.argtypes = [P, P, P, I64, I64, P]
    L.fp8_quant_per_token_group.restype = I32
    L.fp8_quant_weight_block.argtypes = [P, P, P, I64, I64, P]
    L.fp8_quant_weight_block.restype = I32
    L.quant_fp8_static.argtypes = [P, P, P, I64, I64, P]
    L.quant_fp8_static.restype = I32
    L.fp8_status_string.argtypes = [I32]
    L.fp8_status_string.restype = ctypes.c_char_p
    L.fp8_describe_dispatch.argtypes = [I64, I64, I64, I32]
    L.fp8_describe_dispatch.restype = I32
    L.fp8_decode_ctas.argtypes = [I64, I64, I64]
    L.fp8_decode_ctas.restype = I32
    L.fp8_decode_split_for_sms.argtypes = [I64, I64, I64, I32, I32]
    L.fp8_decode_split_for_sms.restype = I32
    L.fp8_decode_ctas_for_sms.argtypes = [I64, I64, I64, I32, I32]
    L.fp8_decode_ctas_for_sms.restype = I32
    L.fp8_decode_exact_for_sms.argtypes = [I64, I64, I64, I32, I32]
    L.fp8_decode_exact_for_sms.restype = I32
    L.fp8_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    L.fp8_get_device_error.restype = I32
    L.fp8_selftest_bounded_wait.argtypes = [ctypes.c_uint32, P]
    L.fp8_selftest_bounded_wait.restype = I32
    L.fp8_clear_device_error.argtypes = []
    L.fp8_clear_device_error.restype = I32
    L.fp8_library_version.argtypes = []
    L.fp8_library_version.restype = I32
    L.fp8_set_device.argtypes = [I32]
    L.fp8_set_device.restype = I32
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().fp8_status_string(int(status)).decode()


def _check(status, what):
    if status != FP8_OK:
        raise Fp8Error(status, what)


def _stream_of(t: torch.Tensor):
    global _current_device
    dev = t.device.index if t.device.index is not None else torch.cuda.current_device()
    if dev != _current_device:
        _check(lib().fp8_set_device(dev), "fp8_set_device")
        _current_device = dev
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t: torch.Tensor, name: str, dtypes, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, has {t.dim()}")


_FP8 = (E4M3, torch.uint8)


def fp8_scaled_mm(A, B, scale_a, scale_b, granularity=None, out_dtype=OUT_BF16, out=None, flags=0):
    """y = bf16((A @ B.T) * scale_a * scale_b) for E4M3 A [M,K] and B [N,K].

    ``granularity`` defaults from the scales: 2-D scales [M, ceil(K/128)] and
    [ceil(N/128), ceil(K/128)] select the blockwise form, otherwise scale_a
    has 1 or M elements and scale_b 1 or N.  ``flags`` are the C ABI's
    fp8_flags (FLAG_WEIGHTS_STATIC, FLAG_NO_PDL)."""
    _need(A, "A", _FP8, 2)
    _need(B, "B", _FP8, 2)
    _need(scale_a, "scale_a", (torch.float32,))
    _need(scale_b, "scale_b", (torch.float32,))
    M, K = A.shape
    N, Kb = B.shape
    if Kb != K:
        raise ValueError(f"A is [{M},{K}] but B is [{N},{Kb}]")
    if granularity is None and (scale_a.dim() == 2 or scale_b.dim() == 2):
        granularity = GRAN_BLOCK_128
    if granularity is None:
        tok = scale_a.numel() == M and M != 1
        ch = scale_b.numel() == N and N != 1
        granularity = {(False, False): 0, (False, True): 1, (True, True): 2, (True, False): 3}[(tok, ch)]
    KB = (K + BLOCK - 1) // BLOCK
    if granularity == GRAN_BLOCK_128:
        want_a, want_b = M * KB, ((N + BLOCK - 1) // BLOCK) * KB
    else:
        want_a = M if granularity in (2, 3) else 1
        want_b = N if granularity in (1, 2) else 1
    if scale_a.numel() < want_a or scale_b.numel() < want_b:
        raise ValueError(f"granularity {granularity} needs scale_a[{want_a}], scale_b[{want_b}]")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    else:
        _need(out, "out", (torch.bfloat16,), 2)
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must be [{M},{N}]")
    _check(lib().fp8_scaled_mm_ex(_ptr(A), _ptr(B), _ptr(scale_a), _ptr(scale_b), int(granularity),
                                  int(out_dtype), M, N, K, _ptr(out), _stream_of(A), int(flags)), "fp8_scaled_mm")
    return out


def rmsnorm_quant_fp8(x, gamma, eps, scale, out=None):
    """Fused RMSNorm -> static E4M3 quantisation of bf16 x [M,K]."""
    _need(x, "x", (torch.bfloat16,), 2)
    _need(gamma, "gamma", (torch.bfloat16,), 1)
    _need(scale, "scale", (torch.float32,))
    M, K = x.shape
    if gamma.numel() != K:
        raise ValueError("gamma must have K elements")
    if out is None:
        out = torch.empty((M, K), dtype=E4M3, device=x.device)
    else:
        _need(out, "out", _FP8, 2)
    _check(lib().rmsnorm_quant_fp8(_ptr(x), _ptr(gamma), float(eps), _ptr(scale), _ptr(out), M, K, _stream_of(x)),
           "rmsnorm_quant_fp8")
    return out


def rmsnorm_quant_scaled_mm(x, gamma, eps, scale_a, B, scale_b, granularity=None, a_out=None, out=None, flags=0):
    """rmsnorm_quant_fp8(x) into a_out, then fp8_scaled_mm(a_out, B) into out,
    as one call (one launch at decode M); returns (a_out, out).  The activation
    scale is per tensor; ``granularity`` (0 or 1) defaults from scale_b."""
    _need(x, "x", (torch.bfloat16,), 2)
    _need(gamma, "gamma", (torch.bfloat16,), 1)
    _need(scale_a, "scale_a", (torch.float32,))
    _need(B, "B", _FP8, 2)
    _need(scale_b, "scale_b", (torch.float32,))
    M, K = x.shape
    N, Kb = B.shape
    if Kb != K or gamma.numel() != K:
        raise ValueError(f"x is [{M},{K}], B is [{N},{Kb}], gamma has {gamma.numel()} elements")
    if granularity is None:
        granularity = 1 if (scale_b.numel() == N and N != 1) else 0
    if scale_b.numel() < (N if granularity == 1 else 1):
        raise ValueError(f"granularity {granularity} needs scale_b[{N if granularity == 1 else 1}]")
    if a_out is None:
        a_out = torch.empty((M, K), dtype=E4M3, device=x.device)
    else:
        _need(a_out, "a_out", _FP8, 2)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    else:
        _need(out, "out", (torch.bfloat16,), 2)
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must be [{M},{N}]")
    _check(lib().fp8_rmsnorm_quant_scaled_mm(_ptr(x), _ptr(gamma), float(eps), _ptr(scale_a), _ptr(B), _ptr(scale_b),
                                             int(granularity), OUT_BF16, M, N, K, _ptr(a_out), _ptr(out),
                                             _stream_of(x), int(flags)), "fp8_rmsnorm_quant_scaled_mm")
    return a_out, out


def add_rmsnorm_quant_fp8(x, residual, gamma, eps, scale, out=None):
    """residual <- bf16(x + residual) in place, then the fused RMSNorm -> static
    E4M3 quantisation of it; returns the E4M3 [M,K] output."""
    _need(x, "x", (torch.bfloat16,), 2)
    _need(residual, "residual", (torch.bfloat16,), 2)
    _need(gamma, "gamma", (torch.bfloat16,), 1)
    _need(scale, "scale", (torch.float32,))
    M, K = x.shape
    if tuple(residual.shape) != (M, K) or gamma.numel() != K:
        raise ValueError("residual must match x; gamma must have K elements")
    if out is None:
        out = torch.empty((M, K), dtype=E4M3, device=x.device)
    else:
        _need(out, "out", _FP8, 2)
    _check(lib().fp8_add_rmsnorm_quant(_ptr(x), _ptr(residual), _ptr(gamma), float(eps), _ptr(scale), _ptr(out), M,
                                       K, _stream_of(x)), "fp8_add_rmsnorm_quant")
    return out


def silu_mul_quant_per_token(gate_up, out=None, scale_out=None):
    """silu(gate) * up for bf16 rows [gate | up] ([M, 2I]), quantised per token;
    returns (q E4M3 [M, I], s f32 [M])."""
    _need(gate_up, "gate_up", (torch.bfloat16,), 2)
    M, W = gate_up.shape
    if W % 2:
        raise ValueError("gate_up rows must hold [gate | up]")
    I = W // 2
    if out is None:
        out = torch.empty((M, I), dtype=E4M3, device=gate_up.device)
    else:
        _need(out, "out", _FP8, 2)
    if scale_out is None:
        scale_out = torch.empty((M,), dtype=torch.float32, device=gate_up.device)
    else:
        _need(scale_out, "scale_out", (torch.float32,))
    _check(lib().fp8_silu_mul_quant_per_token(_ptr(gate_up), _ptr(out), _ptr(scale_out), M, I,
                                              _stream_of(gate_up)), "fp8_silu_mul_quant_per_token")
    return out, scale_out


def requant_merge(shards, scales, out=None, scale_out=None):
    """Merge E4M3 weight shards [rows_j, K] with per-tensor scales (1-element
    f32 tensors) into one [sum rows_j, K] weight requantised to the largest
    scale; returns (merged, scale)."""
    if not shards or len(shards) != len(scales):
        raise ValueError("one scale per shard")
    K = shards[0].shape[1]
    for w, sc in zip(shards, scales):
        _need(w, "shard", _FP8, 2)
        _need(sc, "scale", (torch.float32,))
        if w.shape[1] != K:
            raise ValueError("every shard must have K columns")
    n = len(shards)
    rows = (ctypes.c_int64 * n)(*[int(w.shape[0]) for w in shards])
    ptrs = (ctypes.c_void_p * n)(*[w.data_ptr() for w in shards])
    sptrs = (ctypes.c_void_p * n)(*[sc.data_ptr() for sc in scales])
    total = sum(int(w.shape[0]) for w in shards)
    if out is None:
        out = torch.empty((total, K), dtype=E4M3, device=shards[0].device)
    else:
        _need(out, "out", _FP8, 2)
    if scale_out is None:
        scale_out = torch.empty((1,), dtype=torch.float32, device=shards[0].device)
    _check(lib().fp8_requant_merge(ctypes.cast(ptrs, ctypes.c_void_p), ctypes.cast(sptrs, ctypes.c_void_p),
                                   ctypes.cast(rows, ctypes.c_void_p), n, K, _ptr(out), _ptr(scale_out),
                                   _stream_of(shards[0])), "fp8_requant_merge")
    return out, scale_out


def quant_fp8_per_token(x, out=None, scale_out=None):
    """Dynamic per-token E4M3 quantisation of bf16 x [M,K]; returns (q, s[M])."""
    _need(x, "x", (torch.bfloat16,), 2)
    M, K = x.shape
    if out is None:
        out = torch.empty((M, K), dtype=E4M3, device=x.device)
    else:
        _need(out, "out", _FP8, 2)
    if scale_out is None:
        scale_out = torch.empty((M,), dtype=torch.float32, device=x.device)
    else:
        _need(scale_out, "scale_out", (torch.float32,))
    _check(lib().quant_fp8_per_token(_ptr(x), _ptr(out), _ptr(scale_out), M, K, _stream_of(x)),
           "quant_fp8_per_token")
    return out, scale_out


def w8a16_mm(x, W, scale_b, granularity=None, out=None, flags=0):
    """Weight-only FP8 GEMM: y = bf16((x @ dec(W).T) * scale_b) for bf16 x
    [M,K] and E4M3 W [N,K]; ``granularity`` (0 per-tensor, 1 per-channel)
    defaults from the length of scale_b."""
    _need(x, "x", (torch.bfloat16,), 2)
    _need(W, "W", _FP8, 2)
    _need(scale_b, "scale_b", (torch.float32,))
    M, K = x.shape
    N, Kw = W.shape
    if Kw != K:
        raise ValueError(f"x is [{M},{K}] but W is [{N},{Kw}]")
    if granularity is None:
        granularity = GRAN_PER_CHANNEL if (scale_b.numel() == N and N != 1) else GRAN_PER_TENSOR
    if scale_b.numel() < (N if granularity == GRAN_PER_CHANNEL else 1):
        raise ValueError("scale_b too short for the granularity")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    else:
        _need(out, "out", (torch.bfloat16,), 2)
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must be [{M},{N}]")
    _check(lib().fp8_w8a16_mm_ex(_ptr(x), _ptr(W), _ptr(scale_b), int(granularity), OUT_BF16, M, N, K, _ptr(out),
                                 _stream_of(x), int(flags)), "fp8_w8a16_mm")
    return out


def w8a16_describe_dispatch(M, N, K) -> int:
    return lib().fp8_w8a16_describe_dispatch(M, N, K)


def widen_weight(W, scale_b, granularity=None, out=None):
    """bf16 [N,K] = bf16_rne(fp32(dec(W) * s)), the weight-only large-M branch's weight."""
    _need(W, "W", _FP8, 2)
    _need(scale_b, "scale_b", (torch.float32,))
    N, K = W.shape
    if granularity is None:
        granularity = GRAN_PER_CHANNEL if (scale_b.numel() == N and N != 1) else GRAN_PER_TENSOR
    if out is None:
        out = torch.empty((N, K), dtype=torch.bfloat16, device=W.device)
    else:
        _need(out, "out", (torch.bfloat16,), 2)
    _check(lib().fp8_widen_weight(_ptr(W), _ptr(scale_b), int(granularity), N, K, _ptr(out), _stream_of(W)),
           "fp8_widen_weight")
    return out


def quant_per_token_group(x, out=None, scale_out=None):
    """E4M3 quantisation of bf16 x [M,K] per token and per 128-wide group of K;
    returns (q, s[M, ceil(K/128)])."""
    _need(x, "x", (torch.bfloat16,), 2)
    M, K = x.shape
    KB = (K + BLOCK - 1) // BLOCK
    if out is None:
        out = torch.empty((M, K), dtype=E4M3, device=x.device)
    else:
        _need(out, "out", _FP8, 2)
    if scale_out is None:
        scale_out = torch.empty((M, KB), dtype=torch.float32, device=x.device)
    else:
        _need(scale_out, "scale_out", (torch.float32,))
        if scale_out.numel() < M * KB:
            raise ValueError(f"scale_out needs {M * KB} elements")
    _check(lib().fp8_quant_per_token_group(_ptr(x), _ptr(out), _ptr(scale_out), M, K, _stream_of(x)),
           "fp8_quant_per_token_group")
    return out, scale_out


def quant_weight_block(w, out=None, scale_out=None):
    """E4M3 quantisation of a bf16 weight w [N,K] with one scale per 128 x 128
    block; returns (q, s[ceil(N/128), ceil(K/128)])."""
    _need(w, "w", (torch.bfloat16,), 2)
    N, K = w.shape
    KB, NB = (K + BLOCK - 1) // BLOCK, (N + BLOCK - 1) // BLOCK
    if out is None:
        out = torch.empty((N, K), dtype=E4M3, device=w.device)
    else:
        _need(out, "out", _FP8, 2)
    if scale_out is None:
        scale_out = torch.empty((NB, KB), dtype=torch.float32, device=w.device)
    else:
        _need(scale_out, "scale_out", (torch.float32,))
        if scale_out.numel() < NB * KB:
            raise ValueError(f"scale_out needs {NB * KB} elements")
    _check(lib().fp8_quant_weight_block(_ptr(w), _ptr(out), _ptr(scale_out), N, K, _stream_of(w)),
           "fp8_quant_weight_block")
    return out, scale_out


def quant_fp8_static(x, scale, out=None):
    """Static per-tensor E4M3 quantisation of bf16 x [M,K] by the device scalar `scale`."""
    _need(x, "x", (torch.bfloat16,), 2)
    _need(scale, "scale", (torch.float32,))
    M, K = x.shape
    if out is None:
        out = torch.empty((M, K), dtype=E4M3, device=x.device)
    else:
        _need(out, "out", _FP8, 2)
    _check(lib().quant_fp8_static(_ptr(x), _ptr(scale), _ptr(out), M, K, _stream_of(x)), "quant_fp8_static")
    return out


def describe_dispatch(M, N, K, granularity=0) -> int:
    return lib().fp8_describe_dispatch(M, N, K, granularity)


def decode_ctas(M, N, K) -> int:
    return lib().fp8_decode_ctas(M, N, K)


def _sms(num_sms):
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return int(num_sms)


def decode_split(M, N, K, num_sms=None, granularity=GRAN_PER_CHANNEL) -> int:
    """The decode kernel's mode: S >= 1 CTAs per output tile (clusters, blockwise
    scaling only), 0 for a persistent stream-K grid, -1 if the shape does not
    go to it."""
    return lib().fp8_decode_split_for_sms(M, N, K, int(granularity), _sms(num_sms))


def decode_exact(M, N, K, num_sms=None, granularity=GRAN_PER_CHANNEL) -> int:
    """1 if the shape runs the exact-sum decode kernel, 0 for the TwoSum one,
    -1 if it does not go to the decode kernel."""
    return lib().fp8_decode_exact_for_sms(M, N, K, int(granularity), _sms(num_sms))


def selftest_bounded_wait(timeout_us=1000):
    """Launch the failure-path self-test (a bounded wait nothing completes)."""
    dev = torch.cuda.current_device()
    _check(lib().fp8_selftest_bounded_wait(int(timeout_us), ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)),
           "fp8_selftest_bounded_wait")


def get_device_error(stream=None) -> int:
    """Synchronises the stream and returns the device error word (0 = no error)."""
    word = ctypes.c_uint32(0)
    s = ctypes.c_void_p(stream if stream is not None else torch.cuda.current_stream().cuda_stream)
    st = lib().fp8_get_device_error(s, ctypes.byref(word))
    if st not in (FP8_OK, FP8_ERR_DEVICE):
        raise Fp8Error(st, "fp8_get_device_error")
    return int(word.value)


def clear_device_error():
    _check(lib().fp8_clear_device_error(), "fp8_clear_device_error")
