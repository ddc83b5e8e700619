// api.cu -- the C ABI (include/fp8w8a8.h): argument validation, dispatch,
// TMA descriptor creation, the device error word.  Every entry point validates
// everything before touching the GPU, so the validation paths run (and are
// tested) on a machine without a GPU.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/fp8w8a8.h"
#include "kernels.h"
#include "ptx.cuh"

namespace {

// One error word per device (a module-scope __device__ variable exists once
// per device that loads the library); host code reaches it only through the
// address cudaGetSymbolAddress returns with that device current.
__device__ uint32_t g_error_word;

// fp8_selftest_bounded_wait's kernel: one thread waits, with the kernels'
// bounded wait, on an mbarrier phase that nothing completes; the wait gives up
// after timeout_ns, sets kErrSelfTestWait in the error word and the kernel
// returns normally.
__global__ void bounded_wait_probe_kernel(uint32_t *err, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        const uint32_t b = fp8k::smem_u32(&bar);
        fp8k::mbar_init(b, 1);  // one arrival would complete phase 0; none comes
        fp8k::fence_mbar_init();
        fp8k::mbar_wait_for(b, 0, err, fp8k::kErrSelfTestWait, timeout_ns);
    }
}

constexpr int kMaxDevices = 64;
constexpr int64_t kI32Max = 2147483647;

// Scratch of the split-K kernels' stream-K mode (arrival counters, zero
// between launches, and partial-sum slots), one per stream that runs such a
// launch, allocated on that stream's first one: launches on different streams
// never share it, so they may overlap.
constexpr size_t kWsCounters = size_t(1) << 20;
constexpr int kMaxStreamWorkspaces = 64;

struct StreamWorkspace {
    cudaStream_t stream = nullptr;
    uint32_t *counters = nullptr;
    float *slots = nullptr;
    bool zero_pending = false;  // made during capture: zeroed only inside that graph so far
};

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    uint32_t *err = nullptr;
    StreamWorkspace ws[kMaxStreamWorkspaces];
    int n_ws = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Per-device state, created on first use with the device current.
fp8_status device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FP8_ERR_CUDA;
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_error_word) != cudaSuccess || addr == nullptr) return FP8_ERR_CUDA;
        if (g_encode == nullptr) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return FP8_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        st.num_sms = sms;
        st.err = static_cast<uint32_t *>(addr);
        st.ready = true;
    }
    *out = &st;
    return FP8_OK;
}

// 2-D E4M3 tensor [rows, cols] (cols contiguous) read in boxes of
// box_rows x 128 bytes with the 128-byte swizzle; out-of-range elements read
// as zero.
fp8_status make_tmap_e4m3(CUtensorMap *tm, const void *ptr, int64_t rows, int64_t cols, uint32_t box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {128u, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous) read in boxes of
// box_rows x 64 elements (128 bytes) with the 128-byte swizzle; out-of-range
// elements read as zero.
fp8_status make_tmap_bf16(CUtensorMap *tm, const void *ptr, int64_t rows, int64_t cols, uint32_t box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2u};
    cuuint32_t box[2] = {64u, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA; }

// Rows of the decode kernel's token boxes: the M real rows (the rest of its
// token tiles stays zero).
uint32_t decode_token_box_rows(const fp8k::DecodePlan &plan, int64_t M) {
    return static_cast<uint32_t>(std::min<int64_t>(M, plan.tok_pad));
}

// The stream-K scratch of `stream` on this device (none for cluster plans):
// sized for the largest plan (two CTAs per SM, 32-token tiles, 64-bit parts),
// allocated on the stream's first stream-K launch with its counters zeroed on
// that stream (no device-wide synchronisation).
fp8_status decode_workspace(DeviceState *st, const fp8k::DecodePlan &plan, cudaStream_t stream,
                            fp8k::DecodeWorkspace *ws) {
    ws->counters = nullptr;
    ws->slots = nullptr;
    if (plan.split > 0) return FP8_OK;  // cluster mode: parts summed in distributed shared memory
    if (fp8k::decode_counters_needed(plan) > kWsCounters) return FP8_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    const size_t n_slots = 2u * 2u * 2u * static_cast<size_t>(st->num_sms) * fp8k::kDecodeMaxTokens * fp8k::kDecodeRows;
    if (fp8k::decode_slot_floats(plan) > n_slots) return FP8_ERR_UNSUPPORTED;
    StreamWorkspace *w = nullptr;
    for (int i = 0; i < st->n_ws; ++i)
        if (st->ws[i].stream == stream) w = &st->ws[i];
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return FP8_ERR_CUDA;
    const bool capturing = cap == cudaStreamCaptureStatusActive;
    if (w == nullptr) {
        if (st->n_ws == kMaxStreamWorkspaces) return FP8_ERR_UNSUPPORTED;
        // On a stream that is being captured into a CUDA graph the allocation
        // is made with this thread's capture mode relaxed for the two calls
        // (cudaMalloc enqueues nothing); the counters' zeroing is then part of
        // the graph and runs before the kernel on every replay, and the first
        // call on the stream outside a capture zeroes them once more.
        cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
        if (capturing && cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) return FP8_ERR_CUDA;
        void *c = nullptr, *sl = nullptr;
        cudaError_t e = cudaMalloc(&c, kWsCounters * sizeof(uint32_t));
        if (e == cudaSuccess) {
            e = cudaMalloc(&sl, n_slots * sizeof(float));
            if (e != cudaSuccess) cudaFree(c);
        }
        if (capturing && cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) return FP8_ERR_CUDA;
        if (e != cudaSuccess) return FP8_ERR_CUDA;
        if (cudaMemsetAsync(c, 0, kWsCounters * sizeof(uint32_t), stream) != cudaSuccess) return FP8_ERR_CUDA;
        w = &st->ws[st->n_ws++];
        w->stream = stream;
        w->counters = static_cast<uint32_t *>(c);
        w->slots = static_cast<float *>(sl);
        w->zero_pending = capturing;
    } else if (w->zero_pending && !capturing) {
        if (cudaMemsetAsync(w->counters, 0, kWsCounters * sizeof(uint32_t), stream) != cudaSuccess) return FP8_ERR_CUDA;
        w->zero_pending = false;
    }
    ws->counters = w->counters;
    ws->slots = w->slots;
    return FP8_OK;
}
// ---------------------------------------------------------------- fixed scratch
// Scratch of fp8_scaled_mm_noalloc: arrival counters then partial-sum slots
// of the decode kernel, in one file-scope device array.  The module holds one
// copy per device that loads the library, from load until the process exits.
// In host code the array's name is only a host-side stand-in: its device
// address comes from cudaGetSymbolAddress with the device current.
constexpr size_t kNoAllocCounters = 16384;  // output tiles
// 384 CTAs x 2 slots x 16 tokens x 128 rows of 64-bit exact parts (two floats' room each)
constexpr size_t kNoAllocSlotFloats = 384u * 2u * 16u * 128u * 2u;
constexpr size_t kNoAllocBytes = kNoAllocCounters * sizeof(uint32_t) + kNoAllocSlotFloats * sizeof(float);
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the fixed scratch for the current device (looked up once).
fp8_status noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FP8_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return FP8_OK;
}

// The tile (large-M) kernel's launch for fp8_scaled_mm's arguments (already
// validated); it uses no scratch.
fp8_status tile_gemm(DeviceState *st, const void *A, const void *B, const float *scale_a, const float *scale_b,
                     int granularity, int64_t M, int64_t N, int64_t K, void *out, const fp8k::LaunchOpts &opts,
                     cudaStream_t stream) {
    const fp8k::PrefillPlan plan = fp8k::plan_prefill(M, N, K, st->num_sms, granularity == FP8_GRAN_BLOCK_128);
    if (plan.units > kI32Max) return FP8_ERR_UNSUPPORTED;
    CUtensorMap ta, tb;
    fp8_status s;
    if ((s = make_tmap_e4m3(&ta, A, M, K, fp8k::kPrefillBM)) != FP8_OK) return s;
    if ((s = make_tmap_e4m3(&tb, B, N, K, 128u)) != FP8_OK) return s;  // 128-channel weight boxes
    CUtensorMap to;  // the output, stored in 128-token x 64-channel boxes
    if ((s = make_tmap_bf16(&to, out, M, N, fp8k::kPrefillBM)) != FP8_OK) return s;
    return from_cuda(fp8k::launch_prefill_gemm(ta, tb, to, scale_a, scale_b, granularity, M, N, K, out, st->err,
                                               plan, opts, stream));
}

}  // namespace

extern "C" {

int fp8_library_version(void) { return 100; }

const char *fp8_status_string(int status) {
    switch (status) {
        case FP8_OK: return "FP8_OK";
        case FP8_ERR_INVALID_ARG: return "FP8_ERR_INVALID_ARG: null pointer, bad size or bad enum";
        case FP8_ERR_ALIGNMENT: return "FP8_ERR_ALIGNMENT: pointer not 16-byte aligned or K/N not a multiple of 16/8";
        case FP8_ERR_UNSUPPORTED: return "FP8_ERR_UNSUPPORTED: valid request not implemented (e.g. out_dtype)";
        case FP8_ERR_CUDA: return "FP8_ERR_CUDA: CUDA call or kernel launch failed";
        case FP8_ERR_DEVICE: return "FP8_ERR_DEVICE: a kernel reported an error (bounded wait ran out)";
        case FP8_ERR_TOO_LARGE: return "FP8_ERR_TOO_LARGE: problem exceeds the fixed scratch of fp8_scaled_mm_noalloc";
        default: return "unknown fp8_status";
    }
}

int fp8_describe_dispatch(int64_t M, int64_t N, int64_t K, int granularity) {
    if (M < 0 || N < 1 || K < 1 || M > kI32Max || N > kI32Max || K > kI32Max) return -1;
    if (granularity < 0 || granularity > FP8_GRAN_BLOCK_128) return -1;
    if (M == 0) return FP8_KERNEL_NONE;
    if (M >= fp8k::kPrefillMinM) return FP8_KERNEL_PREFILL;
    // the decode kernel's exact k-block sum holds fewer than 2^20 k-blocks
    if (granularity != FP8_GRAN_BLOCK_128 && (K + fp8k::kBlockK - 1) / fp8k::kBlockK >= fp8k::kExactMaxKb)
        return FP8_KERNEL_PREFILL;
    return FP8_KERNEL_DECODE_SPLITK;
}

int fp8_decode_ctas_for_sms(int64_t M, int64_t N, int64_t K, int granularity, int num_sms) {
    if (fp8_describe_dispatch(M, N, K, granularity) != FP8_KERNEL_DECODE_SPLITK || num_sms < 1) return -1;
    return fp8k::plan_decode(M, N, K, num_sms, granularity == FP8_GRAN_BLOCK_128).ctas;
}

int fp8_decode_split_for_sms(int64_t M, int64_t N, int64_t K, int granularity, int num_sms) {
    if (fp8_describe_dispatch(M, N, K, granularity) != FP8_KERNEL_DECODE_SPLITK || num_sms < 1) return -1;
    return fp8k::plan_decode(M, N, K, num_sms, granularity == FP8_GRAN_BLOCK_128).split;
}

int fp8_decode_exact_for_sms(int64_t M, int64_t N, int64_t K, int granularity, int num_sms) {
    if (fp8_describe_dispatch(M, N, K, granularity) != FP8_KERNEL_DECODE_SPLITK || num_sms < 1) return -1;
    return fp8k::plan_decode(M, N, K, num_sms, granularity == FP8_GRAN_BLOCK_128).exact;
}

int fp8_decode_ctas(int64_t M, int64_t N, int64_t K) {
    DeviceState *st = nullptr;
    if (fp8_describe_dispatch(M, N, K, 0) != FP8_KERNEL_DECODE_SPLITK) return -1;
    if (device_state(&st) != FP8_OK) return -1;
    return fp8k::plan_decode(M, N, K, st->num_sms).ctas;
}

fp8_status fp8_scaled_mm_ex(const void *A, const void *B, const float *scale_a, const float *scale_b,
                            int granularity, int out_dtype, int64_t M, int64_t N, int64_t K, void *out, void *stream,
                            unsigned flags) {
    if (M < 0 || N < 1 || K < 1 || M > kI32Max || N > kI32Max || K > kI32Max) return FP8_ERR_INVALID_ARG;
    if (granularity < 0 || granularity > FP8_GRAN_BLOCK_128) return FP8_ERR_INVALID_ARG;
    if (flags & ~static_cast<unsigned>(FP8_FLAG_WEIGHTS_STATIC | FP8_FLAG_NO_PDL)) return FP8_ERR_INVALID_ARG;
    if (out_dtype != FP8_OUT_BF16) return FP8_ERR_UNSUPPORTED;
    if (M == 0) return FP8_OK;
    if (!A || !B || !scale_a || !scale_b || !out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(out) || !aligned4(scale_a) || !aligned4(scale_b))
        return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0 || N % 8 != 0) return FP8_ERR_ALIGNMENT;

    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    fp8k::LaunchOpts opts;
    opts.pdl = (flags & FP8_FLAG_NO_PDL) == 0;
    opts.weights_static = (flags & FP8_FLAG_WEIGHTS_STATIC) != 0;
    if (fp8_describe_dispatch(M, N, K, granularity) == FP8_KERNEL_PREFILL)
        return tile_gemm(st, A, B, scale_a, scale_b, granularity, M, N, K, out, opts, static_cast<cudaStream_t>(stream));
    const fp8k::DecodePlan plan = fp8k::plan_decode(M, N, K, st->num_sms, granularity == FP8_GRAN_BLOCK_128);
    fp8k::DecodeWorkspace ws;
    if ((s = decode_workspace(st, plan, static_cast<cudaStream_t>(stream), &ws)) != FP8_OK) return s;
    CUtensorMap tw, ta;
    if ((s = make_tmap_e4m3(&tw, B, N, K, fp8k::kDecodeRows)) != FP8_OK) return s;
    if ((s = make_tmap_e4m3(&ta, A, M, K, decode_token_box_rows(plan, M))) != FP8_OK) return s;
    return from_cuda(fp8k::launch_decode_gemm(tw, ta, scale_a, scale_b, granularity, M, N, K, out, st->err, plan,
                                              ws, opts, static_cast<cudaStream_t>(stream)));
}

fp8_status fp8_scaled_mm(const void *A, const void *B, const float *scale_a, const float *scale_b, int granularity,
                         int out_dtype, int64_t M, int64_t N, int64_t K, void *out, void *stream) {
    return fp8_scaled_mm_ex(A, B, scale_a, scale_b, granularity, out_dtype, M, N, K, out, stream, 0u);
}

fp8_status fp8_scaled_mm_noalloc(const void *A, const void *B, const float *scale_a, const float *scale_b,
                                 int granularity, int out_dtype, int64_t M, int64_t N, int64_t K, void *out,
                                 void *stream) {
    if (M < 0 || N < 1 || K < 1 || M > kI32Max || N > kI32Max || K > kI32Max) return FP8_ERR_INVALID_ARG;
    if (granularity < 0 || granularity > FP8_GRAN_BLOCK_128) return FP8_ERR_INVALID_ARG;
    if (out_dtype != FP8_OUT_BF16) return FP8_ERR_UNSUPPORTED;
    if (M == 0) return FP8_OK;
    if (!A || !B || !scale_a || !scale_b || !out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(out) || !aligned4(scale_a) || !aligned4(scale_b))
        return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0 || N % 8 != 0) return FP8_ERR_ALIGNMENT;
    if (M > 16) return FP8_ERR_TOO_LARGE;

    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // a K too long for the decode kernel's exact sums: the tile kernel, which
    // uses no scratch
    if (fp8_describe_dispatch(M, N, K, granularity) == FP8_KERNEL_PREFILL)
        return tile_gemm(st, A, B, scale_a, scale_b, granularity, M, N, K, out, fp8k::LaunchOpts{}, cs);
    const fp8k::DecodePlan plan = fp8k::plan_decode(M, N, K, st->num_sms, granularity == FP8_GRAN_BLOCK_128);
    const size_t n_counters = fp8k::decode_counters_needed(plan);
    if (n_counters > kNoAllocCounters || fp8k::decode_slot_floats(plan) > kNoAllocSlotFloats)
        return FP8_ERR_TOO_LARGE;
    void *scratch = nullptr;
    if ((s = noalloc_scratch(&scratch)) != FP8_OK) return s;
    fp8k::DecodeWorkspace ws;
    ws.counters = static_cast<uint32_t *>(scratch);
    ws.slots = reinterpret_cast<float *>(static_cast<unsigned char *>(scratch) + kNoAllocCounters * sizeof(uint32_t));
    // the counters must start at zero; the previous call may have been cut short
    if (n_counters > 0 && cudaMemsetAsync(ws.counters, 0, n_counters * sizeof(uint32_t), cs) != cudaSuccess)
        return FP8_ERR_CUDA;
    CUtensorMap tw, ta;
    if ((s = make_tmap_e4m3(&tw, B, N, K, fp8k::kDecodeRows)) != FP8_OK) return s;
    if ((s = make_tmap_e4m3(&ta, A, M, K, decode_token_box_rows(plan, M))) != FP8_OK) return s;
    return from_cuda(fp8k::launch_decode_gemm(tw, ta, scale_a, scale_b, granularity, M, N, K, out, st->err, plan,
                                              ws, fp8k::LaunchOpts{}, cs));
}

fp8_status fp8_rmsnorm_quant_scaled_mm(const void *x, const void *gamma, float eps, const float *scale_a,
                                       const void *B, const float *scale_b, int granularity, int out_dtype, int64_t M,
                                       int64_t N, int64_t K, void *a_out, void *out, void *stream, unsigned flags) {
    if (M < 0 || N < 1 || K < 1 || M > kI32Max || N > kI32Max || K > 65536) return FP8_ERR_INVALID_ARG;
    if (granularity != FP8_GRAN_PER_TENSOR && granularity != FP8_GRAN_PER_CHANNEL) return FP8_ERR_INVALID_ARG;
    if (flags & ~static_cast<unsigned>(FP8_FLAG_WEIGHTS_STATIC | FP8_FLAG_NO_PDL)) return FP8_ERR_INVALID_ARG;
    if (out_dtype != FP8_OUT_BF16) return FP8_ERR_UNSUPPORTED;
    if (M == 0) return FP8_OK;
    if (!x || !gamma || !scale_a || !B || !scale_b || !a_out || !out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(a_out) || !aligned16(B) || !aligned16(out) ||
        !aligned4(scale_a) || !aligned4(scale_b))
        return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0 || N % 8 != 0) return FP8_ERR_ALIGNMENT;
    // Every argument is valid for both calls, so the first cannot succeed and
    // the second then fail validation.
    fp8_status s = rmsnorm_quant_fp8(x, gamma, eps, scale_a, a_out, M, K, stream);
    if (s != FP8_OK) return s;
    return fp8_scaled_mm_ex(a_out, B, scale_a, scale_b, granularity, out_dtype, M, N, K, out, stream, flags);
}

fp8_status rmsnorm_quant_fp8(const void *x, const void *gamma, float eps, const float *scale, void *out, int64_t M,
                             int64_t K, void *stream) {
    if (M < 0 || M > kI32Max || K < 1 || K > 65536) return FP8_ERR_INVALID_ARG;
    if (M == 0) return FP8_OK;
    if (!x || !gamma || !scale || !out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(out) || !aligned4(scale)) return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0) return FP8_ERR_ALIGNMENT;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    return from_cuda(
        fp8k::launch_rmsnorm_quant(x, gamma, eps, scale, out, M, K, st->err, static_cast<cudaStream_t>(stream),
                                   st->num_sms, fp8k::LaunchOpts{}));
}

fp8_status fp8_add_rmsnorm_quant(const void *x, void *residual, const void *gamma, float eps, const float *scale,
                                 void *out, int64_t M, int64_t K, void *stream) {
    if (M < 0 || M > kI32Max || K < 1 || K > 65536) return FP8_ERR_INVALID_ARG;
    if (M == 0) return FP8_OK;
    if (!x || !residual || !gamma || !scale || !out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(residual) || !aligned16(gamma) || !aligned16(out) || !aligned4(scale))
        return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0) return FP8_ERR_ALIGNMENT;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    return from_cuda(fp8k::launch_rmsnorm_quant(x, gamma, eps, scale, out, M, K, st->err,
                                                static_cast<cudaStream_t>(stream), st->num_sms, fp8k::LaunchOpts{},
                                                residual));
}

fp8_status fp8_silu_mul_quant_per_token(const void *gate_up, void *out, float *scale_out, int64_t M, int64_t I,
                                        void *stream) {
    if (M < 0 || M > kI32Max || I < 1 || I > 131072) return FP8_ERR_INVALID_ARG;
    if (M == 0) return FP8_OK;
    if (!gate_up || !out || !scale_out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(gate_up) || !aligned16(out) || !aligned4(scale_out)) return FP8_ERR_ALIGNMENT;
    if (I % 16 != 0) return FP8_ERR_ALIGNMENT;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    return from_cuda(fp8k::launch_silu_mul_quant(gate_up, out, scale_out, M, I, st->err,
                                                 static_cast<cudaStream_t>(stream), st->num_sms, fp8k::LaunchOpts{}));
}

fp8_status fp8_requant_merge(const void *const *shards, const float *const *scales, const int64_t *rows,
                             int n_shards, int64_t K, void *out, float *scale_out, void *stream) {
    if (!shards || !scales || !rows || !out || !scale_out) return FP8_ERR_INVALID_ARG;
    if (n_shards < 1 || n_shards > fp8k::kMaxMergeShards || K < 1 || K > kI32Max) return FP8_ERR_INVALID_ARG;
    if (K % 16 != 0) return FP8_ERR_ALIGNMENT;
    if (!aligned16(out) || !aligned4(scale_out)) return FP8_ERR_ALIGNMENT;
    fp8k::MergeArgs a{};
    int64_t total_rows = 0;
    for (int j = 0; j < n_shards; ++j) {
        if (rows[j] < 0 || rows[j] > kI32Max) return FP8_ERR_INVALID_ARG;
        if (rows[j] > 0 && (!shards[j] || !scales[j])) return FP8_ERR_INVALID_ARG;
        if (!scales[j]) return FP8_ERR_INVALID_ARG;
        if ((shards[j] && !aligned16(shards[j])) || !aligned4(scales[j])) return FP8_ERR_ALIGNMENT;
        total_rows += rows[j];
        a.src[j] = static_cast<const uint4 *>(shards[j]);
        a.scale[j] = scales[j];
        a.end16[j] = total_rows * K / 16;
    }
    if (total_rows > kI32Max) return FP8_ERR_INVALID_ARG;
    a.n = n_shards;
    a.out = static_cast<uint4 *>(out);
    a.scale_out = scale_out;
    a.n16 = total_rows * K / 16;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    return from_cuda(fp8k::launch_requant_merge(a, static_cast<cudaStream_t>(stream), st->num_sms, fp8k::LaunchOpts{}));
}

fp8_status quant_fp8_per_token(const void *x, void *out, float *scale_out, int64_t M, int64_t K, void *stream) {
    if (M < 0 || M > kI32Max || K < 1 || K > (int64_t(1) << 30)) return FP8_ERR_INVALID_ARG;
    if (M == 0) return FP8_OK;
    if (!x || !out || !scale_out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned4(scale_out)) return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0) return FP8_ERR_ALIGNMENT;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    return from_cuda(fp8k::launch_quant_per_token(x, out, scale_out, M, K, st->err, static_cast<cudaStream_t>(stream),
                                                  st->num_sms, fp8k::LaunchOpts{}));
}

int fp8_w8a16_describe_dispatch(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 1 || K < 1 || M > kI32Max || N > kI32Max || K > kI32Max) return -1;
    if (M == 0) return FP8_KERNEL_NONE;
    if (fp8k::w8a16_gemv_fits(M, K)) return FP8_KERNEL_W16_GEMV;
    return M >= fp8k::kPrefillMinM ? FP8_KERNEL_W16_DENSE : FP8_KERNEL_W16_DECODE;
}

fp8_status fp8_widen_weight(const void *W, const float *scale_b, int granularity, int64_t N, int64_t K, void *out,
                            void *stream) {
    if (N < 0 || N > kI32Max || K < 1 || K > kI32Max) return FP8_ERR_INVALID_ARG;
    if (granularity != FP8_GRAN_PER_TENSOR && granularity != FP8_GRAN_PER_CHANNEL) return FP8_ERR_INVALID_ARG;
    if (N == 0) return FP8_OK;
    if (!W || !scale_b || !out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(out) || !aligned4(scale_b)) return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0) return FP8_ERR_ALIGNMENT;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    return from_cuda(fp8k::launch_widen_weight(W, scale_b, granularity == FP8_GRAN_PER_CHANNEL ? 1 : 0, N, K, out,
                                               static_cast<cudaStream_t>(stream), st->num_sms, fp8k::LaunchOpts{}));
}

fp8_status fp8_w8a16_mm_ex(const void *x, const void *W, const float *scale_b, int granularity, int out_dtype,
                           int64_t M, int64_t N, int64_t K, void *out, void *stream, unsigned flags) {
    if (M < 0 || N < 1 || K < 1 || M > kI32Max || N > kI32Max || K > kI32Max) return FP8_ERR_INVALID_ARG;
    if (granularity != FP8_GRAN_PER_TENSOR && granularity != FP8_GRAN_PER_CHANNEL) return FP8_ERR_INVALID_ARG;
    if (flags & ~static_cast<unsigned>(FP8_FLAG_WEIGHTS_STATIC | FP8_FLAG_NO_PDL)) return FP8_ERR_INVALID_ARG;
    if (out_dtype != FP8_OUT_BF16) return FP8_ERR_UNSUPPORTED;
    if (M == 0) return FP8_OK;
    if (!x || !W || !scale_b || !out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W) || !aligned16(out) || !aligned4(scale_b)) return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0 || N % 8 != 0) return FP8_ERR_ALIGNMENT;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    fp8k::LaunchOpts opts;
    opts.pdl = (flags & FP8_FLAG_NO_PDL) == 0;
    opts.weights_static = (flags & FP8_FLAG_WEIGHTS_STATIC) != 0;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int per_channel = granularity == FP8_GRAN_PER_CHANNEL ? 1 : 0;
    const int kind = fp8_w8a16_describe_dispatch(M, N, K);
    if (kind == FP8_KERNEL_W16_GEMV) {
        // One to four tokens: the CUDA-core GEMV (whole weight rows per warp,
        // no split of K, no scratch).
        return from_cuda(
            fp8k::launch_w8a16_gemv(W, x, scale_b, per_channel, M, N, K, out, st->err, st->num_sms, opts, cs));
    }
    if (kind == FP8_KERNEL_W16_DENSE) {
        // Large M: the tile kernel, widening each E4M3 weight box to bf16 on
        // chip (exact: every E4M3 value is a bf16 value) for dense bf16 MMAs,
        // the weight scale applied to the fp32 accumulator before the bf16
        // rounding; no widened copy of the weight, no scratch.
        const fp8k::W16TilePlan plan = fp8k::plan_w8a16_tile(M, N, K, st->num_sms);
        if (plan.units > kI32Max) return FP8_ERR_UNSUPPORTED;
        CUtensorMap tw, tx;
        if ((s = make_tmap_e4m3(&tw, W, N, K, fp8k::kDecodeRows)) != FP8_OK) return s;
        if ((s = make_tmap_bf16(&tx, x, M, K, static_cast<uint32_t>(fp8k::kW16TileTokens))) != FP8_OK) return s;
        return from_cuda(fp8k::launch_w8a16_tile(tw, tx, scale_b, per_channel, M, N, out, st->err, plan, opts, cs));
    }
    const fp8k::DecodePlan plan = fp8k::plan_w8a16(M, N, K, st->num_sms);
    fp8k::DecodeWorkspace ws;
    if ((s = decode_workspace(st, plan, cs, &ws)) != FP8_OK) return s;
    CUtensorMap tw, tx;
    if ((s = make_tmap_e4m3(&tw, W, N, K, fp8k::kDecodeRows)) != FP8_OK) return s;
    if ((s = make_tmap_bf16(&tx, x, M, K, static_cast<uint32_t>(plan.tok_pad))) != FP8_OK) return s;
    return from_cuda(fp8k::launch_w8a16_gemm(tw, tx, scale_b, per_channel, M, N, K, out, st->err, plan, ws, opts, cs));
}

fp8_status fp8_w8a16_mm(const void *x, const void *W, const float *scale_b, int granularity, int out_dtype, int64_t M,
                        int64_t N, int64_t K, void *out, void *stream) {
    return fp8_w8a16_mm_ex(x, W, scale_b, granularity, out_dtype, M, N, K, out, stream, 0u);
}

fp8_status fp8_quant_per_token_group(const void *x, void *out, float *scale_out, int64_t M, int64_t K, void *stream) {
    if (M < 0 || M > kI32Max || K < 1 || K > (int64_t(1) << 30)) return FP8_ERR_INVALID_ARG;
    if (M == 0) return FP8_OK;
    if (!x || !out || !scale_out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned4(scale_out)) return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0) return FP8_ERR_ALIGNMENT;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    return from_cuda(fp8k::launch_quant_per_token_group(x, out, scale_out, M, K, static_cast<cudaStream_t>(stream),
                                                        fp8k::LaunchOpts{}));
}

fp8_status fp8_quant_weight_block(const void *w, void *out, float *scale_out, int64_t N, int64_t K, void *stream) {
    if (N < 0 || N > kI32Max || K < 1 || K > (int64_t(1) << 30)) return FP8_ERR_INVALID_ARG;
    if (N == 0) return FP8_OK;
    if (!w || !out || !scale_out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(out) || !aligned4(scale_out)) return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0) return FP8_ERR_ALIGNMENT;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    return from_cuda(fp8k::launch_quant_weight_block(w, out, scale_out, N, K, static_cast<cudaStream_t>(stream),
                                                     fp8k::LaunchOpts{}));
}

fp8_status quant_fp8_static(const void *x, const float *scale, void *out, int64_t M, int64_t K, void *stream) {
    if (M < 0 || M > kI32Max || K < 1 || K > kI32Max) return FP8_ERR_INVALID_ARG;
    if (M == 0) return FP8_OK;
    if (!x || !scale || !out) return FP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned4(scale)) return FP8_ERR_ALIGNMENT;
    if (K % 16 != 0) return FP8_ERR_ALIGNMENT;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    return from_cuda(
        fp8k::launch_quant_static(x, scale, out, M, K, st->err, static_cast<cudaStream_t>(stream), st->num_sms,
                                  fp8k::LaunchOpts{}));
}

fp8_status fp8_set_device(int device) {
    if (device < 0 || device >= kMaxDevices) return FP8_ERR_INVALID_ARG;
    return cudaSetDevice(device) == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status fp8_get_device_error(void *stream, uint32_t *word) {
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8_ERR_CUDA;
    uint32_t w = 0;
    if (cudaMemcpy(&w, st->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return FP8_ERR_CUDA;
    if (word) *word = w;
    return w ? FP8_ERR_DEVICE : FP8_OK;
}

fp8_status fp8_selftest_bounded_wait(uint32_t timeout_us, void *stream) {
    if (timeout_us < 1 || timeout_us > 2000000u) return FP8_ERR_INVALID_ARG;
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    bounded_wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        st->err, static_cast<unsigned long long>(timeout_us) * 1000ull);
    return from_cuda(cudaGetLastError());
}

fp8_status fp8_clear_device_error(void) {
    DeviceState *st = nullptr;
    fp8_status s = device_state(&st);
    if (s != FP8_OK) return s;
    if (cudaMemset(st->err, 0, sizeof(uint32_t)) != cudaSuccess) return FP8_ERR_CUDA;
    // a kernel that gave up may have left arrival counters behind
    {
        std::lock_guard<std::mutex> lock(g_mu);
        for (int i = 0; i < st->n_ws; ++i)
            if (cudaMemset(st->ws[i].counters, 0, kWsCounters * sizeof(uint32_t)) != cudaSuccess) return FP8_ERR_CUDA;
    }
    return cudaDeviceSynchronize() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // extern "C"
