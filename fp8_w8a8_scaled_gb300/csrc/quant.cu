// quant.cu -- the activation producers of the FP8 W8A8 linear layer:
//   * quant_fp8_static     q = e4m3(x / s)                      (QuantFp8Static)
//   * quant_fp8_per_token  s_m = amax_m / 448, q = e4m3(x / s_m)
//   * rmsnorm_quant_fp8    q = e4m3(bf16(x * r * gamma) / s), r = 1/sqrt(mean x^2 + eps)
// Sources: "We emit F32 where vLLM emits bf16 ..." (vllm.cpp #417), section
// "Ranked follow-ons from the same audit" (QuantFp8Static, the fused RMSNorm ->
// fp8 quant, "quantise once"); "The FP8 tower's cuBLASLt default rests on a
// false premise ..." (vllm.cpp #252), "What is owed" item 2 (per-tensor vs
// per-token granularity).
//
// All three are HBM-bound streaming kernels (2 bytes read + 1 byte written per
// element): 128-bit coalesced loads of 8 bf16, 64-bit stores of 8 E4M3 codes.
// The per-row kernels keep the whole row in registers so x is read once.
//
// Rounding is pinned so the bytes match the CPU definition exactly: IEEE
// binary32 division (__fdiv_rn, never a reciprocal multiply), separate
// binary32 multiplies (no FMA), the sum of squares formed exactly and rounded
// once to binary32, binary32 mean / sqrt / reciprocal, round-to-nearest-even
// bf16, and the hardware's saturating round-to-nearest-even E4M3
// conversion (cvt.rn.satfinite.e4m3x2.f32).  Every kernel is launched with
// programmatic dependent launch and waits for its predecessor before reading.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "norm_row.cuh"
#include "ptx.cuh"

namespace fp8k {
namespace {

using norm::bf16_hi;
using norm::bf16_lo;
using norm::e4m3x2;
using norm::ld_stream;


// Eight bf16 (one 16-byte vector) divided by s -> eight E4M3 codes.
__device__ __forceinline__ uint2 quant8(const uint4 v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = e4m3x2(__fdiv_rn(bf16_lo(w[i]), s), __fdiv_rn(bf16_hi(w[i]), s));
    return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// max |x| over eight bf16; NaN entries are ignored (fmaxf semantics).
__device__ __forceinline__ float absmax8(const uint4 v, float m) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, __uint_as_float((w[i] << 16) & 0x7FFFFFFFu));
        m = fmaxf(m, __uint_as_float(w[i] & 0x7FFF0000u));
    }
    return m;
}

__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    return red[0];
}

// ------------------------------------------------------------- static quant --

__global__ void __launch_bounds__(256) quant_static_kernel(const uint4 *__restrict__ x, const float *__restrict__ scale,
                                                           uint4 *__restrict__ out, int64_t n16) {
    grid_dependency_wait();
    grid_launch_dependents();
    const float s = __ldg(scale);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
        const uint4 a = ld_stream(x + 2 * i);
        const uint4 b = ld_stream(x + 2 * i + 1);
        const uint2 qa = quant8(a, s), qb = quant8(b, s);
        out[i] = make_uint4(qa.x, qa.y, qb.x, qb.y);
    }
}

// ---------------------------------------------------------- per-token quant --

// One CTA per row, the row held in registers: blockDim.x threads (up to 1024)
// x V vectors of 8, as few vectors per thread as the row allows so that every
// thread's serial chain is short.
template <int V>
__global__ void __launch_bounds__(1024) quant_per_token_kernel(const uint4 *__restrict__ x, uint2 *__restrict__ out,
                                                               float *__restrict__ scale_out, int nvec) {
    const int T = static_cast<int>(blockDim.x);
    __shared__ float red[32];
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t row = blockIdx.x;
    const uint4 *xr = x + row * nvec;
    uint2 *orow = out + row * nvec;
    uint4 v[V];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = threadIdx.x + j * T;
        if (idx < nvec) {
            v[j] = ld_stream(xr + idx);
            amax = absmax8(v[j], amax);
        }
    }
    amax = block_max(amax, red);
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    if (threadIdx.x == 0) scale_out[row] = s;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = threadIdx.x + j * T;
        if (idx < nvec) orow[idx] = quant8(v[j], s);
    }
}

// Rows too long for registers: one pass for the max, one to quantise.
__global__ void __launch_bounds__(512) quant_per_token_long_kernel(const uint4 *__restrict__ x,
                                                                   uint2 *__restrict__ out,
                                                                   float *__restrict__ scale_out, int64_t nvec) {
    __shared__ float red[32];
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t row = blockIdx.x;
    const uint4 *xr = x + row * nvec;
    uint2 *orow = out + row * nvec;
    float amax = 0.0f;
    for (int64_t i = threadIdx.x; i < nvec; i += 512) amax = absmax8(__ldg(xr + i), amax);
    amax = block_max(amax, red);
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    if (threadIdx.x == 0) scale_out[row] = s;
    for (int64_t i = threadIdx.x; i < nvec; i += 512) orow[i] = quant8(__ldg(xr + i), s);
}

// ------------------------------------------- SiLU(gate) * up -> per-token quant --

// exp in binary32: Cody and Waite's argument reduction (W. J. Cody and W.
// Waite, "Software Manual for the Elementary Functions", 1980) --
// n = rint(y log2 e), r = (y - n C1) - n C2 with C1 + C2 = ln 2 and C1 short
// enough that n C1 is exact -- then e^r by its Taylor series to degree 7 in
// Horner form, times 2^n.  Every step is one IEEE binary32 operation (no
// fused multiply-add), so the result is a fixed function of y; it is within a
// few units in the last place of exp.  y < -87 gives 0 and y > 88 gives +inf
// (every 2^n is then a normal number), NaN gives NaN.
__device__ __forceinline__ float exp_f32(float y) {
    if (y != y) return y;
    if (y < -87.0f) return 0.0f;
    if (y > 88.0f) return __int_as_float(0x7F800000);
    const float kLog2e = 1.44269504088896340736f;   // log2(e) rounded to binary32
    const float kLn2Hi = 0.693145751953125f;        // 0x3F317200: ln 2 to 16 bits
    const float kLn2Lo = 1.428606765330187045e-06f; // ln 2 - kLn2Hi, rounded
    const float n = rintf(__fmul_rn(y, kLog2e));
    const float r = __fsub_rn(__fsub_rn(y, __fmul_rn(n, kLn2Hi)), __fmul_rn(n, kLn2Lo));
    float p = 1.0f / 5040.0f;
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 720.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 120.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 24.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 6.0f);
    p = __fadd_rn(__fmul_rn(p, r), 0.5f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    const float two_n = __int_as_float((static_cast<int>(n) + 127) << 23);
    return __fmul_rn(p, two_n);
}

// bf16( silu(g) * u ) with silu(g) = g / (1 + exp(-g)), binary32 throughout.
__device__ __forceinline__ uint32_t silu_mul_bf16(float g, float u) {
    const float s = __fdiv_rn(g, __fadd_rn(1.0f, exp_f32(-g)));
    return __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(s, u)));
}

__device__ __forceinline__ uint4 silu_mul8(const uint4 g, const uint4 u) {
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
    uint32_t a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        a[i] = silu_mul_bf16(bf16_lo(gw[i]), bf16_lo(uw[i])) | (silu_mul_bf16(bf16_hi(gw[i]), bf16_hi(uw[i])) << 16);
    return make_uint4(a[0], a[1], a[2], a[3]);
}

// One CTA per row of [gate (I) | up (I)]: a = bf16(silu(gate) * up) held in
// registers, then the per-token quantisation of a (the same arithmetic as
// quant_per_token_kernel on a materialised a).
template <int V>
__global__ void __launch_bounds__(1024) silu_mul_quant_kernel(const uint4 *__restrict__ gate_up, uint2 *__restrict__ out,
                                                              float *__restrict__ scale_out, int nvec) {
    const int T = static_cast<int>(blockDim.x);
    __shared__ float red[32];
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t row = blockIdx.x;
    const uint4 *gr = gate_up + row * 2 * nvec;
    const uint4 *ur = gr + nvec;
    uint2 *orow = out + row * nvec;
    uint4 a[V];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = threadIdx.x + j * T;
        if (idx < nvec) {
            a[j] = silu_mul8(ld_stream(gr + idx), ld_stream(ur + idx));
            amax = absmax8(a[j], amax);
        }
    }
    amax = block_max(amax, red);
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    if (threadIdx.x == 0) scale_out[row] = s;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = threadIdx.x + j * T;
        if (idx < nvec) orow[idx] = quant8(a[j], s);
    }
}

// Small M: a row of [gate | up] split over a cluster of CS CTAs (one CTA per
// SM for M rows would leave almost every SM idle and give each thread many
// exp / divisions in series).  Each CTA takes a contiguous chunk of the row;
// the row's amax is the max of the CTAs' maxima, exchanged through
// distributed shared memory between two cluster barriers (max is exact and
// order-free, so every CTA gets the same scale and the bytes equal the
// one-CTA kernel's).
template <int V, int CS>
__global__ void __launch_bounds__(256) silu_mul_quant_cluster_kernel(const uint4 *__restrict__ gate_up,
                                                                     uint2 *__restrict__ out,
                                                                     float *__restrict__ scale_out, int nvec) {
    __shared__ float red[32];
    __shared__ float s_amax;
    grid_dependency_wait();
    grid_launch_dependents();
    const uint32_t rank = cluster_ctarank();
    const int64_t row = blockIdx.x / CS;
    const int chunk = (nvec + CS - 1) / CS;
    const int v0 = static_cast<int>(rank) * chunk, v1 = min(nvec, v0 + chunk);
    const uint4 *gr = gate_up + row * 2 * nvec;
    const uint4 *ur = gr + nvec;
    uint2 *orow = out + row * nvec;
    const int T = static_cast<int>(blockDim.x);
    uint4 a[V];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = v0 + static_cast<int>(threadIdx.x) + j * T;
        if (idx < v1) {
            a[j] = silu_mul8(ld_stream(gr + idx), ld_stream(ur + idx));
            amax = absmax8(a[j], amax);
        }
    }
    amax = block_max(amax, red);
    if (threadIdx.x == 0) s_amax = amax;
    cluster_sync();
    float m = 0.0f;
    const uint32_t my = smem_u32(&s_amax);
#pragma unroll
    for (int r = 0; r < CS; ++r) m = fmaxf(m, ld_cluster_f32(map_to_rank(my, static_cast<uint32_t>(r))));
    cluster_sync();  // no CTA leaves while another may still read its s_amax
    const float s = (m == 0.0f) ? 1.0f : __fdiv_rn(m, 448.0f);
    if (rank == 0 && threadIdx.x == 0) scale_out[row] = s;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = v0 + static_cast<int>(threadIdx.x) + j * T;
        if (idx < v1) orow[idx] = quant8(a[j], s);
    }
}

// ------------------------------------------------------ blockwise quantisers --

// Per-token-group quantisation: each 128-wide group of a row is quantised on
// its own (s = amax/448, 1.0 for an all-zero group).  A half-warp owns a group
// (16 lanes x one 16-byte vector of 8 bf16), so a warp does two groups and a
// CTA of 8 warps sixteen groups of one row; the group max is a 16-lane
// shuffle reduction.  Work item b (grid-stride) is row b / chunks, groups
// 16 * (b % chunks) onwards.
__global__ void __launch_bounds__(256) quant_per_token_group_kernel(const uint4 *__restrict__ x,
                                                                    uint2 *__restrict__ out,
                                                                    float *__restrict__ scale_out, int64_t items,
                                                                    int chunks, int nvec, int KB) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int lane = static_cast<int>(threadIdx.x & 31);
    for (int64_t b = blockIdx.x; b < items; b += gridDim.x) {
        const int64_t row = b / chunks;
        const int grp = static_cast<int>(b - row * chunks) * 16 + static_cast<int>(threadIdx.x >> 4);
        const int vec = grp * 16 + (lane & 15);
        const bool ok = grp < KB && vec < nvec;
        uint4 v = make_uint4(0, 0, 0, 0);
        float amax = 0.0f;
        if (ok) {
            v = ld_stream(x + row * nvec + vec);
            amax = absmax8(v, 0.0f);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
        if (ok) {
            out[row * nvec + vec] = quant8(v, s);
            if ((lane & 15) == 0) scale_out[row * KB + grp] = s;
        }
    }
}

// Per-block weight quantisation: one CTA per 128 x 128 block (2048 vectors of
// 8, eight per thread), s = amax/448 of the block (1.0 if all zero).  Work
// item b (grid-stride) is block row b / KB, k-group b % KB.
__global__ void __launch_bounds__(256) quant_weight_block_kernel(const uint4 *__restrict__ w, uint2 *__restrict__ out,
                                                                 float *__restrict__ scale_out, int64_t N,
                                                                 int64_t items, int nvec, int KB) {
    __shared__ float red[32];
    grid_dependency_wait();
    grid_launch_dependents();
    for (int64_t b = blockIdx.x; b < items; b += gridDim.x) {
        const int64_t nb = b / KB;
        const int g = static_cast<int>(b - nb * KB);
        uint4 v[8];
        bool ok[8];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = static_cast<int>(threadIdx.x) + j * 256;
            const int64_t n = nb * 128 + (t >> 4);
            const int kv = g * 16 + (t & 15);
            ok[j] = n < N && kv < nvec;
            v[j] = make_uint4(0, 0, 0, 0);
            if (ok[j]) {
                v[j] = ld_stream(w + n * nvec + kv);
                amax = absmax8(v[j], amax);
            }
        }
        amax = block_max(amax, red);
        const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
        if (threadIdx.x == 0) scale_out[nb * KB + g] = s;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = static_cast<int>(threadIdx.x) + j * 256;
            const int64_t n = nb * 128 + (t >> 4);
            const int kv = g * 16 + (t & 15);
            if (ok[j]) out[n * nvec + kv] = quant8(v[j], s);
        }
        __syncthreads();  // red[] is reused by the next item
    }
}

// ---------------------------------------------------- shard requantisation --

// Shards [rows_j, K] of E4M3 weights with per-tensor scales s_j, merged into
// one [sum rows_j, K] weight with the scale s_max = max_j s_j: every code
// becomes e4m3( fp32(dec(q) * s_j) / s_max ).  16 codes per thread step (a
// shard's byte size is a multiple of 16, so no vector straddles two shards).
__global__ void __launch_bounds__(256) requant_merge_kernel(const MergeArgs a) {
    grid_dependency_wait();
    grid_launch_dependents();
    float smax = 0.0f;
    for (int j = 0; j < a.n; ++j) smax = fmaxf(smax, __ldg(a.scale[j]));
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.scale_out = smax;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < a.n16; i += stride) {
        int j = 0;
        while (j + 1 < a.n && i >= a.end16[j]) ++j;
        const int64_t start = j ? a.end16[j - 1] : 0;
        const uint4 v = ld_stream(a.src[j] + (i - start));
        const float s_in = __ldg(a.scale[j]);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t packed = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const __nv_fp8x2_storage_t two = static_cast<__nv_fp8x2_storage_t>((w[k] >> (16 * h)) & 0xFFFFu);
                const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
                const float d0 = __half2float(__half(__half_raw{hr.x}));
                const float d1 = __half2float(__half(__half_raw{hr.y}));
                const float v0 = __fdiv_rn(__fmul_rn(d0, s_in), smax);
                const float v1 = __fdiv_rn(__fmul_rn(d1, s_in), smax);
                packed |= e4m3x2(v0, v1) << (16 * h);
            }
            o[k] = packed;
        }
        a.out[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ---------------------------------------------------- fused RMSNorm -> quant --

struct CtaSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// One CTA per row; the row arithmetic (exact sum of squares, binary32 chain)
// is norm::rmsnorm_quant_row.  With R the row is first the residual sum
// bf16(x + resid), which also replaces the residual row.
template <int V, bool R>
__global__ void __launch_bounds__(1024) rmsnorm_quant_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ gamma,
                                                             float eps, const float *__restrict__ scale,
                                                             uint2 *__restrict__ out, int nvec, int K, uint4 *resid) {
    __shared__ norm::RowScratch sc;
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t row = blockIdx.x;
    const float s = __ldg(scale);
    norm::rmsnorm_quant_row<V, (V <= 8), R>(x + row * nvec, gamma, eps, s, out + row * nvec, nvec, K,
                                            norm::Group{static_cast<int>(threadIdx.x), static_cast<int>(blockDim.x)},
                                            &sc, CtaSync{}, R ? resid + row * nvec : nullptr);
}

// Threads per row-CTA for `nvec` vectors at V vectors per thread: a multiple
// of 32, at most 1024.
inline int row_threads(int64_t nvec, int V) {
    const int64_t t = (nvec + V - 1) / V;
    return static_cast<int>(((t + 31) / 32) * 32);
}

template <int V>
cudaError_t launch_rows_pt(const void *x, void *out, float *scale_out, int64_t M, int64_t K, cudaStream_t stream,
                           const LaunchOpts &o) {
    const int64_t nvec = K / 8;
    return launch_with_opts(quant_per_token_kernel<V>, dim3(static_cast<unsigned>(M)), dim3(row_threads(nvec, V)), 0,
                            stream, o, static_cast<const uint4 *>(x), static_cast<uint2 *>(out), scale_out,
                            static_cast<int>(nvec));
}

template <int V>
cudaError_t launch_rows_silu(const void *gate_up, void *out, float *scale_out, int64_t M, int64_t I,
                             cudaStream_t stream, const LaunchOpts &o) {
    const int64_t nvec = I / 8;
    return launch_with_opts(silu_mul_quant_kernel<V>, dim3(static_cast<unsigned>(M)), dim3(row_threads(nvec, V)), 0,
                            stream, o, static_cast<const uint4 *>(gate_up), static_cast<uint2 *>(out), scale_out,
                            static_cast<int>(nvec));
}

template <int V>
cudaError_t launch_rows_rms(const void *x, const void *gamma, float eps, const float *scale, void *out, int64_t M,
                            int64_t K, cudaStream_t stream, const LaunchOpts &o, void *resid) {
    const int64_t nvec = K / 8;
    const dim3 grid(static_cast<unsigned>(M)), block(row_threads(nvec, V));
    if (resid != nullptr)
        return launch_with_opts(rmsnorm_quant_kernel<V, true>, grid, block, 0, stream, o, static_cast<const uint4 *>(x),
                                static_cast<const uint4 *>(gamma), eps, scale, static_cast<uint2 *>(out),
                                static_cast<int>(nvec), static_cast<int>(K), static_cast<uint4 *>(resid));
    return launch_with_opts(rmsnorm_quant_kernel<V, false>, grid, block, 0, stream, o, static_cast<const uint4 *>(x),
                            static_cast<const uint4 *>(gamma), eps, scale, static_cast<uint2 *>(out),
                            static_cast<int>(nvec), static_cast<int>(K), static_cast<uint4 *>(nullptr));
}

}  // namespace

cudaError_t launch_quant_static(const void *x, const float *scale, void *out, int64_t M, int64_t K, uint32_t *err,
                                cudaStream_t stream, int num_sms, const LaunchOpts &o) {
    (void)err;
    const int64_t n16 = M * K / 16;
    int64_t blocks = (n16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_with_opts(quant_static_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, o,
                            static_cast<const uint4 *>(x), scale, static_cast<uint4 *>(out), n16);
}

// Rows per launch from which the per-row kernels trade latency for bytes in
// flight: with few rows, one 16-byte vector per thread makes each row's serial
// chain shortest; with many rows, fewer (and busier) threads per row let more
// rows, and so more loads, be resident on each SM at once.
inline bool many_rows(int64_t M, int num_sms) { return M >= 4 * static_cast<int64_t>(num_sms); }

cudaError_t launch_quant_per_token(const void *x, void *out, float *scale_out, int64_t M, int64_t K, uint32_t *err,
                                   cudaStream_t stream, int num_sms, const LaunchOpts &o) {
    (void)err;
    const int64_t nvec = K / 8;
    if (many_rows(M, num_sms) && nvec <= 1024) return launch_rows_pt<4>(x, out, scale_out, M, K, stream, o);
    if (nvec <= 1024) return launch_rows_pt<1>(x, out, scale_out, M, K, stream, o);
    if (nvec <= 2048) return launch_rows_pt<2>(x, out, scale_out, M, K, stream, o);
    if (nvec <= 4096) return launch_rows_pt<4>(x, out, scale_out, M, K, stream, o);
    if (nvec <= 8192) return launch_rows_pt<8>(x, out, scale_out, M, K, stream, o);
    if (nvec <= 16384) return launch_rows_pt<16>(x, out, scale_out, M, K, stream, o);
    return launch_with_opts(quant_per_token_long_kernel, dim3(static_cast<unsigned>(M)), dim3(512), 0, stream, o,
                            static_cast<const uint4 *>(x), static_cast<uint2 *>(out), scale_out, nvec);
}

cudaError_t launch_quant_per_token_group(const void *x, void *out, float *scale_out, int64_t M, int64_t K,
                                         cudaStream_t stream, const LaunchOpts &o) {
    const int nvec = static_cast<int>(K / 8), KB = static_cast<int>((K + 127) / 128);
    const int chunks = (KB + 15) / 16;
    const int64_t items = M * chunks;
    const unsigned grid = static_cast<unsigned>(items < (int64_t(1) << 20) ? items : (int64_t(1) << 20));
    return launch_with_opts(quant_per_token_group_kernel, dim3(grid), dim3(256), 0, stream, o,
                            static_cast<const uint4 *>(x), static_cast<uint2 *>(out), scale_out, items, chunks, nvec,
                            KB);
}

cudaError_t launch_quant_weight_block(const void *w, void *out, float *scale_out, int64_t N, int64_t K,
                                      cudaStream_t stream, const LaunchOpts &o) {
    const int nvec = static_cast<int>(K / 8), KB = static_cast<int>((K + 127) / 128);
    const int64_t items = ((N + 127) / 128) * KB;
    const unsigned grid = static_cast<unsigned>(items < (int64_t(1) << 20) ? items : (int64_t(1) << 20));
    return launch_with_opts(quant_weight_block_kernel, dim3(grid), dim3(256), 0, stream, o,
                            static_cast<const uint4 *>(w), static_cast<uint2 *>(out), scale_out, N, items, nvec, KB);
}

cudaError_t launch_requant_merge(const MergeArgs &a, cudaStream_t stream, int num_sms, const LaunchOpts &o) {
    int64_t blocks = (a.n16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_with_opts(requant_merge_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, o, a);
}

cudaError_t launch_silu_mul_quant(const void *gate_up, void *out, float *scale_out, int64_t M, int64_t I,
                                  uint32_t *err, cudaStream_t stream, int num_sms, const LaunchOpts &o) {
    (void)err;
    const int64_t nvec = I / 8;
    // Few long rows: 8-CTA clusters per row, 256 threads x up to 4 vectors each.
    constexpr int kCS = 8;
    if (M * kCS <= 2 * static_cast<int64_t>(num_sms) && nvec >= kCS * 256 && nvec <= kCS * 256 * 4) {
        LaunchOpts oc = o;
        oc.cluster_x = kCS;
        return launch_with_opts(silu_mul_quant_cluster_kernel<4, kCS>, dim3(static_cast<unsigned>(M * kCS)), dim3(256),
                                0, stream, oc, static_cast<const uint4 *>(gate_up), static_cast<uint2 *>(out),
                                scale_out, static_cast<int>(nvec));
    }
    if (many_rows(M, num_sms) && nvec <= 1024) return launch_rows_silu<4>(gate_up, out, scale_out, M, I, stream, o);
    if (nvec <= 1024) return launch_rows_silu<1>(gate_up, out, scale_out, M, I, stream, o);
    if (nvec <= 2048) return launch_rows_silu<2>(gate_up, out, scale_out, M, I, stream, o);
    if (nvec <= 4096) return launch_rows_silu<4>(gate_up, out, scale_out, M, I, stream, o);
    if (nvec <= 8192) return launch_rows_silu<8>(gate_up, out, scale_out, M, I, stream, o);
    return launch_rows_silu<16>(gate_up, out, scale_out, M, I, stream, o);
}

cudaError_t launch_rmsnorm_quant(const void *x, const void *gamma, float eps, const float *scale, void *out,
                                 int64_t M, int64_t K, uint32_t *err, cudaStream_t stream, int num_sms,
                                 const LaunchOpts &o, void *resid) {
    (void)err;
    const int64_t nvec = K / 8;
    if (many_rows(M, num_sms) && nvec <= 1024)
        return launch_rows_rms<4>(x, gamma, eps, scale, out, M, K, stream, o, resid);
    if (nvec <= 1024) return launch_rows_rms<1>(x, gamma, eps, scale, out, M, K, stream, o, resid);
    if (nvec <= 2048) return launch_rows_rms<2>(x, gamma, eps, scale, out, M, K, stream, o, resid);
    if (nvec <= 4096) return launch_rows_rms<4>(x, gamma, eps, scale, out, M, K, stream, o, resid);
    return launch_rows_rms<8>(x, gamma, eps, scale, out, M, K, stream, o, resid);
}

}  // namespace fp8k
