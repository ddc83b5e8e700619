// gemm_w8a16.cu -- weight-only FP8 GEMM (W8A16) for small M: bf16 activations
// x [M,K], E4M3 weights W [N,K] with a per-tensor or per-output-channel scale,
// bf16 out:  y[m,n] = bf16( (sum_k x[m,k] * dec(W[n,k])) * sb ).
// Sources: "[Kernel] add Flashinfer cutedsl w4a16 linear" (vllm #53014): the
// FP8 channelwise half of the weight-only path (the weight stays E4M3 in HBM
// and is widened on chip; at decode M the kernel is bound by the weight
// bytes), and its large-M branch (a dense 16-bit GEMM over the widened
// weight), here a tile kernel that widens the weight on chip too.
//
// Design (GB300, sm_103a).  The tensor core's kind::f16 takes both operands in
// one 16-bit type, so the E4M3 weight tile is widened to bf16 (exact: every
// E4M3 value is a bf16 value) before the MMA reads it -- into tensor memory,
// which the MMA can take its A operand from, so that shared memory carries
// only the E4M3 box and the tokens (widening into shared memory tripled its
// traffic per k-block and bounded the kernel).  Units are (128-row output
// tile) x (128-wide k-block), divided among persistent CTAs as in the W8A8
// kernel's stream-K mode: two per SM for the 16-token tile, one for the
// 32-token tile.  Inside a CTA:
//   * warp 0 / lane 0 streams each unit's 128 x 128-byte E4M3 weight box and
//     its two TOK x 64-element bf16 token boxes with TMA into a ring of stages
//     (128-byte swizzle);
//   * warps 6-9, one weight row per thread (the row of the thread's TMEM
//     lane), widen each unit's E4M3 row into 64 TMEM columns of one of two
//     A tiles (two K elements per column) and release the weight stage at
//     once;
//   * warps 2-5 drain each unit's fp32 partial out of TMEM into TwoSum
//     registers -- the same drain, tile store and stream-K fix-up as the W8A8
//     decode kernel;
//   * warp 1 / lane 0 issues eight tcgen05.mma kind::f16 (BF16 x BF16 -> F32,
//     M = 128 weight rows from TMEM, N = TOK tokens from shared memory,
//     K = 16) per unit into one of several TMEM accumulators.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"
#include "splitk.cuh"

#include <algorithm>

namespace fp8k {
namespace {

constexpr uint32_t kW16WeightBytes = kDecodeRows * kBlockK;    // 16 KB of E4M3 per stage

template <int TOK>
struct W16Cfg {
    // producer warp, MMA warp, one drain warpgroup, one widening warpgroup
    // (each thread widens one weight row); kWidenGroups > 1 splits the rows'
    // chunks between several (two were slower than two CTAs per SM of one)
    static constexpr int kWidenGroups = 1;
    static constexpr int kThreads = 64 + 128 + 128 * kWidenGroups;
    // registers per thread: two CTAs per SM for the 16-token tile (10 warps
    // each), one for the 32-token tile, whose drain needs more
    static constexpr int kMaxRegs = TOK <= 16 ? 96 : 168;
    static constexpr int kDrainThreads = 128;
    static constexpr int kBufs = 4;  // TMEM accumulators
    // widened tiles ahead of the MMA, in TMEM after the accumulators: 64
    // columns each (128 rows x 128 bf16); three for the 16-token tile (with
    // four accumulators instead of eight: 1-2% faster at M = 1 to 16)
    static constexpr int kABufs = TOK <= 16 ? 3 : 2;
    static constexpr uint32_t kACol0 = kBufs * TOK;
    static constexpr uint32_t kTmemCols = 256;  // kACol0 + kABufs * 64 = 256 for both tiles; two CTAs per SM at most
    static constexpr uint32_t kXRegion = TOK * 128;              // 64 bf16 of K for TOK tokens
    static constexpr uint32_t kXStageBytes = 2 * kXRegion;       // one unit's token tile
    static constexpr int kXStages = TOK <= 16 ? 4 : 8;          // token ring
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kDecodeRows, TOK);
    static_assert(kACol0 + kABufs * 64 <= kTmemCols, "accumulators and widened tiles fit the allocation");
};

// Two E4M3 codes (the first in the low byte) -> two bf16 (the first in the low
// half); exact, NaN codes give NaN.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t pair) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair), __NV_E4M3);
    const float2 f = __half22float2(__half2(h));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    return static_cast<uint32_t>(__bfloat16_as_ushort(b.x)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b.y)) << 16);
}

// Four E4M3 codes (code i in byte i of w) -> four bf16 (codes 0, 1 in `lo`,
// 2, 3 in `hi`, the first of each pair in the low half), with integer
// operations and one bf16 multiply per pair instead of the conversion pipe.
// A code's seven magnitude bits are placed at bits 4..10 of a bf16 pattern and
// its sign at bit 15: the E4M3 exponent lands in the low four bits of the bf16
// exponent and the three mantissa bits at the top of the bf16 mantissa, a bf16
// number equal to the code's value times 2^-120 (exponent 0 gives the bf16
// subnormal with the same mantissa, as E4M3's subnormals).  The placement:
// a byte permute puts code c in the low byte of a 16-bit lane and its sign
// replicated in the high byte (0x00 or 0xFF), a shift by 4 moves the magnitude
// to bits 4..10 and the sign copies to bits 11..15 (those of the low lane
// spill into bits 16..19), and one mask keeps bits 4..10 and 15 of each lane.
// Multiplying by 2^120 in bf16 is exact, the product being a bf16 number, so
// the result is the decoded value.  The NaN codes (magnitude 0x7F) come out as
// 480: bit 7 of each byte of (magnitude + 1), OR-ed into `nan`, is set exactly
// for them, and the caller converts such chunks again with e4m3x2_to_bf16x2.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(a), "r"(sel));
    return d;
}

__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t &lo, uint32_t &hi, uint32_t &nan) {
    nan |= ((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
    constexpr uint32_t kKeep = 0x87F087F0u, kTwo120 = 0x7B807B80u;  // bf16 2^120 in both halves
    // selector nibbles: byte c copied (c), byte c's sign replicated (8 + c)
    const uint32_t plo = (prmt(w, 0x9180u) << 4) & kKeep;
    const uint32_t phi = (prmt(w, 0xB3A2u) << 4) & kKeep;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(plo), "r"(kTwo120));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(phi), "r"(kTwo120));
}

// Row r of a 128 x 128-byte E4M3 box (128-byte swizzle: 16-byte chunk j of
// row r sits at chunk j ^ (r % 8)), chunks [J0, J0 + NJ), widened into the
// calling thread's TMEM lane: K elements 2c, 2c + 1 in column c of the tile
// at `trow` (this lane's address of the tile's first column).
template <int NJ>
__device__ __forceinline__ void widen_row_tmem(const uint8_t *src, uint32_t trow, int r, int J0) {
    static_assert(NJ % 4 == 0, "whole 64-element halves");
    const int sw = r & 7;
    const uint8_t *srow = src + r * 128;
#pragma unroll
    for (int h = 0; h < NJ / 4; ++h) {
        uint32_t o[32];
        uint32_t nan = 0;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = J0 + 4 * h + jj;
            const uint4 q = *reinterpret_cast<const uint4 *>(srow + ((j ^ sw) << 4));
            e4m3x4_to_bf16x4(q.x, o[8 * jj + 0], o[8 * jj + 1], nan);
            e4m3x4_to_bf16x4(q.y, o[8 * jj + 2], o[8 * jj + 3], nan);
            e4m3x4_to_bf16x4(q.z, o[8 * jj + 4], o[8 * jj + 5], nan);
            e4m3x4_to_bf16x4(q.w, o[8 * jj + 6], o[8 * jj + 7], nan);
        }
        if (nan & 0x80808080u) {  // a NaN code in these 64: convert them again, NaN-preserving
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = J0 + 4 * h + jj;
                const uint4 q = *reinterpret_cast<const uint4 *>(srow + ((j ^ sw) << 4));
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    o[8 * jj + 2 * t] = e4m3x2_to_bf16x2(w[t] & 0xFFFFu);
                    o[8 * jj + 2 * t + 1] = e4m3x2_to_bf16x2(w[t] >> 16);
                }
            }
        }
        __syncwarp();  // the TMEM store is warp-collective
        tmem_st32(trow + static_cast<uint32_t>(J0 * 8 + 32 * h), o);
    }
}

// (No __launch_bounds__: the register cap is set from the warp count.)
template <int TOK>
__global__ void __maxnreg__(W16Cfg<TOK>::kMaxRegs)
    w8a16_decode_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                        const DecodeArgs args) {
    using Cfg = W16Cfg<TOK>;
    constexpr int NB = Cfg::kBufs;
    constexpr int kSlotElems = TOK * kDecodeRows;  // fp32 entries of one partial slot
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base, s_last;
    __shared__ uint32_t s_w_issued, s_w_consumed, s_x_issued, s_x_consumed;  // loads requested / used
    __shared__ int64_t s_slot[2][kMaxFixupSegs];
    __shared__ int s_nseg[2];
    __shared__ volatile uint32_t s_abort;

    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stages = args.stages;  // the weight ring
    constexpr int NX = Cfg::kXStages;
    constexpr int NA = Cfg::kABufs;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    // [weight ring: stages x 16 KB][token ring: NX x TOK*256 B][barriers]; the
    // widened tiles live in TMEM
    const uint32_t xbase = base + static_cast<uint32_t>(stages) * kW16WeightBytes;
    const uint32_t bar0 = xbase + static_cast<uint32_t>(NX) * Cfg::kXStageBytes;
    auto wfull_bar = [&](int s) { return bar0 + 8u * s; };
    auto wempty_bar = [&](int s) { return bar0 + 8u * (stages + s); };
    auto xfull_bar = [&](int s) { return bar0 + 8u * (2 * stages + s); };
    auto xempty_bar = [&](int s) { return bar0 + 8u * (2 * stages + NX + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * stages + 2 * NX + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * stages + 2 * NX + NB + b); };
    auto afull_bar = [&](int a) { return bar0 + 8u * (2 * stages + 2 * NX + 2 * NB + a); };
    auto aempty_bar = [&](int a) { return bar0 + 8u * (2 * stages + 2 * NX + 2 * NB + NA + a); };
    const uint32_t final_bar = bar0 + 8u * (2 * stages + 2 * NX + 2 * NB + 2 * NA);

    const int64_t G = gridDim.x, U = args.units;
    const int64_t me = blockIdx.x;
    const int64_t u0 = unit_begin(me, U, G), u1 = unit_begin(me + 1, U, G);
    const int iters = static_cast<int>(u1 - u0);
    const int kbt = args.kb_total, n_tiles = args.n_tiles;
    uint32_t *const err = args.err;

    if (tid == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_x);
        for (int s = 0; s < stages; ++s) {
            mbar_init(wfull_bar(s), 1);
            mbar_init(wempty_bar(s), 4 * Cfg::kWidenGroups);  // one arrive per widening warp
        }
        for (int s = 0; s < NX; ++s) {
            mbar_init(xfull_bar(s), 1);
            mbar_init(xempty_bar(s), 1);  // the MMA's commit
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4);  // one arrive per drain warp
        }
        for (int a = 0; a < NA; ++a) {
            mbar_init(afull_bar(a), 4 * Cfg::kWidenGroups);  // one arrive per widening warp
            mbar_init(aempty_bar(a), 1);                      // the MMA's commit
        }
        mbar_init(final_bar, 1);
        fence_mbar_init();
        s_w_issued = s_w_consumed = s_x_issued = s_x_consumed = 0;
        s_abort = 0;
    }
    if (warp == 1) tmem_alloc(smem_u32(&s_tmem_base), Cfg::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------------- producer
        // The weight ring is released by the widening warps as soon as they
        // have read a stage, the token ring by the MMA; each runs ahead on its own.
        const uint64_t evict_first = policy_evict_first();
        int i = 0;
        // Weights that no earlier kernel in the stream writes may be fetched
        // before the dependency wait; the tokens always wait.
        const int pre = args.weights_static ? min(iters, stages) : 0;
        for (; i < pre; ++i) {
            const int64_t u = u0 + i, t = u / kbt;
            const int kb = static_cast<int>(u - t * kbt), n_tile = static_cast<int>(t % n_tiles);
            mbar_arrive_expect_tx(wfull_bar(i), kW16WeightBytes);
            tma_load_2d_hint(base + static_cast<uint32_t>(i) * kW16WeightBytes, &tmap_w, wfull_bar(i), kb * kBlockK,
                             n_tile * kDecodeRows, evict_first);
        }
        s_w_issued = static_cast<uint32_t>(i);
        grid_dependency_wait();
        int wi = i, xi = 0;  // units whose weights / tokens are requested
        int wt = static_cast<int>((u0 + wi) / kbt), wkb = static_cast<int>(u0 + wi - static_cast<int64_t>(wt) * kbt);
        int xt = static_cast<int>(u0 / kbt), xkb = static_cast<int>(u0 - static_cast<int64_t>(xt) * kbt);
        bool ok = true;
        while (ok && (wi < iters || xi < iters)) {
            // tokens first while they trail the weights (the MMA needs both)
            if (xi < iters && (xi < wi || wi == iters)) {
                if (xkb == kbt) {
                    xkb = 0;
                    ++xt;
                }
                const int s = xi % NX;
                if (!cta_wait(xempty_bar(s), (static_cast<uint32_t>(xi / NX) & 1u) ^ 1u, err, kErrDecodeEmptyWait,
                              &s_abort)) {
                    ok = false;
                    break;
                }
                const uint32_t xs = xbase + static_cast<uint32_t>(s) * Cfg::kXStageBytes;
                const int m_tile = xt / n_tiles;
                mbar_arrive_expect_tx(xfull_bar(s), Cfg::kXStageBytes);
                tma_load_2d(xs, &tmap_x, xfull_bar(s), xkb * kBlockK, m_tile * TOK);
                tma_load_2d(xs + Cfg::kXRegion, &tmap_x, xfull_bar(s), xkb * kBlockK + 64, m_tile * TOK);
                ++xi;
                ++xkb;
                s_x_issued = static_cast<uint32_t>(xi);
            } else {
                if (wkb == kbt) {
                    wkb = 0;
                    ++wt;
                }
                const int s = wi % stages;
                if (!cta_wait(wempty_bar(s), (static_cast<uint32_t>(wi / stages) & 1u) ^ 1u, err,
                              kErrDecodeEmptyWait, &s_abort)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(wfull_bar(s), kW16WeightBytes);
                tma_load_2d_hint(base + static_cast<uint32_t>(s) * kW16WeightBytes, &tmap_w, wfull_bar(s),
                                 wkb * kBlockK, (wt % n_tiles) * kDecodeRows, evict_first);
                ++wi;
                ++wkb;
                s_w_issued = static_cast<uint32_t>(wi);
            }
        }
        grid_launch_dependents();
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        int i = 0;
        for (; i < iters; ++i) {
            const int s = i % NX, b = i % NB, a = i % NA;
            const uint32_t ph = static_cast<uint32_t>(i / NX) & 1u, tph = static_cast<uint32_t>(i / NB) & 1u,
                           aph = static_cast<uint32_t>(i / NA) & 1u;
            if (!cta_wait(xfull_bar(s), ph, err, kErrDecodeFullWait, &s_abort)) break;
            if (!cta_wait(afull_bar(a), aph, err, kErrW16AFullWait, &s_abort)) break;
            if (!cta_wait(tempty_bar(b), tph ^ 1u, err, kErrDecodeTmemEmptyWait, &s_abort)) break;
            tc_fence_after();
            const uint32_t xs = xbase + static_cast<uint32_t>(s) * Cfg::kXStageBytes;
            const uint32_t at = tmem + Cfg::kACol0 + static_cast<uint32_t>(a) * 64u;
            const uint32_t d = tmem + static_cast<uint32_t>(b * TOK);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // K = 16 bf16 per MMA: 8 TMEM columns of A, 32 bytes of the token tile
                const uint32_t h = static_cast<uint32_t>(kk >> 2), o = 2u * static_cast<uint32_t>(kk & 3);
                mma_bf16_tmem_a(d, at + 8u * static_cast<uint32_t>(kk), sw128_kmajor_desc(xs + h * Cfg::kXRegion) + o,
                                Cfg::kIdesc, kk > 0 ? 1u : 0u);
            }
            mma_commit(xempty_bar(s));
            mma_commit(aempty_bar(a));
            mma_commit(tfull_bar(b));
        }
        s_x_consumed = static_cast<uint32_t>(i);
        mma_commit(final_bar);  // arrives when every MMA issued above has completed
    } else if (warp >= 6) {
        // ---------------------------------------------------------------- widening
        // Unit j's E4M3 weights widened into A tile j % NA once the stage has
        // landed and the MMA of unit j - NA has finished reading the tile; the
        // weight stage is released right after.  Warpgroup g widens chunks
        // [g*8/WG, (g+1)*8/WG) of every row.
        constexpr int kNJ = 8 / Cfg::kWidenGroups;
        const int row = static_cast<int>((warp & 3u) * 32u + lane);
        const int j0 = static_cast<int>((warp - 6) / 4) * kNJ;
        int j = 0;
        for (; j < iters; ++j) {
            const int s = j % stages, a = j % NA;
            // the TMEM stores below are warp-collective: the warp goes on only
            // if every lane's wait succeeded
            bool ok = cta_wait(wfull_bar(s), static_cast<uint32_t>(j / stages) & 1u, err, kErrW16FullWait, &s_abort);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            ok = cta_wait(aempty_bar(a), (static_cast<uint32_t>(j / NA) & 1u) ^ 1u, err, kErrW16AEmptyWait, &s_abort);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            widen_row_tmem<kNJ>(smem_raw + (base + static_cast<uint32_t>(s) * kW16WeightBytes - raw),
                                tmem + ((static_cast<uint32_t>(warp & 3u) * 32u) << 16) + Cfg::kACol0 +
                                    static_cast<uint32_t>(a) * 64u,
                                row, j0);
            tmem_st_wait();  // the stores, before the tensor core reads them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(afull_bar(a));
                mbar_arrive(wempty_bar(s));
            }
        }
        if (warp == 6 && lane == 0) s_w_consumed = static_cast<uint32_t>(j);
    } else if (warp >= 2) {
        // ---------------------------------------------------------------- drain + tile output
        const uint32_t quarter = warp & 3u;                      // TMEM lanes 32*(warp%4) .. +31
        const int row = static_cast<int>(quarter * 32u + lane);  // weight row within the tile
        grid_dependency_wait();  // outputs, scales and the workspace are touched below
        const bool sb_vec = args.gran == 1;
        const float sb0 = __ldg(args.scale_b);
        const int t_first_me = static_cast<int>(u0 / kbt);
        if (tid == 64 && iters > 0) {
            // Which CTAs hold the other parts of this CTA's first and last tile
            // and where their partial sums go.
            for (int w = 0; w < 2; ++w) {
                const int64_t t = (w == 0 ? u0 : u1 - 1) / kbt, tile_u0 = t * kbt;
                const int64_t c_first = unit_owner(tile_u0, U, G), c_last = unit_owner(tile_u0 + kbt - 1, U, G);
                const int nseg = static_cast<int>(c_last - c_first + 1);
                s_nseg[w] = nseg;
                for (int j = 0; j < kMaxFixupSegs && j < nseg; ++j) {
                    const int64_t cc = c_first + j;
                    s_slot[w][j] = (2 * cc + (t == unit_begin(cc, U, G) / kbt ? 0 : 1)) * kSlotElems;
                }
            }
        }
        float hi[TOK], lo[TOK];
#pragma unroll
        for (int c = 0; c < TOK; ++c) hi[c] = lo[c] = 0.0f;

        int t = static_cast<int>(u0 / kbt), kb = static_cast<int>(u0 - static_cast<int64_t>(t) * kbt);
        for (int i = 0; i < iters; ++i, ++kb) {
            if (kb == kbt) {
                kb = 0;
                ++t;
            }
            const int b = i % NB;
            const uint32_t tph = static_cast<uint32_t>(i / NB) & 1u;
            cta_wait(tfull_bar(b), tph, err, kErrDecodeTmemFullWait, &s_abort);
            __syncwarp();
            tc_fence_after();
            const uint32_t taddr = tmem + ((quarter * 32u) << 16) + static_cast<uint32_t>(b * TOK);
#pragma unroll
            for (int c0 = 0; c0 < TOK; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(taddr + static_cast<uint32_t>(c0), r);
                tmem_ld_wait();
                if (c0 + 16 >= TOK) {  // last chunk read: the accumulator is free for the MMA again
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar(b));
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) two_sum_acc(hi[c0 + j], lo[c0 + j], __uint_as_float(r[j]));
            }

            if (kb != kbt - 1 && i != iters - 1) continue;

            // ---- this CTA's part of tile t ends here
            const int n_tile = t % n_tiles, m_tile = t / n_tiles;
            const int n = n_tile * kDecodeRows + row;
            const int m0 = m_tile * TOK;
            const int mt = min(TOK, args.M - m0);
            const int64_t tile_u0 = static_cast<int64_t>(t) * kbt;
            const bool whole = (u0 <= tile_u0) && (kb == kbt - 1);
            if (!whole) {
                // this CTA's part of the tile, rounded once to binary32, then
                // the arrival count; the last of the tile's parts sums them all
                float *mine = args.slots + static_cast<int64_t>(2 * me + (t == t_first_me ? 0 : 1)) * kSlotElems;
#pragma unroll
                for (int c = 0; c < TOK; ++c)
                    if (c < mt) mine[c * kDecodeRows + row] = __fadd_rn(hi[c], lo[c]);
                named_barrier_sync(1, Cfg::kDrainThreads);
                const int w = (t == t_first_me) ? 0 : 1;
                if (tid == 64) {
                    const int nseg = s_nseg[w];
                    __threadfence();
                    const bool last = atomicAdd(args.counters + t, 1u) == static_cast<uint32_t>(nseg - 1);
                    if (last) __threadfence();
                    s_last = last ? static_cast<uint32_t>(nseg) : 0u;
                }
                named_barrier_sync(1, Cfg::kDrainThreads);
                if (s_last != 0u) {
                    int nseg = static_cast<int>(s_last);
                    if (nseg > kMaxFixupSegs) {  // the planner keeps this from happening
                        if (tid == 64) atomicOr(err, kErrDecodeFixup);
                        nseg = kMaxFixupSegs;
                    }
                    fixup_sum<kMaxFixupSegs, 1, Cfg::kDrainThreads>(args, s_slot[w], nseg, mt * kDecodeRows,
                                                                     static_cast<int>(tid) - 64, n_tile, m0, false,
                                                                     sb_vec, 1.0f, sb0);
                    if (tid == 64) args.counters[t] = 0u;  // ready for the next launch
                }
            } else if (n < args.N) {
                const float sb = sb_vec ? __ldg(args.scale_b + n) : sb0;
#pragma unroll
                for (int c = 0; c < TOK; ++c)
                    if (c < mt)
                        args.out[static_cast<int64_t>(m0 + c) * args.N + n] =
                            __float2bfloat16_rn(__fmul_rn(__fadd_rn(hi[c], lo[c]), sb));
            }
#pragma unroll
            for (int c = 0; c < TOK; ++c) hi[c] = lo[c] = 0.0f;
        }
    }
    __syncwarp();
    grid_dependency_wait();
    grid_launch_dependents();
    __syncthreads();

    if (tid == 0) {
        // Loads issued but never consumed (only after a timeout): let them land
        // before the CTA exits.
        for (uint32_t i = s_w_consumed; i < s_w_issued; ++i)
            mbar_wait(wfull_bar(static_cast<int>(i % stages)), (i / stages) & 1u, err, kErrW16FullWait);
        for (uint32_t i = s_x_consumed; i < s_x_issued; ++i)
            mbar_wait(xfull_bar(static_cast<int>(i % NX)), (i / NX) & 1u, err, kErrDecodeFullWait);
    }
    if (warp == 1) {
        mbar_wait(final_bar, 0, err, kErrDecodeAccumWait);  // every MMA has completed
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

template <int TOK>
cudaError_t launch_w16(const CUtensorMap &tw, const CUtensorMap &tx, const DecodeArgs &a, const DecodePlan &p,
                       const LaunchOpts &o, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool attr_done[64] = {};  // benign race: the attribute call is idempotent
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(w8a16_decode_kernel<TOK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(p.smem_bytes));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    return launch_with_opts(w8a16_decode_kernel<TOK>, dim3(static_cast<unsigned>(p.ctas)),
                            dim3(W16Cfg<TOK>::kThreads), p.smem_bytes, stream, o, tw, tx, a);
}

// ------------------------------------------------------------- large-M tile kernel
//
// The weight-only GEMM's large-M branch (the pages' branch widens the weight to
// 16 bits for a dense 16-bit GEMM; here the widening happens on chip, box by
// box, so HBM holds and streams only the E4M3 weight and nothing is
// allocated).  Output tiles of 256 weight rows (two 128-row halves) x 128
// tokens, the whole K range each, walked by persistent CTAs (one per SM),
// token tile fastest, so that the CTAs running at the same time read each
// weight box and token box from L2 many times.  When the last round of tiles
// would leave more than half of the CTAs idle, its tiles run as half tiles
// (one 128-row half each) on twice as many CTAs.  Inside a CTA:
//   * warp 0 / lane 0 loads each k-block's E4M3 weight boxes (128 x 128 bytes
//     per half) and its token boxes (128 tokens x 64 bf16, two) with TMA into
//     two rings;
//   * warps 6-13, one weight row per thread (warps 6-9 the first half, 10-13
//     the second), widen the k-block's E4M3 rows into one of two A tiles in
//     tensor memory (128 lanes x 64 columns per half) and release the weight
//     stage (sixteen widening warps, a half row each, were slower);
//   * warp 1 / lane 0 issues eight tcgen05.mma kind::f16 per half and k-block
//     (M = 128 weight rows from TMEM, N = 128 tokens from shared memory,
//     K = 16) into the half's fp32 accumulator in TMEM;
//   * warps 2-5 (one weight row per thread and half) read the finished
//     accumulator, apply the weight scale in binary32, round to bf16 and
//     store.
// Tensor memory: the accumulator (2 x 128 columns) and two widened k-blocks
// (2 x 2 x 64 columns) fill the 512 columns, so the accumulator is single:
// the next tile's MMAs wait for the drain (a few percent of a tile's time).
struct W16TileCfg {
    static constexpr int kThreads = 448;  // producer, MMA, epilogue warpgroup (2-5), two widening warpgroups (6-13)
    static constexpr int kWidenWarps = 8;
    static constexpr int TN = kW16TileTokens;
    static constexpr uint32_t kWStageBytes = 2 * kW16WeightBytes;  // both halves of one k-block
    static constexpr uint32_t kXRegion = TN * 128;                  // 64 bf16 of K for TN tokens
    static constexpr uint32_t kXStageBytes = 2 * kXRegion;          // one k-block of the token tile
    static constexpr int kABufs = 2;                                 // widened k-blocks, 2 x 64 columns each
    static constexpr uint32_t kACol0 = 2 * TN;                       // after the accumulator's two halves
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kDecodeRows, TN);
    static_assert(kACol0 + kABufs * 128 <= kTmemCols, "accumulator and widened tiles fit the allocation");
};

__global__ void __launch_bounds__(W16TileCfg::kThreads, 1)
    w8a16_tile_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                      const W16TileArgs args) {
    using Cfg = W16TileCfg;
    constexpr int TN = Cfg::TN;
    constexpr int NA = Cfg::kABufs;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ uint32_t s_w_issued, s_w_consumed, s_x_issued, s_x_consumed;  // loads requested / used
    __shared__ volatile uint32_t s_abort;

    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int WS = args.wstages, XS = args.xstages;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    // [weight ring: WS x 32 KB][token ring: XS x 32 KB][barriers]
    const uint32_t xbase = base + static_cast<uint32_t>(WS) * Cfg::kWStageBytes;
    const uint32_t bar0 = xbase + static_cast<uint32_t>(XS) * Cfg::kXStageBytes;
    auto wfull_bar = [&](int s) { return bar0 + 8u * s; };
    auto wempty_bar = [&](int s) { return bar0 + 8u * (WS + s); };
    auto xfull_bar = [&](int s) { return bar0 + 8u * (2 * WS + s); };
    auto xempty_bar = [&](int s) { return bar0 + 8u * (2 * WS + XS + s); };
    const uint32_t dfull_bar = bar0 + 8u * (2 * WS + 2 * XS);
    const uint32_t dempty_bar = dfull_bar + 8u;
    auto afull_bar = [&](int a) { return dempty_bar + 8u * (1 + a); };
    auto aempty_bar = [&](int a) { return dempty_bar + 8u * (1 + NA + a); };
    const uint32_t final_bar = dempty_bar + 8u * (1 + 2 * NA);

    const int kbt = args.kb_total, G = static_cast<int>(gridDim.x), me = static_cast<int>(blockIdx.x);
    const int my_units = args.units > me ? (args.units - me + G - 1) / G : 0;  // units me, me + G, ...
    const int total = my_units * kbt;                                          // k-block steps of this CTA
    uint32_t *const err = args.err;

    if (tid == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_x);
        for (int s = 0; s < WS; ++s) {
            mbar_init(wfull_bar(s), 1);
            mbar_init(wempty_bar(s), Cfg::kWidenWarps);  // one arrive per widening warp
        }
        for (int s = 0; s < XS; ++s) {
            mbar_init(xfull_bar(s), 1);
            mbar_init(xempty_bar(s), 1);  // the MMA's commit
        }
        mbar_init(dfull_bar, 1);   // the MMA's commit after a tile's last k-block
        mbar_init(dempty_bar, 4);  // one arrive per epilogue warp
        for (int a = 0; a < NA; ++a) {
            mbar_init(afull_bar(a), Cfg::kWidenWarps);  // one arrive per widening warp
            mbar_init(aempty_bar(a), 1);  // the MMA's commit
        }
        mbar_init(final_bar, 1);
        fence_mbar_init();
        s_w_issued = s_w_consumed = s_x_issued = s_x_consumed = 0;
        s_abort = 0;
    }
    if (warp == 1) tmem_alloc(smem_u32(&s_tmem_base), Cfg::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;

    // Unit j of this CTA: u = me + j * G.  Units below full_units are whole
    // tiles (both halves), the rest half tiles of the last tiles, two per
    // tile; a half that starts at or beyond N is dropped.  Token tile fastest.
    auto unit_of = [&](int j, int &m_tile, int &n_tile, uint32_t &halves) {
        const int u = me + j * G;
        int t;
        if (u < args.full_units) {
            t = u;
            halves = 3u;
        } else {
            const int v = u - args.full_units;
            t = args.full_units + (v >> 1);
            halves = 1u << (v & 1);
        }
        m_tile = t % args.m_tiles;
        n_tile = t / args.m_tiles;
        if (n_tile * (2 * kDecodeRows) + kDecodeRows >= args.N) halves &= 1u;
    };

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------------- producer
        auto load_w = [&](int q, int s) {
            int mt, nt;
            uint32_t hm;
            unit_of(q / kbt, mt, nt, hm);
            const int kx = (q % kbt) * kBlockK;
            const uint32_t ws = base + static_cast<uint32_t>(s) * Cfg::kWStageBytes;
            mbar_arrive_expect_tx(wfull_bar(s), static_cast<uint32_t>(__popc(hm)) * kW16WeightBytes);
            for (int h = 0; h < 2; ++h)
                if ((hm >> h) & 1u)
                    tma_load_2d(ws + static_cast<uint32_t>(h) * kW16WeightBytes, &tmap_w, wfull_bar(s), kx,
                                (2 * nt + h) * kDecodeRows);
        };
        int wi = 0, xi = 0;  // steps whose weights / tokens are requested
        // Weights that no earlier kernel in the stream writes may be fetched
        // before the dependency wait; the tokens always wait.
        const int pre = args.weights_static ? min(total, WS) : 0;
        for (; wi < pre; ++wi) load_w(wi, wi);
        s_w_issued = static_cast<uint32_t>(wi);
        grid_dependency_wait();
        bool ok = true;
        while (ok && (wi < total || xi < total)) {
            // tokens first while they trail the weights (the MMA needs both)
            if (xi < total && (xi < wi || wi == total)) {
                const int s = xi % XS;
                if (!cta_wait(xempty_bar(s), (static_cast<uint32_t>(xi / XS) & 1u) ^ 1u, err, kErrDecodeEmptyWait,
                              &s_abort)) {
                    ok = false;
                    break;
                }
                int mt, nt;
                uint32_t hm;
                unit_of(xi / kbt, mt, nt, hm);
                const int kx = (xi % kbt) * kBlockK;
                const uint32_t xs = xbase + static_cast<uint32_t>(s) * Cfg::kXStageBytes;
                mbar_arrive_expect_tx(xfull_bar(s), Cfg::kXStageBytes);
                tma_load_2d(xs, &tmap_x, xfull_bar(s), kx, mt * TN);
                tma_load_2d(xs + Cfg::kXRegion, &tmap_x, xfull_bar(s), kx + 64, mt * TN);
                ++xi;
                s_x_issued = static_cast<uint32_t>(xi);
            } else {
                const int s = wi % WS;
                if (!cta_wait(wempty_bar(s), (static_cast<uint32_t>(wi / WS) & 1u) ^ 1u, err, kErrDecodeEmptyWait,
                              &s_abort)) {
                    ok = false;
                    break;
                }
                load_w(wi, s);
                ++wi;
                s_w_issued = static_cast<uint32_t>(wi);
            }
        }
        grid_launch_dependents();
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        int q = 0;
        for (; q < total; ++q) {
            const int s = q % XS, a = q % NA, j = q / kbt, kb = q % kbt;
            if (!cta_wait(xfull_bar(s), static_cast<uint32_t>(q / XS) & 1u, err, kErrDecodeFullWait, &s_abort)) break;
            if (!cta_wait(afull_bar(a), static_cast<uint32_t>(q / NA) & 1u, err, kErrW16AFullWait, &s_abort)) break;
            if (kb == 0 && !cta_wait(dempty_bar, (static_cast<uint32_t>(j) & 1u) ^ 1u, err, kErrDecodeTmemEmptyWait,
                                     &s_abort))
                break;
            tc_fence_after();
            int mt, nt;
            uint32_t hm;
            unit_of(j, mt, nt, hm);
            const uint32_t xs = xbase + static_cast<uint32_t>(s) * Cfg::kXStageBytes;
            for (int h = 0; h < 2; ++h) {
                if (!((hm >> h) & 1u)) continue;
                const uint32_t at = tmem + Cfg::kACol0 + static_cast<uint32_t>(a * 128 + h * 64);
                const uint32_t d = tmem + static_cast<uint32_t>(h * TN);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {  // K = 16 bf16 per MMA: 8 TMEM columns of A, 32 bytes of the tokens
                    const uint32_t r = static_cast<uint32_t>(kk >> 2), o = 2u * static_cast<uint32_t>(kk & 3);
                    mma_bf16_tmem_a(d, at + 8u * static_cast<uint32_t>(kk),
                                    sw128_kmajor_desc(xs + r * Cfg::kXRegion) + o, Cfg::kIdesc,
                                    (kb > 0 || kk > 0) ? 1u : 0u);
                }
            }
            mma_commit(xempty_bar(s));
            mma_commit(aempty_bar(a));
            if (kb == kbt - 1) mma_commit(dfull_bar);
        }
        s_x_consumed = static_cast<uint32_t>(q);
        mma_commit(final_bar);  // arrives when every MMA issued above has completed
    } else if (warp >= 6) {
        // ---------------------------------------------------------------- widening
        const uint32_t quarter = warp & 3u, half = (warp - 6u) >> 2;
        const int row = static_cast<int>(quarter * 32u + lane);
        int q = 0;
        for (; q < total; ++q) {
            const int s = q % WS, a = q % NA;
            // the TMEM stores below are warp-collective: the warp goes on only
            // if every lane's wait succeeded
            bool ok = cta_wait(wfull_bar(s), static_cast<uint32_t>(q / WS) & 1u, err, kErrW16FullWait, &s_abort);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            ok = cta_wait(aempty_bar(a), (static_cast<uint32_t>(q / NA) & 1u) ^ 1u, err, kErrW16AEmptyWait, &s_abort);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            int mt, nt;
            uint32_t hm;
            unit_of(q / kbt, mt, nt, hm);
            if ((hm >> half) & 1u) {
                widen_row_tmem<8>(smem_raw + (base + static_cast<uint32_t>(s) * Cfg::kWStageBytes +
                                              half * kW16WeightBytes - raw),
                                  tmem + ((quarter * 32u) << 16) + Cfg::kACol0 + static_cast<uint32_t>(a) * 128u +
                                      half * 64u,
                                  row, 0);
                tmem_st_wait();  // the stores, before the tensor core reads them
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(afull_bar(a));
                mbar_arrive(wempty_bar(s));
            }
        }
        if (warp == 6 && lane == 0) s_w_consumed = static_cast<uint32_t>(q);
    } else if (warp >= 2) {
        // ---------------------------------------------------------------- epilogue
        const uint32_t quarter = warp & 3u;  // TMEM lanes 32*(warp%4) .. +31
        grid_dependency_wait();              // outputs and scales are touched below
        const float sb0 = __ldg(args.scale_b);
        for (int j = 0; j < my_units; ++j) {
            const bool ok = cta_wait(dfull_bar, static_cast<uint32_t>(j) & 1u, err, kErrDecodeTmemFullWait, &s_abort);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            int mt, nt;
            uint32_t hm;
            unit_of(j, mt, nt, hm);
            const int m0 = mt * TN;
            const int h_last = (hm >> 1) & 1u;
            for (int h = 0; h < 2; ++h) {
                if (!((hm >> h) & 1u)) continue;
                const int n = (2 * nt + h) * kDecodeRows + static_cast<int>(quarter * 32u + lane);
                const float sb = (args.per_channel && n < args.N) ? __ldg(args.scale_b + n) : sb0;
                const uint32_t taddr = tmem + ((quarter * 32u) << 16) + static_cast<uint32_t>(h * TN);
#pragma unroll 1
                for (int c0 = 0; c0 < TN; c0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(taddr + static_cast<uint32_t>(c0), r);
                    tmem_ld_wait();
                    if (h == h_last && c0 + 16 >= TN) {  // last read: the accumulator is free for the next tile
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(dempty_bar);
                    }
                    if (n < args.N) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int m = m0 + c0 + jj;
                            if (m < args.M)
                                args.out[static_cast<int64_t>(m) * args.N + n] =
                                    __float2bfloat16_rn(__fmul_rn(__uint_as_float(r[jj]), sb));
                        }
                    }
                }
            }
        }
    }
    __syncwarp();
    grid_dependency_wait();
    grid_launch_dependents();
    __syncthreads();

    if (tid == 0) {
        // Loads issued but never consumed (only after a timeout): let them land
        // before the CTA exits.
        for (uint32_t i = s_w_consumed; i < s_w_issued; ++i)
            mbar_wait(wfull_bar(static_cast<int>(i % WS)), (i / WS) & 1u, err, kErrW16FullWait);
        for (uint32_t i = s_x_consumed; i < s_x_issued; ++i)
            mbar_wait(xfull_bar(static_cast<int>(i % XS)), (i / XS) & 1u, err, kErrDecodeFullWait);
    }
    if (warp == 1) {
        mbar_wait(final_bar, 0, err, kErrDecodeAccumWait);  // every MMA has completed
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

// w16[n,k] = bf16_rne(fp32(dec(W[n,k]) * s)), one binary32 multiply rounded
// to nearest, then rounded to bf16 (s = 1 when `scale` is null: the exact
// E4M3 value); 16 codes per thread, grid-stride.
__global__ void __launch_bounds__(256) widen_weight_kernel(const uint4 *__restrict__ w, uint4 *__restrict__ out,
                                                           const float *__restrict__ scale, int per_channel,
                                                           int64_t n16, int k16) {
    grid_dependency_wait();
    grid_launch_dependents();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float s = scale ? __ldg(scale + (per_channel ? i / k16 : 0)) : 1.0f;
        const uint4 q = __ldg(w + i);
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
        uint32_t o[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>((wv[t >> 1] >> (16 * (t & 1))) & 0xFFFFu), __NV_E4M3);
            const float2 f = __half22float2(__half2(h));
            const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(f.x, s), __fmul_rn(f.y, s));
            o[t] = static_cast<uint32_t>(__bfloat16_as_ushort(b.x)) |
                   (static_cast<uint32_t>(__bfloat16_as_ushort(b.y)) << 16);
        }
        out[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
        out[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// ------------------------------------------------------------------ GEMV --
// One to four tokens: y[m,n] = bf16(fp32(acc[m,n] * sb)) with acc the binary32
// sum over K of x[m,k] * dec(W[n,k]), on the CUDA cores.  At this M the
// kernel is bound by the weight bytes and the contraction is too small to pay
// for a tensor-core hand-off per k-block (the widening into TMEM, the MMA
// hand-shakes and the cross-CTA fix-up of the split-K kernel cost more than
// the stream; see the W8A16 decode kernel above).  One CTA per SM takes a
// contiguous range of weight rows and each of its kGemvWarps warps an equal
// share of those, whole rows (no split of K: nothing is shared between warps
// or CTAs, and a row's sum stays in its warp's registers).  Each warp streams
// its rows in kGemvSeg-byte segments through its own ring of kGemvWarpStages
// shared-memory stages: lane 0 issues one 1-D bulk copy per segment (the
// first ones before the dependency wait when the weights are static, so the
// whole CTA has its ring in flight while the previous kernel finishes) and
// refills a stage as soon as the warp has read it.  Lane l multiplies the
// segment's 16-byte vectors l, l + 32, ...: each E4M3 code is widened exactly
// to bf16 (e4m3x4_to_bf16x4) and multiplied with the bf16 token into one
// binary32 accumulator per token (mixed-precision fused multiply-adds, bf16
// operands and binary32 accumulator, in k order within the lane); at the
// row's end the warp adds the lanes' sums in a fixed butterfly order and lane
// m stores token m.  A row holding a NaN code gives NaN outputs.  The tokens
// are read once per CTA into shared memory as bf16, half-vector-transposed
// ([token][8-value half h][vector v]) so that the 32 lanes' 16-byte reads of
// one half are consecutive.  (Tokens held as binary32, read once per weight
// value and token, made shared memory the bound at ~5 us per token on the
// QKV shape; multiplying several rows per warp to share those reads kept
// fewer bytes in flight per warp and was slower at one token.  Measured on
// QKV at M = 1 over the ring's shape: 24 warps x 3 stages of 2560 or 2048
// bytes 13.6-13.9 us, 32 warps x 2 x 2048 15.2, 32 x 3 x 1536 17.2, 16 x 4 x
// 2048 16.1; the 2560-byte segments win on the longer weights, gate_up 35.6
// against 38.9 us.)

// acc + w.lo * x.lo, then + w.hi * x.hi: bf16 operands, a binary32
// accumulator, each product exact and the sum rounded once to nearest (the
// same bits as widening both to binary32 and using __fmaf_rn).
__device__ __forceinline__ float fma_bf16x2_acc(uint32_t w, uint32_t x, float acc) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %1;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
        : "+f"(acc)
        : "r"(w), "r"(x));
    return acc;
}

constexpr int kGemvWarps = 24;
constexpr int kGemvThreads = 32 * kGemvWarps;
constexpr int kGemvSeg = 2560;      // bytes of one weight-row segment (one stage; 5 x 32 x 16)
constexpr int kGemvWarpStages = 3;  // stages per warp
constexpr uint32_t kGemvRingBytes = static_cast<uint32_t>(kGemvWarps * kGemvWarpStages * kGemvSeg);
constexpr uint32_t kGemvBarBytes = 8u * kGemvWarps * kGemvWarpStages;

template <int MT>
__global__ void __launch_bounds__(kGemvThreads, 1)
    w8a16_gemv_kernel(const uint8_t *__restrict__ W, const __nv_bfloat16 *__restrict__ x,
                      const float *__restrict__ scale_b, int per_channel, int N, int K,
                      __nv_bfloat16 *__restrict__ out, uint32_t *err, int weights_static) {
    extern __shared__ __align__(128) uint8_t gsm[];
    // [ring: kGemvWarps x kGemvWarpStages x kGemvSeg][barriers][tokens: MT x K bf16]
    const uint32_t ring = smem_u32(gsm);
    const uint32_t bars = ring + kGemvRingBytes;
    uint8_t *const xs = gsm + kGemvRingBytes + kGemvBarBytes;
    const int NV = K >> 4;  // 16-byte vectors per row
    const int segs = (K + kGemvSeg - 1) / kGemvSeg;
    const int tid = static_cast<int>(threadIdx.x), lane = tid & 31, warp = tid >> 5;
    const int r0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * N / gridDim.x);
    const int n = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * N / gridDim.x) - r0;
    const int wr0 = r0 + (warp * n) / kGemvWarps, wr1 = r0 + ((warp + 1) * n) / kGemvWarps;
    const int items = (wr1 - wr0) * segs;  // (row, segment) pairs of this warp, row-major
    const uint32_t stage0 = ring + static_cast<uint32_t>(warp * kGemvWarpStages * kGemvSeg);
    const uint32_t bar0 = bars + 8u * static_cast<uint32_t>(warp * kGemvWarpStages);
    const uint64_t evict_first = policy_evict_first();

    auto seg_bytes = [&](int j) { return min(kGemvSeg, K - (j % segs) * kGemvSeg); };
    // lane 0: segment j of this warp's rows into stage j % kGemvWarpStages
    auto issue = [&](int j) {
        const int s = j % kGemvWarpStages;
        const int r = wr0 + j / segs, sg = j % segs;
        const uint32_t bytes = static_cast<uint32_t>(seg_bytes(j));
        mbar_arrive_expect_tx(bar0 + 8u * s, bytes);
        const uint8_t *src = W + static_cast<int64_t>(r) * K + static_cast<int64_t>(sg) * kGemvSeg;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
            " [%0], [%1], %2, [%3], %4;" ::"r"(stage0 + static_cast<uint32_t>(s * kGemvSeg)),
            "l"(src), "r"(bytes), "r"(bar0 + 8u * s), "l"(evict_first)
            : "memory");
    };

    if (lane == 0) {
        for (int s = 0; s < kGemvWarpStages; ++s) mbar_init(bar0 + 8u * s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const int pre = min(items, kGemvWarpStages);
    // Weights that no earlier kernel in the stream writes may be fetched
    // before the dependency wait; the tokens always wait.
    if (weights_static && lane == 0)
        for (int j = 0; j < pre; ++j) issue(j);
    grid_dependency_wait();
    {
        // tokens -> shared memory, 8 bf16 (one 16-byte half of a 16-value
        // vector) per thread and step, at [token][half h][vector v]
        const int chunks = MT * (K >> 3);
        for (int c = tid; c < chunks; c += kGemvThreads) {
            const int m = c / (K >> 3), k = (c - m * (K >> 3)) << 3;
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(m) * K + k));
            *reinterpret_cast<uint4 *>(xs + ((((m * 2 + ((k >> 3) & 1)) * NV) + (k >> 4)) << 4)) = q;
        }
    }
    __syncthreads();
    // nothing of this grid is read by the next kernel before it completes:
    // let it launch, so that its prologue overlaps this grid's stream
    grid_launch_dependents();
    if (!weights_static && lane == 0)
        for (int j = 0; j < pre; ++j) issue(j);

    float acc[MT];
    uint32_t nan = 0;
    int j = 0;
    for (; j < items; ++j) {
        const int s = j % kGemvWarpStages, sg = j % segs;
        const bool ok =
            mbar_wait(bar0 + 8u * s, static_cast<uint32_t>(j / kGemvWarpStages) & 1u, err, kErrW16FullWait);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (sg == 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
            nan = 0;
        }
        const int nvec = seg_bytes(j) >> 4;
        const uint8_t *stage = gsm + (warp * kGemvWarpStages + s) * kGemvSeg;
#pragma unroll
        for (int u = 0; u < kGemvSeg / 16 / 32; ++u) {
            const int lv = u * 32 + lane;  // vector within the segment
            if (lv < nvec) {
                const uint4 q = *reinterpret_cast<const uint4 *>(stage + 16 * lv);
                const int v = sg * (kGemvSeg / 16) + lv;  // vector within the row
                const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // k = 16 v + 8 h + 0..7: weight words 2h, 2h + 1
                    uint4 xq[MT];
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        xq[m] = *reinterpret_cast<const uint4 *>(xs + ((((m * 2 + h) * NV) + v) << 4));
#pragma unroll
                    for (int t2 = 0; t2 < 2; ++t2) {
                        uint32_t lo, hi;  // bf16 pairs (k, k + 1), (k + 2, k + 3), k = 16 v + 8 h + 4 t2
                        e4m3x4_to_bf16x4(wd[2 * h + t2], lo, hi, nan);
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            acc[m] = fma_bf16x2_acc(lo, t2 == 0 ? xq[m].x : xq[m].z, acc[m]);
                            acc[m] = fma_bf16x2_acc(hi, t2 == 0 ? xq[m].y : xq[m].w, acc[m]);
                        }
                    }
                }
            }
        }
        // every lane has read the stage: refill it with segment j + stages
        __syncwarp();
        if (lane == 0 && j + kGemvWarpStages < items) {
            fence_proxy_async_smem();
            issue(j + kGemvWarpStages);
        }
        if (sg == segs - 1) {
            const int r = wr0 + j / segs;
            const bool has_nan = __any_sync(0xffffffffu, (nan & 0x80808080u) != 0u);
            const float sb = __ldg(scale_b + (per_channel ? r : 0));
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float y = acc[m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) y = __fadd_rn(y, __shfl_xor_sync(0xffffffffu, y, o));
                if (lane == m)
                    out[static_cast<int64_t>(m) * N + r] = has_nan ? __float2bfloat16_rn(__int_as_float(0x7fffffff))
                                                                   : __float2bfloat16_rn(__fmul_rn(y, sb));
            }
        }
    }
    if (j < items && lane == 0) {
        // gave up after a timed-out wait: let the copies already issued land
        // (bounded) before the CTA's shared memory is released
        const int issued = min(items, j + kGemvWarpStages);
        for (int i = j; i < issued; ++i)
            mbar_wait(bar0 + 8u * (i % kGemvWarpStages), static_cast<uint32_t>(i / kGemvWarpStages) & 1u, err,
                      kErrW16FullWait);
    }
}

}  // namespace

// Shared memory of one CTA: alignment slack, the weight ring, the token ring
// and the mbarriers (rounded up); the widened tiles are in TMEM.
static size_t w16_smem_bytes(int tok, int stages) {
    const int nb = tok <= 16 ? W16Cfg<16>::kBufs : W16Cfg<32>::kBufs;
    const int nx = tok <= 16 ? W16Cfg<16>::kXStages : W16Cfg<32>::kXStages;
    const int na = tok <= 16 ? W16Cfg<16>::kABufs : W16Cfg<32>::kABufs;
    const size_t barriers = 8u * static_cast<size_t>(2 * stages + 2 * nx + 2 * nb + 2 * na + 1);
    return 1024 + static_cast<size_t>(stages) * kW16WeightBytes + static_cast<size_t>(nx) * 2u * tok * 128u +
           ((barriers + 127) / 128) * 128;
}

DecodePlan plan_w8a16(int64_t M, int64_t N, int64_t K, int num_sms) {
    DecodePlan p{};
    p.tok_pad = M <= 16 ? 16 : 32;
    // 16 tokens: 5 weight stages and 4 token stages (~98 KB, two CTAs per SM);
    // 32 tokens: 8 and 8 (~194 KB, one CTA per SM)
    p.stages = p.tok_pad == 16 ? 5 : 8;
    p.smem_bytes = w16_smem_bytes(p.tok_pad, p.stages);
    p.n_tiles = static_cast<int>((N + kDecodeRows - 1) / kDecodeRows);
    p.m_tiles = static_cast<int>((M + p.tok_pad - 1) / p.tok_pad);
    p.kb_total = static_cast<int>((K + kBlockK - 1) / kBlockK);
    p.units = static_cast<int64_t>(p.n_tiles) * p.m_tiles * p.kb_total;
    p.split = 0;
    // Persistent CTAs (two or one per SM), at least kb_total / (kMaxFixupSegs
    // - 1) units each (at most kMaxFixupSegs CTAs share a tile).
    const int64_t min_units = (p.kb_total + kMaxFixupSegs - 2) / (kMaxFixupSegs - 1);
    int64_t ctas = p.tok_pad == 16 ? 2 * static_cast<int64_t>(num_sms) : num_sms;
    if (ctas > p.units / min_units) ctas = p.units / min_units;
    if (ctas < 1) ctas = 1;
    p.ctas = static_cast<int>(ctas);
    return p;
}

cudaError_t launch_w8a16_gemm(const CUtensorMap &tmap_w, const CUtensorMap &tmap_x, const float *scale_b,
                              int per_channel, int64_t M, int64_t N, int64_t K, void *out, uint32_t *err,
                              const DecodePlan &plan, const DecodeWorkspace &ws, const LaunchOpts &opts,
                              cudaStream_t stream) {
    (void)K;
    DecodeArgs a{};
    a.scale_a = nullptr;
    a.scale_b = scale_b;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = err;
    a.counters = ws.counters;
    a.slots = ws.slots;
    a.units = plan.units;
    a.gran = per_channel ? 1 : 0;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.kb_total = plan.kb_total;
    a.n_tiles = plan.n_tiles;
    a.stages = plan.stages;
    a.weights_static = opts.weights_static ? 1 : 0;
    a.split = 0;
    if (plan.tok_pad == 32) return launch_w16<32>(tmap_w, tmap_x, a, plan, opts, stream);
    return launch_w16<16>(tmap_w, tmap_x, a, plan, opts, stream);
}

// The large-M tile kernel's plan: 256 x 128 output tiles, one persistent CTA
// per SM (at most one per unit), 3 weight and 3 token stages (~193 KB).  When
// the tiles' last round would fill at most half of the CTAs, its tiles are
// split into half tiles (128 weight rows each), unless the last weight tile
// has a single half, to keep every unit non-empty.
W16TilePlan plan_w8a16_tile(int64_t M, int64_t N, int64_t K, int num_sms) {
    W16TilePlan p{};
    p.m_tiles = static_cast<int>((M + kW16TileTokens - 1) / kW16TileTokens);
    p.n_tiles = static_cast<int>((N + 2 * kDecodeRows - 1) / (2 * kDecodeRows));
    p.kb_total = static_cast<int>((K + kBlockK - 1) / kBlockK);
    p.tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    const int64_t tail = p.tiles % sms;
    const int64_t last_rows = N - static_cast<int64_t>(p.n_tiles - 1) * 2 * kDecodeRows;
    const bool split = p.tiles > sms && tail > 0 && 2 * tail <= sms && last_rows > kDecodeRows;
    p.full_units = split ? p.tiles - tail : p.tiles;
    p.units = split ? p.tiles + tail : p.tiles;
    p.ctas = static_cast<int>(std::min<int64_t>(p.units, sms));
    p.wstages = 3;
    p.xstages = 3;
    const size_t barriers = 8u * static_cast<size_t>(2 * p.wstages + 2 * p.xstages + 2 + 2 * W16TileCfg::kABufs + 1);
    p.smem_bytes = 1024 + static_cast<size_t>(p.wstages) * W16TileCfg::kWStageBytes +
                   static_cast<size_t>(p.xstages) * W16TileCfg::kXStageBytes + ((barriers + 127) / 128) * 128;
    return p;
}

cudaError_t launch_w8a16_tile(const CUtensorMap &tmap_w, const CUtensorMap &tmap_x, const float *scale_b,
                              int per_channel, int64_t M, int64_t N, void *out, uint32_t *err,
                              const W16TilePlan &plan, const LaunchOpts &opts, cudaStream_t stream) {
    W16TileArgs a{};
    a.scale_b = scale_b;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = err;
    a.per_channel = per_channel;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.kb_total = plan.kb_total;
    a.m_tiles = plan.m_tiles;
    a.full_units = static_cast<int>(plan.full_units);
    a.units = static_cast<int>(plan.units);
    a.wstages = plan.wstages;
    a.xstages = plan.xstages;
    a.weights_static = opts.weights_static ? 1 : 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool attr_done[64] = {};  // benign race: the attribute call is idempotent
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(w8a16_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    return launch_with_opts(w8a16_tile_kernel, dim3(static_cast<unsigned>(plan.ctas)), dim3(W16TileCfg::kThreads),
                            plan.smem_bytes, stream, opts, tmap_w, tmap_x, a);
}

cudaError_t launch_widen_weight(const void *w, const float *scale, int per_channel, int64_t N, int64_t K, void *out,
                                cudaStream_t stream, int num_sms, const LaunchOpts &opts) {
    const int64_t n16 = N * K / 16;
    int64_t blocks = (n16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_with_opts(widen_weight_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, opts,
                            static_cast<const uint4 *>(w), static_cast<uint4 *>(out), scale, per_channel, n16,
                            static_cast<int>(K / 16));
}


template <int MT>
static cudaError_t launch_gemv_mt(const void *W, const void *x, const float *scale_b, int per_channel, int64_t N,
                                  int64_t K, void *out, uint32_t *err, int num_sms, const LaunchOpts &opts,
                                  cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool attr_done[64] = {};  // benign race: the attribute call is idempotent
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(w8a16_gemv_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGemvRingBytes + kGemvBarBytes + kW16GemvMaxXBytes));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    // one CTA per SM (its ring and token copy fill most of the shared
    // memory), no more CTAs than rows
    const int64_t ctas = std::min<int64_t>(static_cast<int64_t>(num_sms > 0 ? num_sms : 1), N);
    const size_t smem = kGemvRingBytes + kGemvBarBytes + static_cast<size_t>(MT) * static_cast<size_t>(K) * 2u;
    return launch_with_opts(w8a16_gemv_kernel<MT>, dim3(static_cast<unsigned>(ctas)), dim3(kGemvThreads), smem,
                            stream, opts, static_cast<const uint8_t *>(W), static_cast<const __nv_bfloat16 *>(x),
                            scale_b, per_channel, static_cast<int>(N), static_cast<int>(K),
                            static_cast<__nv_bfloat16 *>(out), err, opts.weights_static ? 1 : 0);
}

cudaError_t launch_w8a16_gemv(const void *W, const void *x, const float *scale_b, int per_channel, int64_t M,
                              int64_t N, int64_t K, void *out, uint32_t *err, int num_sms, const LaunchOpts &opts,
                              cudaStream_t stream) {
    if (!w8a16_gemv_fits(M, K)) return cudaErrorInvalidValue;
    switch (M) {
        case 1: return launch_gemv_mt<1>(W, x, scale_b, per_channel, N, K, out, err, num_sms, opts, stream);
        case 2: return launch_gemv_mt<2>(W, x, scale_b, per_channel, N, K, out, err, num_sms, opts, stream);
        case 3: return launch_gemv_mt<3>(W, x, scale_b, per_channel, N, K, out, err, num_sms, opts, stream);
        default: return launch_gemv_mt<4>(W, x, scale_b, per_channel, N, K, out, err, num_sms, opts, stream);
    }
}

}  // namespace fp8k
