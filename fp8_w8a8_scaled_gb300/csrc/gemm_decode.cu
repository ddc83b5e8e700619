// gemm_decode.cu -- weight-streaming FP8 W8A8 scaled GEMM for small M (decode).
//
// y[m,n] = bf16( (sum_k A[m,k] * B[n,k]) * sa * sb ), A E4M3 [M,K], B E4M3 [N,K].
// Sources: "The FP8 tower's cuBLASLt default rests on a false premise ..."
// (vllm.cpp #252), "What is owed" items 2-3 (the decode tile, the scale
// epilogue and granularity; small-M M<=16 / M<=32 tiles) and "SETTLED BY PAIRED
// TRACE" (decode GEMMs are weight-bandwidth bound: GiB/s per shape; the
// split-K tile "128x32x128...splitK" and its reduce); "Qwen3.6 NVFP4 baselines
// ..." (vllm.cpp #213), "The 27B gap is now FULLY ATTRIBUTED" (a separate
// split-K reduce kernel costs step time -- here it is fused).
//
// Design (GB300, sm_103a).  At decode M every weight byte is used M times, so
// the kernel is bound by streaming B from HBM once, and every SM must stream
// its equal share all the time.  The work is cut into units of one output tile
// (128 weight rows x a 16- or 32-token tile) by one 128-wide k-block, and
// given out in one of two ways:
//   * cluster mode (enough tiles: N >= ~3840 on 152 SMs): a cluster of S CTAs
//     per tile, CTA r taking k-blocks [r*kb/S, (r+1)*kb/S), with S chosen so
//     the grid is ~1.6 CTAs per SM; the S parts are summed through
//     distributed shared memory (below).  S = 1 (as many tiles as ~1.6 x SMs,
//     or a K range of at most two k-blocks) is whole tiles, nothing to sum;
//   * stream-K (few tiles with long K ranges): a persistent grid of two CTAs
//     per SM gives CTA c the contiguous units [c*U/G, (c+1)*U/G), so all CTAs
//     stream the same number of bytes whatever the shape.
// Inside a CTA:
//   * warp 0 / lane 0 streams the units' 128 x 128-byte weight boxes and the
//     matching token boxes (the M real token rows; the rest of each token tile
//     is zeroed once) with TMA into a ring of shared-memory stages (128-byte
//     swizzle), L2 evict-first for the once-read weights;
//   * warp 1 / lane 0 issues tcgen05.mma kind::f8f6f4 with the WEIGHTS as the
//     128-row A operand and the tokens (padded to 16 or 32) as the N side
//     ("swap-AB").  Each k-block is accumulated from zero into one of several
//     TMEM buffers; tcgen05.commit frees the stage and hands the buffer on;
//   * 4 drain warps read each k-block's fp32 partial out of TMEM while later
//     k-blocks are multiplied, and add it up exactly (below).
// Exact sums (per-tensor, per-channel and per-token scales).  Every product of
// two E4M3 values is an integer multiple of 2^-18, so is any sum of them, and
// the tensor core's binary32 partial of one 128-wide k-block (|p| <= 128 *
// 448^2 < 2^25) keeps that grid whatever it rounds away: p * 2^18 is an
// integer below 2^43.  The drain splits p exactly into a multiple of 32 and a
// remainder and adds both, as integers read from the bits of two binary32 sums
// with magic constants (no conversion instruction), into two 32-bit
// accumulators; a tile's part leaves the drain as one 64-bit integer and parts
// are added as integers.  So the sum over a tile's K range is exact: the same
// however K is divided among CTAs (a merged projection and its pieces, or a
// token in a batch and alone, give the same bits), and the only roundings are
// the tensor core's inside a k-block and the final conversion to binary32.
// Blockwise scaling multiplies every k-block's partial by its own scale
// product, which leaves that grid, so there the drain folds the scaled
// partials into a TwoSum (hi, lo) pair (exact to ~2^-48 relative) and parts are
// added with TwoSum in k order.
// When a tile's K range ends inside the CTA, the drain warps either store the
// tile (scales in binary32, then bf16) or, if other CTAs hold the rest of the
// tile's K range: in cluster mode, store their part of each row into the
// shared memory of the cluster CTA that sums that row, and after one cluster
// barrier every CTA sums its rows over the S parts; in stream-K mode, write
// their part to a workspace slot and count in on the tile's arrival counter (a
// barrier, then one thread's release fence and atomic add); the CTA that
// arrives last acquires, adds all other parts to its own, stores the tile and
// resets the counter.  Which CTAs share the first and last tile of a CTA's
// range, and where their slots are, is worked out while the first loads are in
// flight.  No CTA ever spins on another: the only cross-CTA wait is the
// hardware cluster barrier among the co-scheduled CTAs of one cluster, always
// taken by whole converged warps (its .aligned form).  (Exact sums would allow
// the tile's K range to be handed out at run time through an atomic counter in
// the cluster's shared memory, to let CTAs that share an SM take fewer
// k-blocks; measured slower on QKV, 15.1 against 13.6 us at M = 1.)
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"
#include "splitk.cuh"

namespace fp8k {
namespace {

constexpr uint32_t kWTileBytes = kDecodeRows * kBlockK;  // 16 KB of weights per stage

template <int TOK>
struct DecodeCfg {
    static constexpr int kDrainThreads = 128;  // one warpgroup drains TMEM, all TOK token columns per thread
    static constexpr int kThreads = 64 + kDrainThreads;
    // two CTAs of this kernel plus one of the next (programmatic launch) per SM
    // for the 16-token tile; two per SM for the 32-token tile
    static constexpr int kMinBlocks = TOK <= 16 ? 3 : 2;
    static constexpr int kMaxRegs = (65536 / (kMinBlocks * kThreads)) / 8 * 8;
    // TMEM accumulators in flight between the MMA and the drain (the MMA can
    // run this many k-blocks ahead).  kBufs * TOK columns per CTA.
    static constexpr int kBufs = TOK <= 16 ? 8 : 4;  // must match decode_tmem_bufs()
    static constexpr uint32_t kTmemCols = kBufs * TOK < 32 ? 32 : kBufs * TOK;
    static constexpr uint32_t kATileBytes = TOK * kBlockK;
    static constexpr uint32_t kStageBytes = kWTileBytes + kATileBytes;
    static constexpr uint32_t kIdesc = idesc_e4m3_f32(kDecodeRows, TOK);
};

// The exact split of a k-block partial p (an integer multiple of 2^-18 below
// 2^25 in magnitude).  t = p + kSplitHi (ulp 32 at 1.5 * 2^28) rounds p to a
// multiple of 32, p_hi = t - kSplitHi, and bits(t) - bits(kSplitHi) is p_hi / 32
// as an integer (|.| < 2^20); p_lo = p - p_hi is exact (|p_lo| <= 16, a
// multiple of 2^-18), u = p_lo * 2^18 + kSplitLo (ulp 1 at 1.5 * 2^23) is
// exact, and bits(u) - bits(kSplitLo) is p_lo * 2^18 (|.| <= 2^22).  A part's
// sum is hi * 2^23 + lo in units of 2^-18.
constexpr float kSplitHi = 402653184.0f;  // 1.5 * 2^28
constexpr int kSplitHiBits = 0x4DC00000;
constexpr float kSplitLo = 12582912.0f;   // 1.5 * 2^23
constexpr int kSplitLoBits = 0x4B400000;
constexpr float kFixScale = 262144.0f;    // 2^18
constexpr float kFixScaleInv = 1.0f / 262144.0f;
constexpr long long kPartNaN = static_cast<long long>(0x8000000000000000ull);  // a part holding a NaN

// One exact part (units of 2^-18, or kPartNaN) as binary32.
__device__ __forceinline__ float exact_to_f32(long long v) {
    return v == kPartNaN ? __int_as_float(0x7fffffff) : __fmul_rn(__ll2float_rn(v), kFixScaleInv);
}

// Exact parts in distributed shared memory.
__device__ __forceinline__ void st_cluster_s64(uint32_t addr, long long v) {
    asm volatile("st.shared::cluster.s64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ long long lds_s64(uint32_t addr) {
    long long v;
    asm volatile("ld.shared.s64 %0, [%1];" : "=l"(v) : "r"(addr));
    return v;
}

// kBlk: blockwise scaling (one activation scale per token per k-block, one
// weight scale per 128-row tile per k-block).  Every k-block's partial sum is
// multiplied by its scale product as it leaves TMEM, and the tile's output
// takes no further scale.  Lanes 1..TOK of warp 0 write the scale products of
// each unit into a shared-memory slot beside its TMEM accumulator, up to
// kBufs units ahead of the drain (so the scale loads' latency is hidden), and
// the accumulator's "full" barrier waits for them as well as for the MMA.
// kCluster: the grid is one cluster of `split` CTAs per output tile, CTA r of
// the cluster taking k-blocks [r*kb/S, (r+1)*kb/S) of the tile; the parts are
// summed through distributed shared memory instead of the workspace: every CTA
// stores its part of rows [red_row_begin(q), red_row_begin(q+1)) into CTA q's
// reduction area, one cluster barrier, then CTA q sums its rows over the S
// parts and stores them.
template <int TOK, bool kBlk, bool kCluster>
__global__ void __launch_bounds__(DecodeCfg<TOK>::kThreads) __maxnreg__(DecodeCfg<TOK>::kMaxRegs)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                       const DecodeArgs args) {
    using Cfg = DecodeCfg<TOK>;
    constexpr int NB = Cfg::kBufs;
    constexpr int kSlotElems = TOK * kDecodeRows;  // entries of one partial slot, [token][row]
    constexpr uint32_t kRedEntry = kBlk ? 4u : 8u;  // bytes of one reduction entry (binary32 / exact part)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base, s_issued, s_consumed, s_last;
    // slot offsets (entries) of the K-range parts of this CTA's first and last
    // tile (the only tiles it can share with other CTAs), their counts, and
    // which of them is this CTA's own
    __shared__ int64_t s_slot[2][kMaxFixupSegs];
    __shared__ int s_nseg[2], s_own[2];
    __shared__ volatile uint32_t s_abort;
    __shared__ float s_bscale[kBlk ? NB : 1][TOK];  // blockwise: scale products per accumulator
    __shared__ float s_red_sa[kCluster ? TOK : 1], s_red_sb[kCluster ? kDecodeRows : 1];  // cluster-mode scales

    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stages = args.stages;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bar0 = base + static_cast<uint32_t>(stages) * Cfg::kStageBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (stages + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * stages + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * stages + NB + b); };
    const uint32_t final_bar = bar0 + 8u * (2 * stages + 2 * NB);

    const int64_t G = gridDim.x, U = args.units;
    const int64_t me = blockIdx.x;
    const int S = kCluster ? args.split : 1;
    const int c_rank = kCluster ? static_cast<int>(me % S) : 0;  // == %cluster_ctarank (clusters along x)
    const int64_t u0 = kCluster ? (me / S) * args.kb_total + (static_cast<int64_t>(c_rank) * args.kb_total) / S
                                : unit_begin(me, U, G);
    const int64_t u1 = kCluster ? (me / S) * args.kb_total + (static_cast<int64_t>(c_rank + 1) * args.kb_total) / S
                                : unit_begin(me + 1, U, G);
    const int red_rows = (kDecodeRows + S - 1) / S;  // cluster mode: rows per reduction slot
    // cluster mode: the reduction area, [S parts][TOK tokens][red_rows rows], after the barriers
    const uint32_t red_base = bar0 + ((8u * static_cast<uint32_t>(2 * stages + 2 * NB + 1) + 127u) & ~127u);
    const int iters = static_cast<int>(u1 - u0);
    const int kbt = args.kb_total, n_tiles = args.n_tiles;
    uint32_t *const err = args.err;
    // the token boxes carry the M real rows of the token tile
    const uint32_t stage_bytes = kWTileBytes + static_cast<uint32_t>(args.tok_rows) * kBlockK;

    if (tid == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_a);
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(tfull_bar(b), kBlk ? 2 : 1);  // MMA commit (+ scale writer)
            mbar_init(tempty_bar(b), 4);            // one arrive per drain warp
        }
        mbar_init(final_bar, 1);
        fence_mbar_init();
        s_issued = 0;
        s_consumed = 0;
        s_abort = 0;
    }
    if (warp == 1) tmem_alloc(smem_u32(&s_tmem_base), Cfg::kTmemCols);
    {
        // rows M..TOK-1 of every stage's token tile: zeroed once, never
        // written again (the MMA reads the whole tile)
        const uint32_t pad16 = static_cast<uint32_t>(TOK - args.tok_rows) * (kBlockK / 16);  // 16-byte vectors
        for (uint32_t v = tid; v < static_cast<uint32_t>(stages) * pad16; v += Cfg::kThreads) {
            const uint32_t s = v / pad16, o = v - s * pad16;
            const uint32_t a = base + s * Cfg::kStageBytes + kWTileBytes +
                               static_cast<uint32_t>(args.tok_rows) * kBlockK + 16u * o;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
        }
        fence_proxy_async_smem();  // before the tensor core reads them
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;
    // Cluster mode: a first cluster barrier, waited for before the first store
    // into another CTA's shared memory, so that every CTA of the cluster is
    // known to be running by then.
    if (kCluster && S > 1) cluster_arrive_relaxed();

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------------- producer
        const uint64_t evict_first = policy_evict_first();
        int i = 0;
        // Weights that no earlier kernel in the stream writes may be fetched
        // before the dependency wait; the tokens always wait.
        const int pre = args.weights_static ? min(iters, stages) : 0;
        for (; i < pre; ++i) {
            const int64_t u = u0 + i, t = u / kbt;
            const int kb = static_cast<int>(u - t * kbt), n_tile = static_cast<int>(t % n_tiles);
            mbar_arrive_expect_tx(full_bar(i), stage_bytes);
            tma_load_2d_hint(base + static_cast<uint32_t>(i) * Cfg::kStageBytes, &tmap_w, full_bar(i), kb * kBlockK,
                             n_tile * kDecodeRows, evict_first);
        }
        grid_dependency_wait();
        for (int j = 0; j < pre; ++j) {
            const int64_t u = u0 + j, t = u / kbt;
            const int kb = static_cast<int>(u - t * kbt), m_tile = static_cast<int>(t / n_tiles);
            tma_load_2d(base + static_cast<uint32_t>(j) * Cfg::kStageBytes + kWTileBytes, &tmap_a, full_bar(j),
                        kb * kBlockK, m_tile * TOK);
        }
        int t = static_cast<int>((u0 + i) / kbt), kb = static_cast<int>(u0 + i - static_cast<int64_t>(t) * kbt);
        for (; i < iters; ++i, ++kb) {
            if (kb == kbt) {
                kb = 0;
                ++t;
            }
            const int s = i % stages;
            const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
            if (!cta_wait(empty_bar(s), ph ^ 1u, err, kErrDecodeEmptyWait, &s_abort)) break;
            const int n_tile = t % n_tiles, m_tile = t / n_tiles;
            const uint32_t stage = base + static_cast<uint32_t>(s) * Cfg::kStageBytes;
            mbar_arrive_expect_tx(full_bar(s), stage_bytes);
            tma_load_2d_hint(stage, &tmap_w, full_bar(s), kb * kBlockK, n_tile * kDecodeRows, evict_first);
            tma_load_2d(stage + kWTileBytes, &tmap_a, full_bar(s), kb * kBlockK, m_tile * TOK);
        }
        s_issued = static_cast<uint32_t>(i);
        // Every load of this CTA is issued (and this grid's dependency was
        // waited for above): the next kernel in the stream may now launch, so
        // its prologue and weight prefetch overlap this CTA's drain and fixup.
        grid_launch_dependents();
    } else if (kBlk && warp == 0 && lane >= 1 && lane <= 16) {
        // ---------------------------------------------------------------- scale writer (blockwise)
        constexpr unsigned kMask = 0xFFFFu << 1;  // lanes 1..16, token columns lane-1 (+16)
        grid_dependency_wait();  // the scales may come from the previous kernel
        const int c0 = static_cast<int>(lane) - 1;
        int t = static_cast<int>(u0 / kbt), kb = static_cast<int>(u0 - static_cast<int64_t>(t) * kbt);
        for (int i = 0; i < iters; ++i, ++kb) {
            if (kb == kbt) {
                kb = 0;
                ++t;
            }
            const int b = i % NB;
            const uint32_t tph = static_cast<uint32_t>(i / NB) & 1u;
            const int nt = t % n_tiles, m0 = (t / n_tiles) * TOK;
            const float sbk = __ldg(args.scale_b + static_cast<int64_t>(nt) * kbt + kb);
            float sak[TOK / 16];
#pragma unroll
            for (int j = 0; j < TOK / 16; ++j) {
                const int m = m0 + c0 + 16 * j;
                sak[j] = m < args.M ? __ldg(args.scale_a + static_cast<int64_t>(m) * kbt + kb) : 0.0f;
            }
            uint32_t ok = 1;
            if (lane == 1) ok = cta_wait(tempty_bar(b), tph ^ 1u, err, kErrDecodeTmemEmptyWait, &s_abort) ? 1u : 0u;
            ok = __shfl_sync(kMask, ok, 1);
            if (!ok) break;
#pragma unroll
            for (int j = 0; j < TOK / 16; ++j) s_bscale[b][c0 + 16 * j] = __fmul_rn(sak[j], sbk);
            __syncwarp(kMask);  // every lane's slot write before lane 1's (release) arrival
            if (lane == 1) mbar_arrive(tfull_bar(b));
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        int i = 0;
        for (; i < iters; ++i) {
            const int s = i % stages;
            const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
            const int b = i % NB;
            const uint32_t tph = static_cast<uint32_t>(i / NB) & 1u;
            if (!cta_wait(full_bar(s), ph, err, kErrDecodeFullWait, &s_abort)) break;
            if (!cta_wait(tempty_bar(b), tph ^ 1u, err, kErrDecodeTmemEmptyWait, &s_abort)) break;
            tc_fence_after();
            const uint32_t w_addr = base + static_cast<uint32_t>(s) * Cfg::kStageBytes;
            const uint64_t dw = sw128_kmajor_desc(w_addr), da = sw128_kmajor_desc(w_addr + kWTileBytes);
            const uint32_t d = tmem + static_cast<uint32_t>(b * TOK);
#pragma unroll
            for (int kk = 0; kk < kBlockK / 32; ++kk)  // +32 bytes along K = +2 in the address field
                mma_e4m3(d, dw + 2u * kk, da + 2u * kk, Cfg::kIdesc, kk > 0 ? 1u : 0u);
            mma_commit(empty_bar(s));
            mma_commit(tfull_bar(b));
        }
        s_consumed = static_cast<uint32_t>(i);
        mma_commit(final_bar);  // arrives when every MMA issued above has completed
    } else if (warp >= 2) {
        // ---------------------------------------------------------------- drain + tile output
        grid_dependency_wait();  // outputs, scales and the workspace are touched below
        const uint32_t quarter = warp & 3u;          // a warp reaches TMEM lanes 32*(warp%4) .. +31
        const int row = static_cast<int>(quarter * 32u + lane);  // weight row within the tile
        const bool sa_vec = !kBlk && (args.gran == 2 || args.gran == 3);
        const bool sb_vec = !kBlk && (args.gran == 1 || args.gran == 2);
        const float sa0 = kBlk ? 1.0f : __ldg(args.scale_a), sb0 = kBlk ? 1.0f : __ldg(args.scale_b);
        const int t_first_me = static_cast<int>(u0 / kbt);
        if (!kCluster && tid == 64 && iters > 0) {
            // Which CTAs hold the other parts of this CTA's first and last tile
            // and where their partial sums go, worked out while the first
            // loads are in flight.
            for (int w = 0; w < 2; ++w) {
                const int64_t t = (w == 0 ? u0 : u1 - 1) / kbt, tile_u0 = t * kbt;
                const int64_t c_first = unit_owner(tile_u0, U, G), c_last = unit_owner(tile_u0 + kbt - 1, U, G);
                const int nseg = static_cast<int>(c_last - c_first + 1);
                s_nseg[w] = nseg;
                s_own[w] = static_cast<int>(me - c_first);
                for (int j = 0; j < kMaxFixupSegs && j < nseg; ++j) {
                    const int64_t cc = c_first + j;
                    s_slot[w][j] = (2 * cc + (t == unit_begin(cc, U, G) / kbt ? 0 : 1)) * kSlotElems;
                }
            }
        }
        // this CTA's part of the current tile: exact (hi[c] * 2^23 + lo[c] units
        // of 2^-18) or, blockwise, a TwoSum pair (hi, lo as binary32 bits)
        int hi[TOK], lo[TOK];
        uint32_t nan_cols = 0;  // exact sums: token columns whose sum met a NaN
#pragma unroll
        for (int c = 0; c < TOK; ++c) hi[c] = lo[c] = 0;

        int t = t_first_me, kb = static_cast<int>(u0 - static_cast<int64_t>(t) * kbt);
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
                if (!kBlk && c0 + 16 >= TOK) {  // last chunk read: the buffer is free for the MMA again
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar(b));
                }
                if constexpr (kBlk) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float h = __int_as_float(hi[c0 + j]), l = __int_as_float(lo[c0 + j]);
                        two_sum_acc(h, l, __fmul_rn(__uint_as_float(r[j]), s_bscale[b][c0 + j]));
                        hi[c0 + j] = __float_as_int(h);
                        lo[c0 + j] = __float_as_int(l);
                    }
                } else {
                    float chk = 0.0f;  // NaN iff some partial of the chunk is NaN (none is infinite)
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float p = __uint_as_float(r[j]);
                        chk = __fadd_rn(chk, p);
                        const float tt = __fadd_rn(p, kSplitHi);
                        const float uu = __fmaf_rn(__fsub_rn(p, __fsub_rn(tt, kSplitHi)), kFixScale, kSplitLo);
                        hi[c0 + j] += __float_as_int(tt) - kSplitHiBits;
                        lo[c0 + j] += __float_as_int(uu) - kSplitLoBits;
                    }
                    if (chk != chk) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (__uint_as_float(r[j]) != __uint_as_float(r[j])) nan_cols |= 1u << (c0 + j);
                    }
                }
            }
            if constexpr (kBlk) {  // TMEM and the scale slot both free: the writer may refill it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(b));
            } else if ((kb & 255) == 255) {
                // lo grows by at most 2^22 a k-block: carry it into hi every
                // 256 k-blocks (hi grows by less than 2^20 a k-block, and a
                // tile has fewer than kExactMaxKb of them)
#pragma unroll
                for (int c = 0; c < TOK; ++c) {
                    const int q = lo[c] >> 23;
                    hi[c] += q;
                    lo[c] -= q * (1 << 23);
                }
            }

            if (kb != kbt - 1 && i != iters - 1) continue;

            // ---- this CTA's part of tile t ends here
            const int n_tile = t % n_tiles, m_tile = t / n_tiles;
            const int n = n_tile * kDecodeRows + row;
            const int m0 = m_tile * TOK;
            const int mt = min(TOK, args.M - m0);
            const int64_t tile_u0 = static_cast<int64_t>(t) * kbt;
            const bool whole = (u0 <= tile_u0) && (kb == kbt - 1);
            // the part of each token column: exact (units of 2^-18, or
            // kPartNaN), or the TwoSum pair rounded once to binary32
            long long part[TOK];
#pragma unroll
            for (int c = 0; c < TOK; ++c) {
                if constexpr (kBlk)
                    part[c] = __float_as_int(__fadd_rn(__int_as_float(hi[c]), __int_as_float(lo[c])));
                else
                    part[c] = ((nan_cols >> c) & 1u) ? kPartNaN
                                                     : static_cast<long long>(hi[c]) * (1ll << 23) + lo[c];
            }
            bool store = whole;
            if (kCluster && !whole) {
                // this CTA's part into the reduction area of the CTA that sums this row
                __syncwarp();    // (an aligned cluster barrier needs a converged warp)
                cluster_wait();  // (the drain warps' half of the first cluster barrier)
                const int q = (row * S) / kDecodeRows;
                const int lr = row - red_row_begin(q, S);
                const uint32_t dst = map_to_rank(
                    red_base + kRedEntry * static_cast<uint32_t>((c_rank * TOK) * red_rows + lr),
                    static_cast<uint32_t>(q));
#pragma unroll
                for (int c = 0; c < TOK; ++c) {
                    if (c < mt) {
                        const uint32_t a = dst + kRedEntry * static_cast<uint32_t>(c * red_rows);
                        if constexpr (kBlk)
                            st_cluster_f32(a, __int_as_float(static_cast<int>(part[c])));
                        else
                            st_cluster_s64(a, part[c]);
                    }
                }
            } else if (!kCluster && !whole) {
                const int w = (t == t_first_me) ? 0 : 1;
                if constexpr (kBlk) {
                    float *mine = args.slots + static_cast<int64_t>(2 * me + w) * kSlotElems;
#pragma unroll
                    for (int c = 0; c < TOK; ++c)
                        if (c < mt) mine[c * kDecodeRows + row] = __int_as_float(static_cast<int>(part[c]));
                } else {
                    long long *mine = reinterpret_cast<long long *>(args.slots) +
                                      static_cast<int64_t>(2 * me + w) * kSlotElems;
#pragma unroll
                    for (int c = 0; c < TOK; ++c)
                        if (c < mt) __stcg(mine + c * kDecodeRows + row, part[c]);
                }
                // Arrival: the barrier orders every drain thread's slot writes
                // before tid 64's release fence and count (the usual
                // barrier + single-thread release pattern); the last of the
                // tile's parts to arrive acquires and sums them all.
                named_barrier_sync(1, Cfg::kDrainThreads);
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
                    if constexpr (kBlk) {
                        // sum the tile over its K range in k order (this CTA's
                        // own part is read back from its slot like the others)
                        const int entries = mt * kDecodeRows;  // [col][row], valid token columns only
                        const int dt = static_cast<int>(tid) - 64;
                        fixup_sum<kMaxFixupSegs, 1, Cfg::kDrainThreads>(args, s_slot[w], nseg, entries, dt, n_tile, m0,
                                                                         sa_vec, sb_vec, sa0, sb0);
                    } else {
                        // every other part of this thread's row added to its
                        // own (integers: the order does not matter)
                        const int own = s_own[w];
                        for (int j = 0; j < nseg; ++j) {
                            if (j == own) continue;
                            const long long *pp = reinterpret_cast<const long long *>(args.slots) + s_slot[w][j] + row;
                            long long v[TOK];
#pragma unroll
                            for (int c = 0; c < TOK; ++c) v[c] = c < mt ? __ldcg(pp + c * kDecodeRows) : 0;
#pragma unroll
                            for (int c = 0; c < TOK; ++c)
                                part[c] = (part[c] == kPartNaN || v[c] == kPartNaN) ? kPartNaN : part[c] + v[c];
                        }
                        store = true;
                    }
                    if (tid == 64) args.counters[t] = 0u;  // ready for the next launch
                }
            }
            if (store && n < args.N) {
                const float sb = sb_vec ? __ldg(args.scale_b + n) : sb0;
#pragma unroll
                for (int c = 0; c < TOK; ++c) {
                    if (c < mt) {
                        const float acc = kBlk ? __int_as_float(static_cast<int>(part[c])) : exact_to_f32(part[c]);
                        const float sa = sa_vec ? __ldg(args.scale_a + m0 + c) : sa0;
                        args.out[static_cast<int64_t>(m0 + c) * args.N + n] =
                            __float2bfloat16_rn(__fmul_rn(__fmul_rn(acc, sa), sb));
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < TOK; ++c) hi[c] = lo[c] = 0;
            nan_cols = 0;
        }
    }
    __syncwarp();
    grid_dependency_wait();
    // (The producer thread triggered the dependent launch after its last load;
    // a grid only triggers after its own dependency wait, so at most one
    // dependent grid is ever waiting.)
    grid_launch_dependents();
    __syncthreads();

    if constexpr (kCluster) {
        if (S > 1) {
            const int tile = static_cast<int>(me / S);
            const int rb = red_row_begin(c_rank, S), nr = red_row_begin(c_rank + 1, S) - rb;
            const int mt = min(TOK, args.M);
            if (warp >= 2) {
                // the scales of this CTA's rows and of the tokens, staged in
                // shared memory while the other CTAs of the cluster finish
                const int dt = static_cast<int>(tid) - 64;
                const bool sa_vec = !kBlk && (args.gran == 2 || args.gran == 3);
                const bool sb_vec = !kBlk && (args.gran == 1 || args.gran == 2);
                if (dt < mt) s_red_sa[dt] = kBlk ? 1.0f : __ldg(args.scale_a + (sa_vec ? dt : 0));
                const int n = tile * kDecodeRows + rb + dt;
                if (dt < nr) s_red_sb[dt] = kBlk ? 1.0f : __ldg(args.scale_b + (sb_vec && n < args.N ? n : 0));
            }
            __syncwarp();  // (an aligned cluster barrier needs a converged warp)
            if (warp < 2) cluster_wait();  // the other warps' half of the first cluster barrier
            // every part of every row this CTA sums has landed (and no CTA of
            // the cluster touches another's shared memory after this point)
            cluster_sync();
            {
                // Every thread of the CTA (the producer and MMA warps are done
                // too) takes one of this CTA's rows and every g-th token
                // column; consecutive threads: consecutive channels.
                const int groups = Cfg::kThreads / nr;  // nr <= 64 < kThreads
                const int lr = static_cast<int>(tid) % nr, m0 = static_cast<int>(tid) / nr;
                const int n = tile * kDecodeRows + rb + lr;
                if (m0 < groups && n < args.N) {
                    const float sb = s_red_sb[lr];
                    __nv_bfloat16 *o = args.out + static_cast<int64_t>(m0) * args.N + n;
                    const int64_t ostep = static_cast<int64_t>(groups) * args.N;
#pragma unroll 4
                    for (int m = m0; m < mt; m += groups, o += ostep) {
                        float acc;
                        if constexpr (kBlk) {
                            float v[kMaxClusterParts];
#pragma unroll
                            for (int src = 0; src < kMaxClusterParts; ++src)
                                if (src < S)
                                    v[src] = lds_f32(red_base + 4u * static_cast<uint32_t>((src * TOK + m) * red_rows + lr));
                            float h = 0.0f, l = 0.0f;
#pragma unroll
                            for (int src = 0; src < kMaxClusterParts; ++src)
                                if (src < S) two_sum_acc(h, l, v[src]);
                            acc = __fadd_rn(h, l);
                        } else {
                            long long v[kMaxClusterParts];
#pragma unroll
                            for (int src = 0; src < kMaxClusterParts; ++src)
                                if (src < S)
                                    v[src] = lds_s64(red_base + 8u * static_cast<uint32_t>((src * TOK + m) * red_rows + lr));
                            long long sum = 0;
                            bool nan = false;
#pragma unroll
                            for (int src = 0; src < kMaxClusterParts; ++src) {
                                if (src < S) {
                                    nan |= v[src] == kPartNaN;
                                    sum += v[src];
                                }
                            }
                            acc = exact_to_f32(nan ? kPartNaN : sum);
                        }
                        *o = __float2bfloat16_rn(__fmul_rn(__fmul_rn(acc, s_red_sa[m]), sb));
                    }
                }
            }
        }
    }

    if (tid == 0) {
        // Loads issued but never consumed (only after a timeout): let them land
        // before the CTA exits.
        const uint32_t issued = s_issued, consumed = s_consumed;
        for (uint32_t i = consumed; i < issued; ++i)
            mbar_wait(full_bar(static_cast<int>(i % stages)), (i / stages) & 1u, err, kErrDecodeFullWait);
    }
    if (warp == 1) {
        mbar_wait(final_bar, 0, err, kErrDecodeAccumWait);  // every MMA has completed
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

template <int TOK, bool kBlk, bool kCluster>
cudaError_t launch_tok(const CUtensorMap &tw, const CUtensorMap &ta, const DecodeArgs &a, const DecodePlan &p,
                       const LaunchOpts &o, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool attr_done[64] = {};  // benign race: the attribute call is idempotent
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(decode_gemm_kernel<TOK, kBlk, kCluster>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 200 * 1024);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    LaunchOpts oc = o;
    oc.cluster_x = kCluster ? p.split : 1;
    return launch_with_opts(decode_gemm_kernel<TOK, kBlk, kCluster>, dim3(static_cast<unsigned>(p.ctas)),
                            dim3(DecodeCfg<TOK>::kThreads), p.smem_bytes, stream, oc, tw, ta, a);
}

}  // namespace

// TMEM accumulators of the decode kernel for a token tile (DecodeCfg::kBufs).
static int decode_tmem_bufs(int tok) { return tok <= 16 ? 8 : 4; }

// Shared memory one CTA needs: the 1024-byte alignment slack, `stages` stages
// of weights + tokens, the mbarriers (full/empty per stage, full/empty per
// TMEM accumulator, one final) rounded up to 128 bytes, and in cluster mode
// (split > 1) the reduction area of S parts x tok tokens x ceil(128/S) rows of
// 8-byte exact parts (4-byte binary32 parts for blockwise scaling).
static size_t decode_smem_bytes(int tok, int stages, int split, bool blockwise) {
    const size_t barriers = 8u * static_cast<size_t>(2 * stages + 2 * decode_tmem_bufs(tok) + 1);
    const size_t entry = blockwise ? 4u : 8u;
    const size_t red = split > 1 ? entry * static_cast<size_t>(split) * tok * ((kDecodeRows + split - 1) / split) : 0;
    return 1024 + static_cast<size_t>(stages) * (kDecodeRows * kBlockK + tok * kBlockK) + ((barriers + 127) / 128) * 128 +
           red;
}

// Cluster mode: S = (8 * SMs / 5) / tiles CTAs per tile (at least 1, at most
// the tile's k-blocks), used when S <= kMaxClusterSplit; with fewer tiles (a
// long K range over few channels) the persistent stream-K grid keeps every SM
// streaming.  The grid is kept near 1.6 CTAs per SM because of how clusters
// are placed: on the QKV shape (80 tiles) 3-CTA clusters (240 CTAs) took 13.7
// us per launch and 4-CTA ones (320 CTAs) 22 us, the latter leaving SMs idle
// and starting some clusters only after others had finished; on N 5120 (40
// tiles) 6-CTA clusters took 12.0 us and 8-CTA ones 19.4 us.  (A persistent
// grid of one CTA per SM with a deeper ring, sized so the next launch's CTA
// fits beside it, was measured slower on QKV: 19.3 us, each CTA taking ~0.6 us
// per 16 KB weight box; two per SM under stream-K, 16.6 us, most of the
// difference being the workspace fix-up at the end.)
constexpr int kMaxClusterSplit = kMaxClusterParts;

DecodePlan plan_decode(int64_t M, int64_t N, int64_t K, int num_sms, bool blockwise) {
    DecodePlan p{};
    p.tok_pad = M <= 16 ? 16 : 32;
    p.exact = blockwise ? 0 : 1;
    p.stages = 3;  // ~55-85 KB: two CTAs of this kernel and one of the next fit on an SM
    p.n_tiles = static_cast<int>((N + kDecodeRows - 1) / kDecodeRows);
    p.m_tiles = static_cast<int>((M + p.tok_pad - 1) / p.tok_pad);
    p.kb_total = static_cast<int>((K + kBlockK - 1) / kBlockK);
    p.units = static_cast<int64_t>(p.n_tiles) * p.m_tiles * p.kb_total;
    int64_t split = (8 * static_cast<int64_t>(num_sms) / 5) / p.n_tiles;
    if (split < 1) split = 1;
    if (split > p.kb_total) split = p.kb_total;
    // a K range of one or two k-blocks: whole tiles (the cluster barrier and
    // exchange cost more than the second k-block; 4 x 512 x 256: 4.3 -> 3.7
    // us per call, while at four k-blocks the split still wins, 4.1 vs 4.7)
    if (p.kb_total <= 2) split = 1;
    if (p.m_tiles == 1 && split <= kMaxClusterSplit) {
        p.split = static_cast<int>(split);
        p.ctas = static_cast<int>(static_cast<int64_t>(p.n_tiles) * split);
        p.smem_bytes = decode_smem_bytes(p.tok_pad, p.stages, p.split, blockwise);
        return p;
    }
    p.split = 0;
    p.smem_bytes = decode_smem_bytes(p.tok_pad, p.stages, 0, blockwise);
    // Two persistent CTAs per SM, each with the same number of units (+-1),
    // and at least kb_total / (kMaxFixupSegs - 1) units each, so that no more
    // than kMaxFixupSegs CTAs share one tile.
    const int64_t min_units = (p.kb_total + kMaxFixupSegs - 2) / (kMaxFixupSegs - 1);
    int64_t ctas = 2 * static_cast<int64_t>(num_sms);
    if (ctas > p.units / min_units) ctas = p.units / min_units;
    if (ctas < 1) ctas = 1;
    p.ctas = static_cast<int>(ctas);
    return p;
}

size_t decode_counters_needed(const DecodePlan &p) {
    return p.split > 0 ? 0 : static_cast<size_t>(p.n_tiles) * p.m_tiles;
}

size_t decode_slot_floats(const DecodePlan &p) {
    const size_t per_entry = p.exact ? 2u : 1u;  // exact parts are 64-bit integers: two floats' room
    return p.split > 0 ? 0 : per_entry * 2u * static_cast<size_t>(p.ctas) * static_cast<size_t>(p.tok_pad) * kDecodeRows;
}

cudaError_t launch_decode_gemm(const CUtensorMap &tmap_w, const CUtensorMap &tmap_a, const float *scale_a,
                               const float *scale_b, int granularity, int64_t M, int64_t N, int64_t K, void *out,
                               uint32_t *err, const DecodePlan &plan, const DecodeWorkspace &ws,
                               const LaunchOpts &opts, cudaStream_t stream) {
    (void)K;
    DecodeArgs a;
    a.scale_a = scale_a;
    a.scale_b = scale_b;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = err;
    a.counters = ws.counters;
    a.slots = ws.slots;
    a.units = plan.units;
    a.gran = granularity;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.kb_total = plan.kb_total;
    a.n_tiles = plan.n_tiles;
    a.stages = plan.stages;
    a.weights_static = opts.weights_static ? 1 : 0;
    a.split = plan.split;
    a.tok_rows = static_cast<int>(std::min<int64_t>(M, plan.tok_pad));
    const bool blk = granularity == kGranBlock128;
    if (plan.exact != (blk ? 0 : 1)) return cudaErrorInvalidValue;  // a plan made for the other kind of scales
    if (plan.tok_pad == 32) {
        if (plan.split > 0)
            return blk ? launch_tok<32, true, true>(tmap_w, tmap_a, a, plan, opts, stream)
                       : launch_tok<32, false, true>(tmap_w, tmap_a, a, plan, opts, stream);
        return blk ? launch_tok<32, true, false>(tmap_w, tmap_a, a, plan, opts, stream)
                   : launch_tok<32, false, false>(tmap_w, tmap_a, a, plan, opts, stream);
    }
    if (plan.split > 0)
        return blk ? launch_tok<16, true, true>(tmap_w, tmap_a, a, plan, opts, stream)
                   : launch_tok<16, false, true>(tmap_w, tmap_a, a, plan, opts, stream);
    return blk ? launch_tok<16, true, false>(tmap_w, tmap_a, a, plan, opts, stream)
               : launch_tok<16, false, false>(tmap_w, tmap_a, a, plan, opts, stream);
}

}  // namespace fp8k
