// gemm_prefill.cu -- FP8 W8A8 scaled GEMM for large M (prefill).
//
// y[m,n] = bf16( (sum_k A[m,k] * B[n,k]) * sa * sb ), A E4M3 [M,K] (tokens),
// B E4M3 [N,K] (weights), per-tensor / per-token sa, per-tensor / per-channel sb.
// Sources: "[Kernel] add Flashinfer cutedsl w4a16 linear" (vllm #53014), the
// commit message on the large-M dequant + 16-bit GEMM dispatch (at prefill M
// the GEMM is compute-bound, so a dense tensor-core tile wins there); "We emit
// F32 where vLLM emits bf16 on the biggest prefill buffers ..." (vllm.cpp
// #417), FINDING 1 (the prefill outputs are the largest activation buffers and
// must be written as bf16, not F32).
//
// Design (GB300, sm_103a).  At prefill M every weight byte feeds >= 128 tokens
// and the kernel is bound by the FP8 tensor-core rate.  Above 128 tokens the
// CTAs work in pairs (thread-block clusters of two, cta_group::2 MMAs of 256
// tokens x 256 channels issued by the pair's leader, each CTA loading its own
// 128 tokens and 128 channels per stage: half the weight bytes per SM of a
// one-CTA 128 x 256 tile; measured 1-3% faster, the kernel being bound by the
// tensor pipe under the power cap rather than by its loads); at most 128
// tokens, single CTAs.  One persistent CTA per
// SM walks the 128-token x 256-channel output tiles t = blockIdx.x + i*gridDim.x
// (128-channel tiles when M is small and 256-channel ones would leave most SMs
// idle: there the time goes into streaming the weights, and twice the CTAs
// stream them twice as fast)
// (token tile fastest, so the CTAs resident at one time share their weight
// rows through L2 and the whole token matrix stays L2-resident).  When the
// tiles' last round would fill at most half of the SMs, its tiles run as two
// 128-channel halves each (N = 128 MMAs into the half's accumulator columns),
// on twice as many CTAs:
//   * warp 0 / lane 0 loads, per 128-byte k-block, the 128 x 128-byte token box
//     and the weight boxes (128 x 128 bytes each, one per 128 channels of the
//     tile) with TMA (128-byte swizzle) into a ring of 48 KB shared-memory
//     stages;
//   * warp 1 / lane 0 issues four tcgen05.mma kind::f8f6f4 (M=128, N=256, K=32)
//     per k-block.  A tile's K range is cut into groups of kPrefillDrainKb
//     k-blocks; each group accumulates from zero into one of two 256-column
//     TMEM accumulators, so the MMAs of one group overlap the epilogue's work
//     on the previous one;
//   * warps 2..9 are the epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (one
//     token row per thread) and half of the 256 columns, adds each group's
//     partial sums into binary32 registers, and at the end of the tile applies
//     the scales in binary32 ((acc * sa) * sb), rounds to bf16, writes its
//     row into the half's 16 KB staging box in shared memory (128 rows x 64
//     columns, 128-byte swizzle) and one thread of the half stores the box
//     with a TMA bulk tensor store (coalesced, asynchronous, clipped to M and
//     N), so the epilogue goes back to draining the next tile at once (plain
//     16-byte stores of 32 rows per warp instruction cost 12% of the kernel).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

#include <algorithm>

namespace fp8k {
namespace {

constexpr int kPrefillThreads = 64 + 256;  // producer warp, MMA warp, 8 epilogue warps
constexpr int kPrefillEpiWarps = 8;
constexpr uint32_t kPrefillATile = kPrefillBM * kBlockK;  // 16 KB of tokens per stage
// The output tile is 128 tokens x BN channels, BN = 256 (the largest MMA N) or
// 128 (twice the CTAs for small M, whose time goes into streaming weights).
// kPair: a CTA pair (cta_group::2) computes a 256-token x 256-channel tile;
// each CTA loads its own 128 tokens and 128 of the channels per stage.
template <int BN, bool kPair = false>
struct PrefillCfg {
    static constexpr uint32_t kBTile = (kPair ? 128 : BN) * kBlockK;  // weights per stage
    static constexpr uint32_t kStageBytes = kPrefillATile + kBTile;
    static constexpr uint32_t kTmemCols = 2 * BN;                      // two accumulators
    static constexpr uint32_t kIdesc = idesc_e4m3_f32(kPair ? 2 * kPrefillBM : kPrefillBM, BN);
    static constexpr int kStages = kPair ? 6 : (BN == 256 ? 4 : 6);    // 192 KB of stages
    static constexpr int kTileM = kPair ? 2 * kPrefillBM : kPrefillBM; // tokens per output tile
};
// Output staging: one 128-row x 64-column bf16 box (128-byte swizzle) per
// epilogue half.
constexpr uint32_t kPrefillOutBox = kPrefillBM * 128;
// k-blocks (of 128) the tensor core accumulates in TMEM before the epilogue
// adds the partial sum into fp32 registers.  The tensor core's accumulation is
// less exact than binary32 round-to-nearest over many MMAs: on prefill-chunk
// data (M 2048, N 10240, K 5120) one accumulation over all 160 MMAs left 5 of
// 2.1e7 outputs beyond the acceptance bound (max 1.25 of it), groups of 20
// k-blocks reached 0.87 of it and groups of 10 k-blocks 0.49 (bf16 rounding
// alone: 0.39), for about 3% of the throughput of one accumulation.  At small
// M the kernel is bound by streaming the weights, not by the tensor core, and
// draining more often costs little (only the warps holding valid token rows
// read TMEM); there the weights may be uniformly random codes, whose partial
// sums are large next to the bound (groups of 10 k-blocks: 1.95 of it on the
// 32-token decode data, groups of 2: 0.54), so M <= kPrefillSmallM drains
// every kPrefillDrainKbSmall k-blocks.
constexpr int kPrefillDrainKb = 10;
constexpr int kPrefillDrainKbSmall = 2;
constexpr int64_t kPrefillSmallM = 128;

struct PrefillArgs {
    const float *scale_a;
    const float *scale_b;
    __nv_bfloat16 *out;
    uint32_t *err;
    int gran, M, N, kb_total, m_tiles, full_units, units, stages, drain_kb;
};

// Bounded wait of one thread; gives up at once once the CTA has given up.
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, uint32_t *err, uint32_t code,
                                        volatile uint32_t *abort) {
    if (*abort) return false;
    if (mbar_wait(bar, parity, err, code)) return true;
    *abort = 1u;
    return false;
}

// The same wait taken by lane 0 for the whole warp: the warp's control flow
// stays uniform, which tcgen05.ld (a .sync.aligned instruction) requires.
__device__ __forceinline__ bool pf_warp_wait(uint32_t bar, uint32_t parity, uint32_t *err, uint32_t code,
                                             volatile uint32_t *abort, uint32_t lane) {
    uint32_t ok = 0;
    if (lane == 0) ok = pf_wait(bar, parity, err, code, abort) ? 1u : 0u;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat16 a = __float2bfloat16_rn(lo), b = __float2bfloat16_rn(hi);
    return static_cast<uint32_t>(__bfloat16_as_ushort(a)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// kBlk: blockwise scaling.  The K range is drained after every k-block
// (drain_kb == 1) and each k-block's partial sum is multiplied by its scale
// product sa[m, kb] * sb[n / 128, kb] as it is added into the registers; the
// tile's output then takes no further scale.
// kPair: clusters of two CTAs; rank 0 (the leader) issues cta_group::2 MMAs
// of M = 256 tokens (its 128 and the peer's 128) x N = 256 channels (its
// 128 and the peer's 128), whose accumulator rows land in each CTA's own
// TMEM.  Both CTAs' loads signal the leader's full barrier; the leader's
// commits arrive on both CTAs' barriers (multicast); both CTAs' epilogues
// arrive on the leader's accumulator-empty barrier.
template <int BN, bool kBlk, bool kPair>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_out, const PrefillArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base, s_issued, s_consumed;
    __shared__ volatile uint32_t s_abort;

    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stages = args.stages;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    using Cfg = PrefillCfg<BN, kPair>;
    constexpr int kTileM = Cfg::kTileM;
    const uint32_t staging = base + static_cast<uint32_t>(stages) * Cfg::kStageBytes;  // 2 output boxes
    const uint32_t bar0 = staging + 2u * kPrefillOutBox;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (stages + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * stages + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * stages + 2 + b); };
    const uint32_t final_bar = bar0 + 8u * (2 * stages + 4);

    const int kbt = args.kb_total, m_tiles = args.m_tiles, units = args.units, dkb = args.drain_kb;
    // the pair's rank (0 = leader) and its cluster index among the clusters
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const int G = static_cast<int>(kPair ? gridDim.x / 2 : gridDim.x);
    const int c = static_cast<int>(kPair ? blockIdx.x / 2 : blockIdx.x);
    const bool leader = !kPair || rank == 0;
    uint32_t *const err = args.err;
    // Unit u (u = c, c + G, ...): units below full_units are whole tiles
    // (halves = 3), the rest 128-channel halves of the last tiles, two per
    // tile (halves = 1 or 2; only with BN = 256).  A half that starts at or
    // beyond N is dropped.  Token tile fastest.
    auto unit_of = [&](int u, int &m_tile, int &n_tile, uint32_t &halves) {
        int t = u;
        halves = 3u;
        if (u >= args.full_units) {
            const int v = u - args.full_units;
            t = args.full_units + (v >> 1);
            halves = 1u << (v & 1);
        }
        m_tile = t % m_tiles;
        n_tile = t / m_tiles;
        if (!kPair && BN == 256 && n_tile * BN + 128 >= args.N) halves &= 1u;
    };

    if (tid == 0) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
        tma_prefetch_desc(&tmap_out);
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), kPair ? 2 * kPrefillEpiWarps : kPrefillEpiWarps);  // per epilogue warp
        }
        mbar_init(final_bar, 1);
        fence_mbar_init();
        s_issued = 0;
        s_consumed = 0;
        s_abort = 0;
    }
    if (warp == 1) {
        if constexpr (kPair)
            tmem_alloc_pair(smem_u32(&s_tmem_base), Cfg::kTmemCols);
        else
            tmem_alloc(smem_u32(&s_tmem_base), Cfg::kTmemCols);
    }
    tc_fence_before();
    if constexpr (kPair)
        cluster_sync();  // both CTAs' barriers initialised before any remote arrive or commit
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------------- producer
        grid_dependency_wait();  // the tokens (and possibly the weights) come from earlier kernels
        uint32_t it = 0;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int u = c; u < units && ok; u += G) {
            int m_tile, n_tile;
            uint32_t halves;
            unit_of(u, m_tile, n_tile, halves);
            const uint32_t bytes =
                kPair ? 2u * Cfg::kStageBytes  // both CTAs' boxes, on the leader's barrier
                      : kPrefillATile + (BN == 256 ? static_cast<uint32_t>(__popc(halves)) * 128u * kBlockK : Cfg::kBTile);
            for (int kb = 0; kb < kbt; ++kb) {
                if (!pf_wait(empty_bar(s), ph ^ 1u, err, kErrPrefillEmptyWait, &s_abort)) {
                    ok = false;
                    break;
                }
                const uint32_t stage = base + static_cast<uint32_t>(s) * Cfg::kStageBytes;
                if (leader) mbar_arrive_expect_tx(full_bar(s), bytes);
                if constexpr (kPair) {
                    const uint32_t fb = map_to_rank(full_bar(s), 0);  // the leader's barrier
                    tma_load_2d_pair(stage, &tmap_a, fb, kb * kBlockK, m_tile * kTileM + static_cast<int>(rank) * 128);
                    tma_load_2d_pair(stage + kPrefillATile, &tmap_b, fb, kb * kBlockK,
                                     n_tile * BN + static_cast<int>(rank) * 128);
                } else {
                    tma_load_2d(stage, &tmap_a, full_bar(s), kb * kBlockK, m_tile * kPrefillBM);
                    for (int h = 0; h < BN / 128; ++h)  // 128-channel weight boxes
                        if ((halves >> h) & 1u)
                            tma_load_2d(stage + kPrefillATile + static_cast<uint32_t>(h) * 128u * kBlockK, &tmap_b,
                                        full_bar(s), kb * kBlockK, n_tile * BN + 128 * h);
                }
                ++it;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        s_issued = it;
        grid_launch_dependents();
    } else if (warp == 1 && lane == 0 && leader) {
        // ---------------------------------------------------------------- MMA issuer
        // Each tile's K range is cut into groups of drain_kb k-blocks; every
        // group accumulates from zero into the next TMEM accumulator (two in
        // rotation) and is handed to the epilogue, which adds it into fp32
        // registers.
        uint32_t it = 0;
        int s = 0;
        uint32_t ph = 0;
        uint32_t dc = 0;  // groups issued so far (accumulator = dc & 1)
        bool ok = true;
        for (int u = c; u < units && ok; u += G) {
            int m_tile, n_tile;
            uint32_t halves;
            unit_of(u, m_tile, n_tile, halves);
            // a half unit: N = 128 MMAs on its weight box, into its half of the accumulator
            const uint32_t hoff = (halves == 2u) ? 128u : 0u;
            const uint32_t idesc = halves == 3u ? Cfg::kIdesc : idesc_e4m3_f32(kPrefillBM, 128);
            for (int kb0 = 0; kb0 < kbt && ok; kb0 += dkb, ++dc) {
                const int acc = static_cast<int>(dc & 1u);
                if (!pf_wait(tempty_bar(acc), ((dc >> 1) & 1u) ^ 1u, err, kErrPrefillAccumEmptyWait, &s_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * BN) + hoff;
                const int kb1 = min(kb0 + dkb, kbt);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!pf_wait(full_bar(s), ph, err, kErrPrefillFullWait, &s_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t stage = base + static_cast<uint32_t>(s) * Cfg::kStageBytes;
                    const uint64_t da = sw128_kmajor_desc(stage),
                                   db = sw128_kmajor_desc(stage + kPrefillATile + hoff * kBlockK);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 32; ++kk) {  // +32 bytes along K = +2 in the address field
                        if constexpr (kPair)
                            mma_e4m3_pair(d, da + 2u * kk, db + 2u * kk, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                        else
                            mma_e4m3(d, da + 2u * kk, db + 2u * kk, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
                    if constexpr (kPair)
                        mma_commit_pair(empty_bar(s), 0x3);  // both CTAs' stages are free
                    else
                        mma_commit(empty_bar(s));
                    ++it;
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) {
                    if constexpr (kPair)
                        mma_commit_pair(tfull_bar(acc), 0x3);
                    else
                        mma_commit(tfull_bar(acc));
                }
            }
        }
        s_consumed = it;
        // arrives when every MMA issued above has completed (on both CTAs of a pair)
        if constexpr (kPair)
            mma_commit_pair(final_bar, 0x3);
        else
            mma_commit(final_bar);
    } else if (warp >= 2) {
        // ---------------------------------------------------------------- epilogue
        grid_dependency_wait();  // scales may come from the previous kernel; the output may be read by it
        const uint32_t quarter = warp & 3u;
        const int half = static_cast<int>(warp - 2) >> 2;
        const int row = static_cast<int>(quarter * 32u + lane);
        const bool issuer = ((warp - 2u) & 3u) == 0 && lane == 0;  // the half's TMA store thread
        const uint32_t stg = staging + static_cast<uint32_t>(half) * kPrefillOutBox;
        const bool sa_vec = !kBlk && (args.gran == 2 || args.gran == 3);
        const bool sb_vec = !kBlk && (args.gran == 1 || args.gran == 2);
        const float sa0 = kBlk ? 1.0f : __ldg(args.scale_a), sb0 = kBlk ? 1.0f : __ldg(args.scale_b);
        const int M = args.M, N = args.N;
        constexpr int kCols = BN / 2;  // columns of one thread
        uint32_t dc = 0;
        bool ok = true;
        for (int u = c; u < units && ok; u += G) {
            int m_tile, n_tile;
            uint32_t halves;
            unit_of(u, m_tile, n_tile, halves);
            float y[kCols];
#pragma unroll
            for (int j = 0; j < kCols; ++j) y[j] = 0.0f;
            // a warp whose 32 token rows all lie beyond M (small M), or whose
            // channel half is not in this unit, only takes part in the hand-shake
            const bool mine = BN == 128 || ((halves >> half) & 1u);
            const int m0 = m_tile * kTileM + static_cast<int>(rank) * kPrefillBM;  // this CTA's token rows
            const bool live = mine && m0 + static_cast<int>(quarter * 32u) < M;
            const int m_row = m0 + row;                                           // this thread's token row
            const int n_col = n_tile * BN + half * kCols;                 // its first channel
            // Blockwise: the scales of k-block kb (sa of this row, sb of this
            // column block) are requested two k-blocks ahead of their use, so
            // that their latency hides behind the epilogue's work.
            const float *const sa_row = args.scale_a + static_cast<int64_t>(m_row < M ? m_row : 0) * kbt;
            const float *const sb_row = args.scale_b + static_cast<int64_t>(n_col < N ? n_col / 128 : 0) * kbt;
            const bool sc_ok = kBlk && live && m_row < M && n_col < N;
            // (a, b) pairs for k-blocks kb0 + 1 and kb0 + 2; the product is taken at the use
            float pa1 = 0.0f, pb1 = 0.0f, pa2 = 0.0f, pb2 = 0.0f;
            if (kBlk && sc_ok) {
                pa1 = __ldg(sa_row);
                pb1 = __ldg(sb_row);
                if (kbt > 1) {
                    pa2 = __ldg(sa_row + 1);
                    pb2 = __ldg(sb_row + 1);
                }
            }
            for (int kb0 = 0; kb0 < kbt; kb0 += dkb, ++dc) {
                const int acc = static_cast<int>(dc & 1u);
                float bsc = 0.0f;  // blockwise: scale product of k-block kb0 (drain_kb == 1)
                if constexpr (kBlk) {
                    bsc = __fmul_rn(pa1, pb1);
                    pa1 = pa2;
                    pb1 = pb2;
                    if (sc_ok && kb0 + 2 < kbt) {
                        pa2 = __ldg(sa_row + kb0 + 2);
                        pb2 = __ldg(sb_row + kb0 + 2);
                    }
                }
                if (!pf_warp_wait(tfull_bar(acc), (dc >> 1) & 1u, err, kErrPrefillAccumWait, &s_abort, lane)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (live) {
                const uint32_t tbase = tmem + ((quarter * 32u) << 16) +
                                       static_cast<uint32_t>(acc * BN + half * kCols);
                // 16-column chunks, the next one loading while the current one
                // is added (paired FP32 instructions)
                uint32_t v[2][16];
                tmem_ld16(tbase, v[0]);
#pragma unroll
                for (int j = 0; j < kCols; j += 16) {
                    const int cur = (j / 16) & 1;
                    tmem_ld_wait();
                    if (j + 16 < kCols) tmem_ld16(tbase + static_cast<uint32_t>(j + 16), v[cur ^ 1]);
#pragma unroll
                    for (int q = 0; q < 16; q += 2) {
                        const float a0 = __uint_as_float(v[cur][q]), a1 = __uint_as_float(v[cur][q + 1]);
                        if constexpr (kBlk)
                            fma2_rn(y[j + q], y[j + q + 1], a0, a1, bsc);
                        else
                            add2_rn(y[j + q], y[j + q + 1], a0, a1);
                    }
                }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair)
                        mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));  // the leader's barrier
                    else
                        mbar_arrive(tempty_bar(acc));
                }
            }
            if (!ok) break;
            const int m = m0 + row;
            if (mine) {  // the whole half (4 warps) alike: every warp reaches the named barriers
                const float sa = (sa_vec && m < M) ? __ldg(args.scale_a + m) : sa0;
                const int nbase = n_tile * BN + half * kCols;
#pragma unroll
                for (int b = 0; b < kCols / 64; ++b) {
                    if (issuer) bulk_wait_read_all();  // the box's previous store has read the buffer
                    named_bar_sync(1u + static_cast<uint32_t>(half), 128u);
                    if (m < M) {  // rows beyond M are not stored (the TMA store clips them)
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const int j = b * 64 + c * 8, n = nbase + j;
                            uint32_t p[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {  // N % 8 == 0: 8 columns all in or all out
                                const float b0 = (sb_vec && n < N) ? __ldg(args.scale_b + n + 2 * q) : sb0;
                                const float b1 = (sb_vec && n < N) ? __ldg(args.scale_b + n + 2 * q + 1) : sb0;
                                p[q] = pack_bf16x2(__fmul_rn(__fmul_rn(y[j + 2 * q], sa), b0),
                                                   __fmul_rn(__fmul_rn(y[j + 2 * q + 1], sa), b1));
                            }
                            // 16-byte chunk c of row `row` at chunk c ^ (row % 8): the 128-byte swizzle
                            st_shared_v4(stg + static_cast<uint32_t>(row) * 128u +
                                             (static_cast<uint32_t>(c ^ (row & 7)) << 4),
                                         p[0], p[1], p[2], p[3]);
                        }
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(1u + static_cast<uint32_t>(half), 128u);
                    if (issuer) {
                        tma_store_2d(&tmap_out, stg, nbase + b * 64, m0);
                        bulk_commit_group();
                    }
                }
            }
            __syncwarp();
        }
        if (issuer) bulk_wait_all();  // every output box written before the CTA exits
    }

    // Every thread triggers only here, after the producer's dependency wait
    // (the producer triggered once more right after its last load).
    __syncwarp();
    if constexpr (kPair)
        cluster_sync();  // no CTA of the pair arrives remotely after this
    else
        __syncthreads();
    grid_launch_dependents();

    if (tid == 0 && leader) {
        // Loads issued but never consumed (only after a timeout): let them land
        // before the CTAs exit.  A pair's loads all signal the leader's
        // barriers; the peer's count is read from its shared memory.
        uint32_t issued = s_issued;
        if constexpr (kPair) {
            uint32_t peer;
            asm volatile("ld.shared::cluster.u32 %0, [%1];"
                         : "=r"(peer)
                         : "r"(map_to_rank(smem_u32(&s_issued), 1))
                         : "memory");
            issued = max(issued, peer);
        }
        const uint32_t consumed = s_consumed;
        for (uint32_t i = consumed; i < issued; ++i)
            mbar_wait(full_bar(static_cast<int>(i % static_cast<uint32_t>(stages))),
                      (i / static_cast<uint32_t>(stages)) & 1u, err, kErrPrefillFullWait);
    }
    if constexpr (kPair) {
        __syncwarp();
        cluster_sync();  // the peer stays until the leader's check of its loads
    }
    if (warp == 1) {
        mbar_wait(final_bar, 0, err, kErrPrefillAccumWait);  // every MMA has completed
        tc_fence_after();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem, Cfg::kTmemCols);
        else
            tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

}  // namespace

// Shared memory of one CTA: alignment slack, the stages, the mbarriers
// (full/empty per stage, full/empty per accumulator, one final), rounded up.
static size_t prefill_smem_bytes(int stages, int bn, bool pair) {
    const size_t barriers = 8u * static_cast<size_t>(2 * stages + 5);
    const size_t stage = static_cast<size_t>(kPrefillBM + (pair ? 128 : bn)) * kBlockK;
    return 1024 + static_cast<size_t>(stages) * stage + 2u * kPrefillOutBox + ((barriers + 127) / 128) * 128;
}

PrefillPlan plan_prefill(int64_t M, int64_t N, int64_t K, int num_sms, bool blockwise) {
    PrefillPlan p{};
    p.m_tiles = static_cast<int>((M + kPrefillBM - 1) / kPrefillBM);
    // 256-channel tiles, unless they would leave most SMs idle while the
    // kernel is bound by streaming the weights (small M): then 128 channels.
    const int64_t tiles256 = static_cast<int64_t>(p.m_tiles) * ((N + 255) / 256);
    p.bn = (M <= kPrefillSmallM && 2 * tiles256 <= num_sms) ? 128 : 256;
    p.n_tiles = static_cast<int>((N + p.bn - 1) / p.bn);
    p.kb_total = static_cast<int>((K + kBlockK - 1) / kBlockK);
    // CTA pairs (256-token tiles) once there are two token tiles of 128, but
    // not for blockwise scaling: its per-k-block drains would hand each
    // accumulator back across the pair (measured 239 against 142 us on
    // 2048 x 10240 x 5120)
    p.pair = (!blockwise && p.bn == 256 && M > kPrefillBM && num_sms >= 2) ? 1 : 0;
    if (p.pair) {
        p.m_tiles = static_cast<int>((M + 2 * kPrefillBM - 1) / (2 * kPrefillBM));
        const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
        const int64_t clusters = std::min<int64_t>(tiles, num_sms / 2);
        p.tiles = tiles;
        p.full_units = p.units = tiles;
        p.ctas = static_cast<int>(2 * clusters);
        p.stages = PrefillCfg<256, true>::kStages;
        p.drain_kb = (kPrefillDrainKb > 0 && kPrefillDrainKb < p.kb_total) ? kPrefillDrainKb : p.kb_total;
        p.smem_bytes = prefill_smem_bytes(p.stages, p.bn, true);
        return p;
    }
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    // A last round that would fill at most half of the SMs runs as half tiles
    // (256-channel tiles whose last one has two halves only).
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    const int64_t tail = tiles % sms;
    const int64_t last_rows = N - static_cast<int64_t>(p.n_tiles - 1) * p.bn;
    const bool split = p.bn == 256 && tiles > sms && tail > 0 && 2 * tail <= sms && last_rows > 128;
    p.tiles = tiles;
    p.full_units = split ? tiles - tail : tiles;
    p.units = split ? tiles + tail : tiles;
    p.ctas = static_cast<int>(p.units < sms ? p.units : sms);
    if (p.ctas < 1) p.ctas = 1;
    p.stages = p.bn == 256 ? PrefillCfg<256>::kStages : PrefillCfg<128>::kStages;
    const int dkb = M <= kPrefillSmallM ? kPrefillDrainKbSmall : kPrefillDrainKb;
    p.drain_kb = (dkb > 0 && dkb < p.kb_total) ? dkb : p.kb_total;
    p.smem_bytes = prefill_smem_bytes(p.stages, p.bn, false);
    return p;
}

template <int BN, bool kBlk, bool kPair>
static cudaError_t launch_bn(const CUtensorMap &tmap_a, const CUtensorMap &tmap_b, const CUtensorMap &tmap_out,
                             const PrefillArgs &a, const PrefillPlan &plan, const LaunchOpts &opts_in,
                             cudaStream_t stream) {
    LaunchOpts opts = opts_in;
    opts.cluster_x = kPair ? 2 : 1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool attr_done[64] = {};  // benign race: the attribute call is idempotent
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(prefill_gemm_kernel<BN, kBlk, kPair>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(prefill_smem_bytes(PrefillCfg<BN, kPair>::kStages, BN, kPair)));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    int ctas = plan.ctas;
    if constexpr (kPair) {
        // A persistent grid of pairs only works if every pair is resident at
        // once: at most as many clusters as the GPU can hold together (SMs
        // that have no partner in their GPC hold none).
        static int max_clusters[64] = {};  // benign race: the query is idempotent
        int mc = (dev >= 0 && dev < 64) ? max_clusters[dev] : 0;
        if (mc == 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(plan.ctas));
            cfg.blockDim = dim3(kPrefillThreads);
            cfg.dynamicSmemBytes = plan.smem_bytes;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&mc, prefill_gemm_kernel<BN, kBlk, kPair>, &cfg);
            if (e != cudaSuccess) return e;
            if (mc < 1) return cudaErrorInvalidConfiguration;
            if (dev >= 0 && dev < 64) max_clusters[dev] = mc;
        }
        ctas = std::min(ctas, 2 * mc);
    }
    return launch_with_opts(prefill_gemm_kernel<BN, kBlk, kPair>, dim3(static_cast<unsigned>(ctas)),
                            dim3(kPrefillThreads), plan.smem_bytes, stream, opts, tmap_a, tmap_b, tmap_out, a);
}

cudaError_t launch_prefill_gemm(const CUtensorMap &tmap_a, const CUtensorMap &tmap_b, const CUtensorMap &tmap_out,
                                const float *scale_a,
                                const float *scale_b, int granularity, int64_t M, int64_t N, int64_t K, void *out,
                                uint32_t *err, const PrefillPlan &plan, const LaunchOpts &opts,
                                cudaStream_t stream) {
    (void)K;
    PrefillArgs a;
    a.scale_a = scale_a;
    a.scale_b = scale_b;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = err;
    a.gran = granularity;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.kb_total = plan.kb_total;
    a.m_tiles = plan.m_tiles;
    a.full_units = static_cast<int>(plan.full_units);
    a.units = static_cast<int>(plan.units);
    a.stages = plan.stages;
    a.drain_kb = plan.drain_kb;
    if (granularity == kGranBlock128) {
        // every k-block has its own scales: drain after each one
        if (plan.pair) return cudaErrorInvalidValue;  // the plan must be made for blockwise scaling
        a.drain_kb = 1;
        if (plan.bn == 128) return launch_bn<128, true, false>(tmap_a, tmap_b, tmap_out, a, plan, opts, stream);
        if (plan.pair) return launch_bn<256, true, true>(tmap_a, tmap_b, tmap_out, a, plan, opts, stream);
        return launch_bn<256, true, false>(tmap_a, tmap_b, tmap_out, a, plan, opts, stream);
    }
    if (plan.bn == 128) return launch_bn<128, false, false>(tmap_a, tmap_b, tmap_out, a, plan, opts, stream);
    if (plan.pair) return launch_bn<256, false, true>(tmap_a, tmap_b, tmap_out, a, plan, opts, stream);
    return launch_bn<256, false, false>(tmap_a, tmap_b, tmap_out, a, plan, opts, stream);
}

}  // namespace fp8k
