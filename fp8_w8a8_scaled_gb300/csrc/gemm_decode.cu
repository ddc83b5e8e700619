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
// the kernel is bound by streaming B from HBM once.  Each CTA owns 128 weight
// rows (output channels) and a contiguous slice of K:
//   * warp 0 / lane 0 streams 128 x 128-byte weight boxes (and the matching
//     token box of A) with TMA into a ring of shared-memory stages (128-byte
//     swizzle), L2 evict-first for the once-read weights;
//   * warp 1 / lane 0 issues tcgen05.mma kind::f8f6f4 with the WEIGHTS as the
//     128-row A operand and the tokens (padded to 16/32/64/128) as the N side
//     ("swap-AB"), accumulating fp32 in TMEM, and frees each stage with
//     tcgen05.commit;
//   * the CTAs that split one tile's K range form a thread-block cluster; after
//     the mainloop each dumps its TMEM partial into its own shared memory, and
//     every CTA reduces a disjoint slice of the tile by reading the peers'
//     partials over distributed shared memory in fixed rank order
//     (deterministic, no atomics, no global workspace), applies the scales in
//     binary32 and writes bf16.
// The grid is one wave: the host picks the split so that all CTAs are
// resident at once and every CTA streams the same number of bytes.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace fp8k {
namespace {

constexpr uint32_t kWTileBytes = kDecodeRows * kBlockK;  // 16 KB of weights per stage

template <int TOK>
struct DecodeCfg {
    static constexpr uint32_t kATileBytes = TOK * kBlockK;
    static constexpr uint32_t kStageBytes = kWTileBytes + kATileBytes;
    static constexpr uint32_t kTmemCols = TOK < 32 ? 32 : TOK;  // power of two >= 32
    static constexpr uint32_t kIdesc = idesc_e4m3_f32(kDecodeRows, TOK);
};

template <int TOK>
__global__ void __launch_bounds__(128, 4)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                       const float *__restrict__ scale_a, const float *__restrict__ scale_b, int gran, int M, int N,
                       int kb_total, int stages, __nv_bfloat16 *__restrict__ out, uint32_t *err) {
    using Cfg = DecodeCfg<TOK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base, s_issued, s_consumed;

    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const base_gen = smem_raw + (base - raw);
    const uint32_t bar0 = base + static_cast<uint32_t>(stages) * Cfg::kStageBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (stages + s); };
    const uint32_t accum_bar = bar0 + 16u * stages;

    const uint32_t split = gridDim.x;
    const uint32_t rank = cluster_ctarank();
    const int n_tile = blockIdx.y, m_tile = blockIdx.z;
    const int kb_begin = static_cast<int>((static_cast<int64_t>(rank) * kb_total) / split);
    const int kb_end = static_cast<int>((static_cast<int64_t>(rank + 1) * kb_total) / split);
    const int iters = kb_end - kb_begin;

    if (tid == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_a);
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(accum_bar, 1);
        fence_mbar_init();
        s_issued = 0;
        s_consumed = 0;
    }
    if (warp == 1) tmem_alloc(smem_u32(&s_tmem_base), Cfg::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------------- producer
        const uint64_t evict_first = policy_evict_first();
        int i = 0;
        // Weights do not depend on earlier kernels in the stream; activations do.
        grid_dependency_wait();
        for (; i < iters; ++i) {
            const int s = i % stages;
            const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
            if (!mbar_wait(empty_bar(s), ph ^ 1u, err, kErrDecodeEmptyWait)) break;
            const uint32_t stage = base + static_cast<uint32_t>(s) * Cfg::kStageBytes;
            mbar_arrive_expect_tx(full_bar(s), Cfg::kStageBytes);
            const int kx = (kb_begin + i) * kBlockK;
            tma_load_2d_hint(stage, &tmap_w, full_bar(s), kx, n_tile * kDecodeRows, evict_first);
            tma_load_2d(stage + kWTileBytes, &tmap_a, full_bar(s), kx, m_tile * TOK);
        }
        s_issued = static_cast<uint32_t>(i);
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        int i = 0;
        for (; i < iters; ++i) {
            const int s = i % stages;
            const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
            if (!mbar_wait(full_bar(s), ph, err, kErrDecodeFullWait)) break;
            tc_fence_after();
            const uint32_t w_addr = base + static_cast<uint32_t>(s) * Cfg::kStageBytes;
            const uint32_t a_addr = w_addr + kWTileBytes;
#pragma unroll
            for (int kk = 0; kk < kBlockK / 32; ++kk) {
                mma_e4m3(tmem, sw128_kmajor_desc(w_addr + 32u * kk), sw128_kmajor_desc(a_addr + 32u * kk),
                         Cfg::kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(empty_bar(s));
        }
        s_consumed = static_cast<uint32_t>(i);
        mma_commit(accum_bar);  // arrives once every MMA issued above has completed
    }
    __syncwarp();
    grid_launch_dependents();
    grid_dependency_wait();  // the scales may come from the previous kernel in the stream
    __syncthreads();

    // ------------------------------------------------------------------ epilogue
    const uint32_t issued = s_issued, consumed = s_consumed;
    const bool acc_ok = mbar_wait(accum_bar, 0, err, kErrDecodeAccumWait);
    tc_fence_after();
    if (tid == 0) {
        // Loads issued but never consumed (only after a timeout): let them land
        // before the stage memory is reused.
        for (uint32_t i = consumed; i < issued; ++i)
            mbar_wait(full_bar(static_cast<int>(i % stages)), (i / stages) & 1u, err, kErrDecodeFullWait);
    }
    __syncthreads();

    float *part = reinterpret_cast<float *>(base_gen);  // [TOK][128] fp32, reuses the stage ring
    // CTA-uniform, since the TMEM loads below are warp-collective (.sync.aligned)
    const bool have = __syncthreads_and(acc_ok) && iters > 0 && consumed == static_cast<uint32_t>(iters);
    if (have) {
#pragma unroll 1
        for (int c0 = 0; c0 < TOK; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tmem + ((warp * 32u) << 16) + static_cast<uint32_t>(c0), r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) part[(c0 + j) * kDecodeRows + tid] = __uint_as_float(r[j]);
        }
    } else {
        for (int c = 0; c < TOK; ++c) part[c * kDecodeRows + tid] = 0.0f;
    }
    tc_fence_before();
    cluster_sync();  // every partial of the tile is now visible to the whole cluster

    const int rows_per = (kDecodeRows + static_cast<int>(split) - 1) / static_cast<int>(split);
    const int r0 = static_cast<int>(rank) * rows_per;
    const int r1 = min(kDecodeRows, r0 + rows_per);
    const int nrows = max(0, r1 - r0);
    const int m0 = m_tile * TOK;
    const int mt = min(TOK, M - m0);
    const uint32_t part_addr = smem_u32(part);
    const bool sa_vec = (gran == 2 || gran == 3);
    const bool sb_vec = (gran == 1 || gran == 2);
    const float sa0 = __ldg(scale_a), sb0 = __ldg(scale_b);
    for (int e = tid; e < nrows * mt; e += 128) {
        const int nl = r0 + e % nrows;
        const int m = e / nrows;
        const int n = n_tile * kDecodeRows + nl;
        if (n >= N) continue;
        const uint32_t off = part_addr + 4u * static_cast<uint32_t>(m * kDecodeRows + nl);
        float acc = 0.0f;
        for (uint32_t src = 0; src < split; ++src) acc = __fadd_rn(acc, ld_cluster_f32(map_to_rank(off, src)));
        const float sa = sa_vec ? __ldg(scale_a + m0 + m) : sa0;
        const float sb = sb_vec ? __ldg(scale_b + n) : sb0;
        out[static_cast<int64_t>(m0 + m) * N + n] = __float2bfloat16_rn(__fmul_rn(__fmul_rn(acc, sa), sb));
    }
    cluster_sync();  // peers are done reading this CTA's partial

    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

template <int TOK>
cudaError_t launch_tok(const CUtensorMap &tw, const CUtensorMap &ta, const float *sa, const float *sb, int gran,
                       int64_t M, int64_t N, void *out, uint32_t *err, const DecodePlan &p, cudaStream_t stream) {
    static bool attr_done = false;  // benign race: the attribute call is idempotent
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(decode_gemm_kernel<TOK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             200 * 1024);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.split), static_cast<unsigned>(p.n_tiles),
                       static_cast<unsigned>(p.m_tiles));
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = static_cast<unsigned>(p.split);
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_gemm_kernel<TOK>, tw, ta, sa, sb, gran, static_cast<int>(M),
                              static_cast<int>(N), p.kb_total, p.stages, static_cast<__nv_bfloat16 *>(out), err);
}

}  // namespace

// Shared memory one CTA needs for `stages` stages of `tok` tokens, plus the
// 1024-byte alignment slack and the barriers.
static size_t decode_smem_bytes(int tok, int stages) {
    return 1024 + static_cast<size_t>(stages) * (kDecodeRows * kBlockK + tok * kBlockK) + 256;
}

DecodePlan plan_decode(int64_t M, int64_t N, int64_t K, int num_sms) {
    DecodePlan p{};
    p.tok_pad = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
    const int stage_bytes = kDecodeRows * kBlockK + p.tok_pad * kBlockK;
    // About 60 KB of stages per CTA; several CTAs share an SM.
    p.stages = 60 * 1024 / stage_bytes;
    if (p.stages < 2) p.stages = 2;
    p.smem_bytes = decode_smem_bytes(p.tok_pad, p.stages);
    p.n_tiles = static_cast<int>((N + kDecodeRows - 1) / kDecodeRows);
    p.m_tiles = static_cast<int>((M + p.tok_pad - 1) / p.tok_pad);
    p.kb_total = static_cast<int>((K + kBlockK - 1) / kBlockK);
    // CTAs resident per SM: 228 KB of shared memory per SM (1 KB reserved per
    // CTA), at most 4 by the register budget of __launch_bounds__(128, 4), and
    // TMEM columns (512 per SM).
    const int tmem_cols = p.tok_pad < 32 ? 32 : p.tok_pad;
    int per_sm = static_cast<int>((228 * 1024) / (p.smem_bytes + 1024));
    if (per_sm > 512 / tmem_cols) per_sm = 512 / tmem_cols;
    if (per_sm > 4) per_sm = 4;
    if (per_sm < 1) per_sm = 1;
    const int64_t slots = static_cast<int64_t>(per_sm) * num_sms;
    const int64_t tiles = static_cast<int64_t>(p.n_tiles) * p.m_tiles;
    // Pick the split S (1..8, at most one k-block per CTA) that minimises
    // waves * (k-blocks per CTA + fixed per-CTA cost); ties keep the smaller S.
    const int kOverheadKb = 2;
    int best_s = 1;
    int64_t best_cost = -1;
    for (int s = 1; s <= 8 && s <= p.kb_total; ++s) {
        const int64_t ctas = tiles * s;
        const int64_t waves = (ctas + slots - 1) / slots;
        const int64_t per_cta = (p.kb_total + s - 1) / s;
        const int64_t cost = waves * (per_cta + kOverheadKb);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_s = s;
        }
    }
    p.split = best_s;
    return p;
}

cudaError_t launch_decode_gemm(const CUtensorMap &tmap_w, const CUtensorMap &tmap_a, const float *scale_a,
                               const float *scale_b, int granularity, int64_t M, int64_t N, int64_t K, void *out,
                               uint32_t *err, const DecodePlan &plan, cudaStream_t stream) {
    (void)K;
    switch (plan.tok_pad) {
        case 16: return launch_tok<16>(tmap_w, tmap_a, scale_a, scale_b, granularity, M, N, out, err, plan, stream);
        case 32: return launch_tok<32>(tmap_w, tmap_a, scale_a, scale_b, granularity, M, N, out, err, plan, stream);
        case 64: return launch_tok<64>(tmap_w, tmap_a, scale_a, scale_b, granularity, M, N, out, err, plan, stream);
        default: return launch_tok<128>(tmap_w, tmap_a, scale_a, scale_b, granularity, M, N, out, err, plan, stream);
    }
}

}  // namespace fp8k
