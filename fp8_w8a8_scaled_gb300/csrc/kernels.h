// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

namespace fp8k {

// Launch options shared by the kernels.
struct LaunchOpts {
    bool pdl = true;              // programmatic dependent launch (prologue overlaps the previous kernel)
    bool weights_static = false;  // B is not written by the kernel just before this one in the stream
    int cluster_x = 1;            // CTAs per thread-block cluster (along x); 1 = no clusters
};

// Launch with the programmatic-stream-serialisation attribute when opts.pdl:
// the kernel may start while its predecessor in the stream is finishing, and
// waits for it (griddepcontrol.wait) before touching memory it may have written.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_with_opts(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, const LaunchOpts &opts, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = opts.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (opts.cluster_x > 1) {  // thread-block clusters of cluster_x CTAs along x
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(opts.cluster_x);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// ---------------------------------------------------------------- quantisers --

cudaError_t launch_quant_static(const void *x, const float *scale, void *out, int64_t M, int64_t K,
                                uint32_t *err, cudaStream_t stream, int num_sms, const LaunchOpts &opts);

cudaError_t launch_quant_per_token(const void *x, void *out, float *scale_out, int64_t M, int64_t K,
                                   uint32_t *err, cudaStream_t stream, int num_sms, const LaunchOpts &opts);

// Blockwise quantisers: 128-wide token groups (scales [M, ceil(K/128)]) and
// 128 x 128 weight blocks (scales [ceil(N/128), ceil(K/128)]).
cudaError_t launch_quant_per_token_group(const void *x, void *out, float *scale_out, int64_t M, int64_t K,
                                         cudaStream_t stream, const LaunchOpts &opts);
cudaError_t launch_quant_weight_block(const void *w, void *out, float *scale_out, int64_t N, int64_t K,
                                      cudaStream_t stream, const LaunchOpts &opts);

// Weight shards (each [rows_j, K] E4M3 with a per-tensor scale) merged into one
// weight requantised to the largest scale.
constexpr int kMaxMergeShards = 16;
struct MergeArgs {
    const uint4 *src[kMaxMergeShards];
    const float *scale[kMaxMergeShards];
    int64_t end16[kMaxMergeShards];  // cumulative end of each shard, in 16-byte vectors
    int n;
    uint4 *out;
    float *scale_out;
    int64_t n16;
};
cudaError_t launch_requant_merge(const MergeArgs &a, cudaStream_t stream, int num_sms, const LaunchOpts &opts);

// gate_up [M, 2I] bf16 rows [gate | up] -> E4M3 [M, I] of silu(gate) * up, per-token scales.
cudaError_t launch_silu_mul_quant(const void *gate_up, void *out, float *scale_out, int64_t M, int64_t I,
                                  uint32_t *err, cudaStream_t stream, int num_sms, const LaunchOpts &opts);

// resid != nullptr: the row is bf16(x + resid) (which replaces resid) before the norm.
cudaError_t launch_rmsnorm_quant(const void *x, const void *gamma, float eps, const float *scale, void *out,
                                 int64_t M, int64_t K, uint32_t *err, cudaStream_t stream, int num_sms,
                                 const LaunchOpts &opts, void *resid = nullptr);

// ------------------------------------------------------------- decode GEMM --

// Tile geometry of the weight-streaming kernel: 128 weight rows (output
// channels) per tile on the tensor core's M side, up to 64 tokens on its N side.
// Granularity code of blockwise scaling (fp8_granularity FP8_GRAN_BLOCK_128):
// scales per 128-wide k-block, per token and per 128-row weight block.
constexpr int kGranBlock128 = 4;
constexpr int kDecodeRows = 128;
constexpr int kBlockK = 128;  // bytes (= E4M3 elements) of K per pipeline stage
constexpr int kDecodeMaxTokens = 32;
// The decode kernel's exact 32-bit accumulators hold the sums of fewer than
// 2048 k-blocks (K <= 262,016); longer K goes to the tile kernel (blockwise
// scaling, summed in binary32 TwoSum pairs, has no such limit).
constexpr int64_t kExactMaxKb = 2048;

struct DecodePlan {
    int tok_pad;      // tokens per tile on the MMA N side: 16 (M <= 16) or 32
    int stages;       // pipeline depth
    int n_tiles;      // ceil(N / 128)
    int m_tiles;      // ceil(M / tok_pad)
    int kb_total;     // ceil(K / 128)
    int64_t units;    // n_tiles * m_tiles * kb_total (one unit = one tile x one k-block)
    int ctas;         // stream-K: persistent CTAs, CTA c owning units [c*units/ctas, (c+1)*units/ctas);
                      // cluster mode: n_tiles * split
    int split;        // cluster mode: CTAs (one cluster) per output tile; 0 = stream-K
    int exact;        // 1: the k-block partials are summed exactly as integers (every granularity but
                      // blockwise), so the result does not depend on how K is divided among CTAs
    size_t smem_bytes;
};

// The decode kernel's plan, a pure function of the shape, the scaling kind and
// the SM count (the grid and its division of K are the same for both kinds;
// blockwise scaling sums TwoSum parts, every other granularity exact ones).
DecodePlan plan_decode(int64_t M, int64_t N, int64_t K, int num_sms, bool blockwise = false);

// Scratch of the decode kernel: a zeroed arrival counter per output tile, and
// two partial-sum slots per CTA (128 x tok_pad entries each: 64-bit integer
// exact parts -- two floats' room -- or binary32 TwoSum parts for blockwise
// scaling) for the tiles whose K range is split between CTAs under stream-K.
// Every launch leaves the counters at zero.
struct DecodeWorkspace {
    uint32_t *counters;
    float *slots;
};
size_t decode_counters_needed(const DecodePlan &p);  // number of counters
size_t decode_slot_floats(const DecodePlan &p);      // number of fp32 slot entries

cudaError_t launch_decode_gemm(const CUtensorMap &tmap_w, const CUtensorMap &tmap_a, const float *scale_a,
                               const float *scale_b, int granularity, int64_t M, int64_t N, int64_t K, void *out,
                               uint32_t *err, const DecodePlan &plan, const DecodeWorkspace &ws, const LaunchOpts &opts,
                               cudaStream_t stream);

// ------------------------------------------------------- weight-only GEMM --

// The W8A16 decode kernel (bf16 activations, E4M3 weights, M <= 32): the
// decode plan's fields with one persistent CTA per SM (stream-K, split = 0);
// tmap_x is a bf16 tensor map with 64-element x tok_pad boxes.
DecodePlan plan_w8a16(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_w8a16_gemm(const CUtensorMap &tmap_w, const CUtensorMap &tmap_x, const float *scale_b,
                              int per_channel, int64_t M, int64_t N, int64_t K, void *out, uint32_t *err,
                              const DecodePlan &plan, const DecodeWorkspace &ws, const LaunchOpts &opts,
                              cudaStream_t stream);
// The weight-only GEMV for one to kW16GemvMaxTokens tokens on the CUDA cores
// (no tensor core, no split of K, nothing shared between CTAs): one CTA per
// SM, whole weight rows per warp streamed through a per-warp ring of bulk
// copies, the tokens staged in shared memory as bf16 (M * K * 2 bytes, at
// most kW16GemvMaxXBytes beside the 180 KB ring).
constexpr int kW16GemvMaxTokens = 4;
constexpr int64_t kW16GemvMaxXBytes = 40 * 1024;
inline bool w8a16_gemv_fits(int64_t M, int64_t K) {
    return M >= 1 && M <= kW16GemvMaxTokens && M * K * 2 <= kW16GemvMaxXBytes;
}
cudaError_t launch_w8a16_gemv(const void *W, const void *x, const float *scale_b, int per_channel, int64_t M,
                              int64_t N, int64_t K, void *out, uint32_t *err, int num_sms, const LaunchOpts &opts,
                              cudaStream_t stream);
// The weight-only large-M tile kernel (M >= 33): output tiles of 2 x 128
// weight rows x kW16TileTokens tokens (or one 128-row half in a split last
// round), the E4M3 weight widened to bf16 on chip.
constexpr int kW16TileTokens = 128;
struct W16TileArgs {
    const float *scale_b;
    __nv_bfloat16 *out;
    uint32_t *err;
    int per_channel, M, N, kb_total, m_tiles, full_units, units, wstages, xstages, weights_static;
};
struct W16TilePlan {
    int m_tiles, n_tiles, kb_total;
    int64_t tiles, full_units, units;  // units: whole tiles below full_units, then half tiles
    int ctas, wstages, xstages;
    size_t smem_bytes;
};
W16TilePlan plan_w8a16_tile(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_w8a16_tile(const CUtensorMap &tmap_w, const CUtensorMap &tmap_x, const float *scale_b,
                              int per_channel, int64_t M, int64_t N, void *out, uint32_t *err,
                              const W16TilePlan &plan, const LaunchOpts &opts, cudaStream_t stream);
// w16 [N,K] bf16 = bf16_rne(fp32(dec(W) * s)) (K % 16 == 0); scale == nullptr
// gives the exact E4M3 values (the large-M branch's weight).
cudaError_t launch_widen_weight(const void *w, const float *scale, int per_channel, int64_t N, int64_t K, void *out,
                                cudaStream_t stream, int num_sms, const LaunchOpts &opts);

// ------------------------------------------------------------ prefill GEMM --

// Tile geometry of the large-M kernel: 128 tokens (MMA M) x 256 output
// channels (MMA N) per tile, 128-byte k-blocks.
constexpr int kPrefillBM = 128;
constexpr int kPrefillBN = 256;
constexpr int64_t kPrefillMinM = 33;  // fp8_scaled_mm sends M >= this to the prefill kernel

struct PrefillPlan {
    int bn;    // output channels per tile: 256, or 128 for small M with few tiles
    int pair;  // 1: CTA pairs (cta_group::2) on 256-token x 256-channel tiles
    int m_tiles, n_tiles, kb_total;
    int64_t tiles, full_units, units;  // units: whole tiles below full_units, then 128-channel halves
    int ctas;       // persistent CTAs (one per SM at most)
    int stages;
    int drain_kb;   // k-blocks accumulated in TMEM before the epilogue folds them into registers
    size_t smem_bytes;
};

PrefillPlan plan_prefill(int64_t M, int64_t N, int64_t K, int num_sms, bool blockwise);

cudaError_t launch_prefill_gemm(const CUtensorMap &tmap_a, const CUtensorMap &tmap_b, const CUtensorMap &tmap_out,
                                const float *scale_a,
                                const float *scale_b, int granularity, int64_t M, int64_t N, int64_t K, void *out,
                                uint32_t *err, const PrefillPlan &plan, const LaunchOpts &opts, cudaStream_t stream);

}  // namespace fp8k
