// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fp8k {

// ---------------------------------------------------------------- quantisers --

cudaError_t launch_quant_static(const void *x, const float *scale, void *out, int64_t M, int64_t K,
                                uint32_t *err, cudaStream_t stream, int num_sms);

cudaError_t launch_quant_per_token(const void *x, void *out, float *scale_out, int64_t M, int64_t K,
                                   uint32_t *err, cudaStream_t stream);

cudaError_t launch_rmsnorm_quant(const void *x, const void *gamma, float eps, const float *scale, void *out,
                                 int64_t M, int64_t K, uint32_t *err, cudaStream_t stream);

// ------------------------------------------------------------- decode GEMM --

// Tile geometry of the weight-streaming kernel: 128 weight rows (output
// channels) per CTA on the tensor core's M side, the tokens on its N side.
constexpr int kDecodeRows = 128;
constexpr int kBlockK = 128;  // bytes (= E4M3 elements) of K per pipeline stage
constexpr int kDecodeMaxTokens = 128;

struct DecodePlan {
    int tok_pad;   // tokens per CTA on the MMA N side: 16, 32, 64 or 128
    int split;     // CTAs per cluster sharing one tile's K range (1..8)
    int stages;    // pipeline depth
    int n_tiles;   // ceil(N / 128)
    int m_tiles;   // ceil(M / tok_pad)
    int kb_total;  // ceil(K / 128)
    size_t smem_bytes;
};

DecodePlan plan_decode(int64_t M, int64_t N, int64_t K, int num_sms);

cudaError_t launch_decode_gemm(const CUtensorMap &tmap_w, const CUtensorMap &tmap_a, const float *scale_a,
                               const float *scale_b, int granularity, int64_t M, int64_t N, int64_t K, void *out,
                               uint32_t *err, const DecodePlan &plan, cudaStream_t stream);

}  // namespace fp8k
