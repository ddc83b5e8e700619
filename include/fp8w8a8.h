/*
 * fp8w8a8.h -- C ABI of the GB300 (sm_103a) FP8 (E4M3) W8A8 scaled-GEMM library.
 *
 * The library computes the linear layer of an FP8 "W8A8" model:
 *
 *     y_bf16[m,n] = bf16( (sum_k A[m,k] * B[n,k]) * scale_a[.] * scale_b[.] )
 *
 * with A the E4M3 activations [M,K], B the E4M3 weights [N,K] (K contiguous,
 * one row per output channel), per-tensor / per-output-channel / per-token
 * scales and a bf16 output, plus the producers that quantise activations to
 * E4M3: a fused RMSNorm -> static quant, a dynamic per-token quant and a plain
 * static quant.
 *
 * Where each call comes from (page title, then section):
 *   [P1] "The FP8 tower's cuBLASLt default rests on a false premise: vLLM selects
 *        FlashInferFP8ScaledMMLinearKernel, not nvjet/cuBLASLt" (vllm.cpp #252)
 *   [P2] "Qwen3.6 NVFP4 baselines (27B and 35B-A3B) must reach vLLM speed parity"
 *        (vllm.cpp #213)
 *   [P3] "We emit F32 where vLLM emits bf16 on the biggest prefill buffers (GDN
 *        in_proj, attn gate, q/k/v) -- 2x traffic ..." (vllm.cpp #417)
 *   [P4] "[Kernel] add Flashinfer cutedsl w4a16 linear" (vllm #53014), the
 *        commit message that references it (Marlin large-M dispatch).
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *     caller owns and allocates every buffer.  The library allocates no device
 *     memory per call: its only allocation is a ~9 MB scratch area per device
 *     (arrival counters and partial sums of the decode GEMM), made on the
 *     first fp8_scaled_mm call on that device -- make that first call before
 *     capturing a CUDA graph.  Because the scratch is shared, GEMM calls that
 *     may run concurrently on different streams of one device race; order
 *     them on one stream (or with events).
 *   - Row-major layouts.  E4M3 is the OCP FP8 "E4M3" finite encoding
 *     (torch.float8_e4m3fn): 1 byte, max 448, NaN = 0x7F/0xFF, no Inf.
 *     bf16 is IEEE binary32's upper half.  Scales are IEEE binary32.
 *   - Every call validates its arguments first and returns a status.  On any
 *     error nothing is launched and no memory is written.  M == 0 is a no-op
 *     that returns FP8_OK.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream), never synchronise the host, and read scales only from
 *     device memory, so a sequence of calls can be captured in a CUDA graph.
 *   - No exception crosses this boundary; the functions are thread-safe.
 *   - Results are deterministic: the same inputs give the same bytes, run
 *     after run (no floating-point atomics).
 */
#ifndef FP8W8A8_H_
#define FP8W8A8_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8_OK = 0,
    FP8_ERR_INVALID_ARG = 1,  /* null pointer, negative or too-large size, bad enum */
    FP8_ERR_ALIGNMENT = 2,    /* pointer not 16-byte aligned, or K / N not a multiple of 16 / 8 */
    FP8_ERR_UNSUPPORTED = 3,  /* a valid request this library does not implement (e.g. out_dtype) */
    FP8_ERR_CUDA = 4,         /* a CUDA runtime / driver call or a kernel launch failed */
    FP8_ERR_DEVICE = 5,       /* a kernel reported an error through the device error word */
    FP8_ERR_TOO_LARGE = 6     /* the problem needs more scratch than fp8_scaled_mm_noalloc's fixed area */
} fp8_status;

/* Which scale element multiplies output y[m,n] ([P1] "What is owed", item 2,
 * names per-tensor, per-channel and per-token scaling). */
typedef enum {
    FP8_GRAN_PER_TENSOR = 0,         /* scale_a[1], scale_b[1] */
    FP8_GRAN_PER_CHANNEL = 1,        /* scale_a[1], scale_b[N]: one scale per output channel */
    FP8_GRAN_PER_TOKEN_CHANNEL = 2,  /* scale_a[M], scale_b[N] */
    FP8_GRAN_PER_TOKEN = 3,          /* scale_a[M], scale_b[1] */
    /* Blockwise: scale_a[M][ceil(K/128)] (one per token per 128-wide group of
     * K), scale_b[ceil(N/128)][ceil(K/128)] (one per 128 x 128 weight block),
     * both row-major; y[m,n] = sum_g sa[m,g] * sb[n/128,g] * acc_g[m,n] with
     * acc_g the group's sum of products ([P4] commit message: "dense FP8
     * non-blockwise" implies a blockwise FP8 variant). */
    FP8_GRAN_BLOCK_128 = 4
} fp8_granularity;

/* Output dtype.  Only bf16: the pages' finding is that an F32 GEMM output
 * doubles the traffic on the largest activation buffers ([P3] "FINDING 1 --
 * F32-vs-bf16 output dtype on the fp8 path").  Anything else returns
 * FP8_ERR_UNSUPPORTED. */
typedef enum { FP8_OUT_BF16 = 0 } fp8_out_dtype;

/* Kernel identifiers returned by fp8_describe_dispatch. */
typedef enum {
    FP8_KERNEL_NONE = 0,          /* M == 0: nothing is launched */
    FP8_KERNEL_DECODE_SPLITK = 1, /* weight-streaming split-K kernel (small M) */
    FP8_KERNEL_PREFILL = 2,       /* persistent tensor-core tile kernel (large M) */
    FP8_KERNEL_W16_DECODE = 3,    /* weight-only: widen-on-chip split-K kernel (M <= 32, where the GEMV does not apply) */
    FP8_KERNEL_W16_DENSE = 4,     /* weight-only: tile kernel, weight widened on chip, dense bf16 MMAs (M >= 33) */
    FP8_KERNEL_W16_GEMV = 5       /* weight-only: CUDA-core GEMV, whole weight rows per warp (M <= 4) */
} fp8_kernel_id;

/* fp8_scaled_mm -- the FP8 W8A8 scaled GEMM.
 *
 * Source: [P1] "CORRECTION -- my headline claim was too strong": the FP8 linear
 * runs bmm_fp8(a, b, scale_a, scale_b, out_dtype, ...); [P3] "FINDING 1": the
 * output is the model dtype (bf16), not F32; [P1] "The real finding: shape
 * and fusion, not library" and [P2] "Lever 2": a merged QKV or gate|up
 * projection is one call over the row-concatenated weight (and its
 * concatenated per-channel scales); [P2] "Root-cause theme", item 1: the
 * weight is kept [N,K], not transposed to [K,N].
 *
 *   A        E4M3 [M,K] row-major, 16-byte aligned
 *   B        E4M3 [N,K] row-major (K contiguous), 16-byte aligned
 *   scale_a  f32, 1 or M elements by `granularity`
 *   scale_b  f32, 1 or N elements by `granularity`
 *   out      bf16 [M,N] row-major, 16-byte aligned, written in full
 *   M, N, K  0 <= M, 1 <= N, 1 <= K, each below 2^31; K % 16 == 0, N % 8 == 0
 *
 * y[m,n] = bf16_rne( fp32(fp32(acc[m,n] * sa) * sb) ) with acc the fp32
 * tensor-core accumulation of the exact E4M3 products.  Which kernel runs is a
 * pure function of (M, N, K, granularity), see fp8_describe_dispatch, so a
 * captured CUDA graph replays the same kernel the eager call would run:
 * M <= 32 the weight-streaming decode kernel (16-token tile for M <= 16,
 * 32-token tile above), M >= 33 the tensor-core tile kernel.  The decode
 * kernel's stream-K mode (few 128-row tiles with a long K, see
 * fp8_decode_split_for_sms) uses scratch memory: one area per stream, about
 * 20 MB, allocated on that stream's first stream-K call (cudaMalloc, counters
 * zeroed with cudaMemsetAsync on the stream; during graph capture the
 * allocation is made with the thread's capture mode relaxed and the zeroing
 * becomes part of the graph), for at most 64 streams per device
 * (FP8_ERR_UNSUPPORTED beyond); calls on different streams may overlap.  A
 * captured graph uses its capture stream's area: graphs captured on one
 * stream must not be replayed at the same time as each other.  Its
 * cluster mode and the tile kernel use none.  The result is deterministic
 * (bitwise the same on every run); row m does not depend on the other rows of
 * A (on the decode kernel for any M <= 32, on the tile kernel for any M >= 33),
 * and, with exact sums (every granularity but blockwise), a projection split
 * along N gives the same bits as the merged one.
 * Errors: FP8_ERR_INVALID_ARG, FP8_ERR_ALIGNMENT, FP8_ERR_UNSUPPORTED,
 * FP8_ERR_CUDA. */
fp8_status fp8_scaled_mm(const void *A, const void *B, const float *scale_a, const float *scale_b,
                         int granularity, int out_dtype, int64_t M, int64_t N, int64_t K, void *out,
                         void *stream);

/* Flags of fp8_scaled_mm_ex. */
typedef enum {
    /* B is not written by the kernel that runs just before this call in the
     * stream (typical for model weights), so the kernel may start streaming B
     * before that kernel has finished.  Wrong if the previous kernel writes B. */
    FP8_FLAG_WEIGHTS_STATIC = 1,
    /* Launch without programmatic dependent launch (plain stream order). */
    FP8_FLAG_NO_PDL = 2
} fp8_flags;

/* fp8_scaled_mm_ex -- fp8_scaled_mm with launch flags (fp8_flags, OR-ed).
 * By default every kernel of this library is launched with programmatic
 * dependent launch: it may begin its prologue while the previous kernel in the
 * stream is finishing and waits (griddepcontrol.wait) for that kernel before
 * reading anything it could have written.  Same arguments and errors as
 * fp8_scaled_mm; unknown flag bits return FP8_ERR_INVALID_ARG. */
fp8_status fp8_scaled_mm_ex(const void *A, const void *B, const float *scale_a, const float *scale_b,
                            int granularity, int out_dtype, int64_t M, int64_t N, int64_t K, void *out,
                            void *stream, unsigned flags);

/* fp8_scaled_mm_noalloc -- fp8_scaled_mm for callers that cannot allocate.
 *
 * The pages have no counterpart of this call; it exists for callers that may
 * not call cudaMalloc at all: code running inside a memory pool or arena
 * that must own every device allocation, hosts whose allocator is locked
 * while a CUDA graph is being built, or embedders that forbid hidden
 * allocations.  fp8_scaled_mm allocates a per-stream scratch area on a
 * stream's first stream-K call; this entry point instead uses a fixed scratch
 * area compiled into the library (a file-scope device array of 12 MB + 64 KB
 * that every GPU which loads the library holds until the process exits), and
 * never calls cudaMalloc, cudaFree or any allocating routine.
 *
 * Arguments, layouts and results are those of fp8_scaled_mm (same kernel,
 * same plan, so the same bytes).  Limits: M <= 16 (else FP8_ERR_TOO_LARGE).
 * Only the decode kernel's stream-K mode uses the fixed area: it needs one
 * arrival counter per 128-row output tile (at most 16384 tiles) and two slots
 * of 16 x 128 partial sums per CTA (at most 384 CTAs: its grid has at most
 * two CTAs per SM, so any GPU with up to 192 SMs); beyond that it returns
 * FP8_ERR_TOO_LARGE without launching anything.  Cluster-mode shapes (most
 * shapes, see fp8_decode_split_for_sms) use none of it and have no further
 * limit.
 *
 * The first call on a device looks up the device address of the scratch area
 * for that device (cudaGetSymbolAddress), so make the first call on each
 * device before capturing a CUDA graph.  Every stream-K call zeroes the area's
 * arrival counters on `stream` before its kernel.  All calls share the one
 * area and it keeps the last call's contents: calls that may run at the same
 * time on the GPU (different streams, no ordering) race and give wrong
 * results; order them.  Errors: those of fp8_scaled_mm, plus
 * FP8_ERR_TOO_LARGE. */
fp8_status fp8_scaled_mm_noalloc(const void *A, const void *B, const float *scale_a, const float *scale_b,
                                 int granularity, int out_dtype, int64_t M, int64_t N, int64_t K, void *out,
                                 void *stream);

/* rmsnorm_quant_fp8 -- fused RMSNorm -> static per-tensor E4M3 quantisation,
 * one pass ("quantise once" per layer).
 *
 * Source: [P3] "Ranked follow-ons from the same audit", third bullet: a fused
 * RMSNorm -> fp8 quant that is byte-exact with the unfused path; [P2] "The GDN
 * fp8 merge predicate FIRES": the fused producer requires the consumers to share
 * one bitwise-equal activation input_scale, which is why it takes one scale.
 *
 *   x        bf16 [M,K] row-major, 16-byte aligned
 *   gamma    bf16 [K], 16-byte aligned
 *   eps      added to mean(x^2) inside the square root
 *   scale    f32 [1] (device): the static activation scale s (x ~= dec(q) * s)
 *   out      E4M3 [M,K], 16-byte aligned
 *   K % 16 == 0, 1 <= K <= 65536
 *
 * Per row: ss = the exact sum of the squares of the row's bf16 values, rounded
 * once to binary32 (round to nearest even); then mean = ss / K, t = mean + eps,
 * d = sqrt(t), r = 1 / d, each one IEEE binary32 operation rounded to nearest
 * even; h = bf16_rne((x * r) * gamma) with two binary32 multiplies (no fused
 * multiply-add); q = e4m3_rne_sat(h / s) with an IEEE binary32 division.  The
 * bytes equal "RMSNorm to bf16, then quant_fp8_static" exactly.  With eps = 0
 * a row whose mean square underflows to zero in binary32 has r = inf: its
 * nonzero elements saturate to +-448 and its zero elements give NaN codes. */
fp8_status rmsnorm_quant_fp8(const void *x, const void *gamma, float eps, const float *scale, void *out,
                             int64_t M, int64_t K, void *stream);

/* fp8_add_rmsnorm_quant -- residual add, then rmsnorm_quant_fp8, one pass.
 *
 * Source: [P3] "Ranked follow-ons from the same audit", second bullet: each
 * FP8 projection's input should leave its producer already quantised; a
 * decoder layer's norm input is the residual stream plus the previous block's
 * output, so the add is folded into the norm-quant producer.
 *
 *   x         bf16 [M,K] (the block output), 16-byte aligned
 *   residual  bf16 [M,K], 16-byte aligned: read, then overwritten IN PLACE
 *             with h = bf16_rne( fp32(x) + fp32(residual) ) (one binary32
 *             addition, round to nearest even), the updated residual stream
 *   gamma, eps, scale, out, M, K   as rmsnorm_quant_fp8, applied to h
 *
 * out holds exactly the bytes rmsnorm_quant_fp8(h, ...) would write.  x and
 * residual must not overlap.  Errors: as rmsnorm_quant_fp8. */
fp8_status fp8_add_rmsnorm_quant(const void *x, void *residual, const void *gamma, float eps, const float *scale,
                                 void *out, int64_t M, int64_t K, void *stream);

/* fp8_silu_mul_quant_per_token -- SiLU(gate) * up, then dynamic per-token
 * E4M3 quantisation: the producer of the down projection's input.
 *
 * Source: [P3] "Ranked follow-ons from the same audit", second bullet: every
 * FP8 projection's input should leave its producer already quantised (here
 * the MLP's activation, which feeds the down projection).
 *
 *   gate_up    bf16 [M, 2I] row-major, 16-byte aligned: each row is
 *              [gate (I) | up (I)] (the merged gate_up GEMM's output)
 *   out        E4M3 [M, I], 16-byte aligned
 *   scale_out  f32 [M] (device): s_m = amax_m / 448 (1.0 for an all-zero row)
 *   I % 16 == 0, 1 <= I <= 131072
 *
 * a = bf16_rne( silu(g) * u ) with silu(g) = g / (1 + e(-g)) in binary32 and
 * e a fixed binary32 exp (Cody-Waite argument reduction, degree-7 Taylor
 * polynomial, one IEEE operation per step, within a few ulp of exp); then
 * out = e4m3(a / s_m) exactly as quant_fp8_per_token on a.
 * Errors: FP8_ERR_INVALID_ARG, FP8_ERR_ALIGNMENT, FP8_ERR_CUDA. */
fp8_status fp8_silu_mul_quant_per_token(const void *gate_up, void *out, float *scale_out, int64_t M, int64_t I,
                                        void *stream);

/* fp8_requant_merge -- merge weight shards that carry different per-tensor
 * scales into one weight with one scale, the largest (max_w_scale).
 *
 * Source: [P3] "Ranked follow-ons from the same audit", first bullet: a merged
 * QKV projection is one physical GEMM, and shards whose per-tensor scales
 * differ are requantised to the largest scale (lossy), instead of declining
 * to merge.  (With per-output-channel scales, concatenating the shards and
 * their scales merges them losslessly and needs no requantisation.)
 *
 *   shards     HOST array of n_shards DEVICE pointers, shard j E4M3
 *              [rows[j], K] row-major, 16-byte aligned (may be NULL if
 *              rows[j] == 0)
 *   scales     HOST array of n_shards DEVICE pointers to f32 [1]: s_j
 *   rows       HOST array of n_shards row counts
 *   out        E4M3 [sum rows, K], 16-byte aligned: the shards in order,
 *              code q of shard j becoming e4m3( fp32(dec(q) * s_j) / s_max )
 *   scale_out  f32 [1] (device): s_max = max_j s_j (must not alias an input)
 *   1 <= n_shards <= 16, K % 16 == 0, sum rows < 2^31
 *
 * Errors: FP8_ERR_INVALID_ARG, FP8_ERR_ALIGNMENT, FP8_ERR_CUDA. */
fp8_status fp8_requant_merge(const void *const *shards, const float *const *scales, const int64_t *rows,
                             int n_shards, int64_t K, void *out, float *scale_out, void *stream);

/* fp8_rmsnorm_quant_scaled_mm -- rmsnorm_quant_fp8 followed by fp8_scaled_mm
 * on its output, as one call ("quantise once": the normalised, quantised
 * activations are written to a_out for the layer's other projections, and
 * this projection consumes them at once).
 *
 * Source: [P3] "Ranked follow-ons from the same audit" (the fused RMSNorm ->
 * fp8 quant feeding the FP8 GEMMs of a layer, quantise once); [P1] "SETTLED
 * BY PAIRED TRACE" (at decode M the cost is per launch and per weight byte).
 *
 *   x, gamma, eps   as rmsnorm_quant_fp8 (x bf16 [M,K], gamma bf16 [K])
 *   scale_a         f32 [1] (device): the static activation scale, used both
 *                   to quantise and as the GEMM's activation scale
 *   B, scale_b      as fp8_scaled_mm; granularity FP8_GRAN_PER_TENSOR or
 *                   FP8_GRAN_PER_CHANNEL (the activation scale is one value)
 *   a_out           E4M3 [M,K], 16-byte aligned: written with exactly the bytes
 *                   rmsnorm_quant_fp8 writes
 *   out             bf16 [M,N]: exactly the bytes fp8_scaled_mm(a_out, ...)
 *                   writes
 *   flags           as fp8_scaled_mm_ex
 *   K % 16 == 0, 1 <= K <= 65536, N % 8 == 0
 *
 * It runs the norm kernel and then the GEMM kernel, chained with programmatic
 * dependent launch (the GEMM's CTAs launch early, fetch their first weights
 * and wait for the normalised rows).  Errors: those of the two calls; an
 * argument error is reported before anything is launched. */
fp8_status fp8_rmsnorm_quant_scaled_mm(const void *x, const void *gamma, float eps, const float *scale_a,
                                       const void *B, const float *scale_b, int granularity, int out_dtype, int64_t M,
                                       int64_t N, int64_t K, void *a_out, void *out, void *stream, unsigned flags);

/* quant_fp8_per_token -- dynamic per-token E4M3 quantisation.
 *
 * Source: [P1] "What is owed", item 2 (per-token scaling granularity and where
 * the activation quantisation happens).
 *
 *   x          bf16 [M,K] row-major, 16-byte aligned
 *   out        E4M3 [M,K], 16-byte aligned
 *   scale_out  f32 [M]: s_m = amax_m / 448 in binary32 (1.0 for an all-zero
 *              row); q = e4m3_rne_sat(x / s_m).  NaN entries do not take part
 *              in the max.
 *   K % 16 == 0, K <= 2^30.  Applied to a weight [N,K] this is per-output-
 *   channel weight quantisation; applied to a tensor viewed as one row it is
 *   per-tensor quantisation with s = amax/448. */
fp8_status quant_fp8_per_token(const void *x, void *out, float *scale_out, int64_t M, int64_t K,
                               void *stream);

/* fp8_quant_per_token_group -- dynamic E4M3 quantisation per token and per
 * 128-wide group of K, the activation side of FP8_GRAN_BLOCK_128.
 *
 * Source: [P4] commit message ("dense FP8 non-blockwise" sets a blockwise
 * variant apart); the group width 128 is this library's reading.
 *
 *   x          bf16 [M,K] row-major, 16-byte aligned
 *   out        E4M3 [M,K], 16-byte aligned
 *   scale_out  f32 [M][ceil(K/128)] row-major: each group quantised exactly as
 *              quant_fp8_per_token would quantise that group alone (the last
 *              group of a row may be narrower than 128).
 *   K % 16 == 0, K <= 2^30.
 * Errors: FP8_ERR_INVALID_ARG, FP8_ERR_ALIGNMENT, FP8_ERR_CUDA. */
fp8_status fp8_quant_per_token_group(const void *x, void *out, float *scale_out, int64_t M, int64_t K,
                                     void *stream);

/* fp8_quant_weight_block -- E4M3 quantisation of a weight [N,K] with one scale
 * per 128 x 128 block, the weight side of FP8_GRAN_BLOCK_128.
 *
 * Source: as fp8_quant_per_token_group.
 *
 *   w          bf16 [N,K] row-major, 16-byte aligned
 *   out        E4M3 [N,K], 16-byte aligned
 *   scale_out  f32 [ceil(N/128)][ceil(K/128)] row-major: s = amax over the
 *              block / 448 in binary32 (1.0 for an all-zero block; NaN
 *              entries do not take part); q = e4m3_rne_sat(w / s).  Edge
 *              blocks cover what is left of N and K.
 *   K % 16 == 0, K <= 2^30, N < 2^31.
 * Errors: FP8_ERR_INVALID_ARG, FP8_ERR_ALIGNMENT, FP8_ERR_CUDA. */
fp8_status fp8_quant_weight_block(const void *w, void *out, float *scale_out, int64_t N, int64_t K, void *stream);

/* fp8_w8a16_mm -- weight-only FP8 GEMM: bf16 activations, E4M3 weights.
 *
 * Source: [P4] "[Kernel] add Flashinfer cutedsl w4a16 linear" (vllm #53014):
 * the FP8 channelwise half of the weight-only path, and its large-M branch
 * (a dense 16-bit GEMM over the weight widened to 16 bits; here the widening
 * is done on chip, tile by tile).
 *
 *   x        bf16 [M,K] row-major, 16-byte aligned
 *   W        E4M3 [N,K] row-major (K contiguous), 16-byte aligned
 *   scale_b  f32, 1 (FP8_GRAN_PER_TENSOR) or N (FP8_GRAN_PER_CHANNEL) elements
 *   out      bf16 [M,N], 16-byte aligned, written in full
 *   M, N, K  as fp8_scaled_mm (K % 16 == 0, N % 8 == 0)
 *
 * y[m,n] = bf16( (sum_k x[m,k] * dec(W[n,k])) * sb ).  M <= 4 (and M * K <=
 * 20480): a GEMV on the CUDA cores, each warp whole weight rows, the weight
 * widened exactly to bf16 and multiplied with the bf16 tokens into binary32
 * (one fused multiply-add per product, k order within a lane, the lanes added
 * in a fixed order), so a token's row is the same alone or among up to four;
 * nothing is shared between CTAs and no scratch is used.  Otherwise
 * M <= 32: a split-K
 * kernel that widens each E4M3 weight tile to bf16 in tensor memory (exact)
 * and multiplies on the tensor core (fp32 accumulation inside 128-wide
 * k-blocks, TwoSum across them, the scale in binary32 at the end); its
 * stream-K mode uses the per-stream scratch of fp8_scaled_mm.  M >= 33: a tile
 * kernel (256 weight rows x 128 tokens per tile, the whole K) that widens each
 * E4M3 weight box to bf16 in tensor memory on chip for dense bf16 MMAs (fp32
 * accumulation over K in tensor memory), then y = bf16(fp32(acc * sb)); no
 * widened copy of the weight is made and nothing is allocated.
 * fp8_w8a16_describe_dispatch tells which.  Errors: FP8_ERR_INVALID_ARG (also
 * a granularity other than per-tensor / per-channel), FP8_ERR_ALIGNMENT,
 * FP8_ERR_UNSUPPORTED, FP8_ERR_CUDA. */
fp8_status fp8_w8a16_mm(const void *x, const void *W, const float *scale_b, int granularity, int out_dtype,
                        int64_t M, int64_t N, int64_t K, void *out, void *stream);

/* fp8_w8a16_mm with launch flags (fp8_flags), as fp8_scaled_mm_ex. */
fp8_status fp8_w8a16_mm_ex(const void *x, const void *W, const float *scale_b, int granularity, int out_dtype,
                           int64_t M, int64_t N, int64_t K, void *out, void *stream, unsigned flags);

/* FP8_KERNEL_W16_GEMV for 1 <= M <= 4 with M * K <= 20480 (the GEMV keeps the
 * tokens in 40 KB of shared memory as bf16), otherwise FP8_KERNEL_W16_DECODE
 * for 1 <= M <= 32 and FP8_KERNEL_W16_DENSE for M >= 33; FP8_KERNEL_NONE for
 * M == 0, -1 for sizes fp8_w8a16_mm rejects.  Pure. */
int fp8_w8a16_describe_dispatch(int64_t M, int64_t N, int64_t K);

/* fp8_widen_weight -- out[n,k] = bf16_rne( fp32(dec(W[n,k]) * s) ), s =
 * scale_b[0] (FP8_GRAN_PER_TENSOR) or scale_b[n] (FP8_GRAN_PER_CHANNEL): one
 * binary32 multiply rounded to nearest, then rounded to bf16 (the weight the
 * pages' large-M branch dequantises; fp8_w8a16_mm's own branch widens with s
 * = 1, exactly, and scales the result instead).  W E4M3 [N,K], out bf16
 * [N,K], both 16-byte aligned; K % 16 == 0.
 * Errors: FP8_ERR_INVALID_ARG, FP8_ERR_ALIGNMENT, FP8_ERR_CUDA. */
fp8_status fp8_widen_weight(const void *W, const float *scale_b, int granularity, int64_t N, int64_t K, void *out,
                            void *stream);

/* quant_fp8_static -- static per-tensor E4M3 quantisation, q = e4m3_rne_sat(x / s).
 *
 * Source: [P3] "Ranked follow-ons from the same audit" (QuantFp8Static).
 *
 *   x      bf16 [M,K], 16-byte aligned;  scale f32 [1] (device);
 *   out    E4M3 [M,K], 16-byte aligned;  K % 16 == 0. */
fp8_status quant_fp8_static(const void *x, const float *scale, void *out, int64_t M, int64_t K,
                            void *stream);

/* Human-readable name of a status code (a static string; never NULL). */
const char *fp8_status_string(int status);

/* Which kernel fp8_scaled_mm runs for this problem (an fp8_kernel_id), or -1
 * for arguments fp8_scaled_mm would reject.  Host-only, pure: it reads no
 * device state, so a caller can assert the kernel before capturing a graph.
 * FP8_KERNEL_DECODE_SPLITK for 1 <= M <= 32, FP8_KERNEL_PREFILL for M >= 33.
 * Source: [P4] commit message: the M-vs-threshold branch is a pure function
 * of M so that a graph captured at a padded M freezes the branch eager
 * execution would take. */
int fp8_describe_dispatch(int64_t M, int64_t N, int64_t K, int granularity);

/* Number of CTAs the decode kernel launches for this shape on the current
 * device with per-tensor / per-channel / per-token scales, or -1 if the shape
 * does not go to the decode kernel.  Host-only. */
int fp8_decode_ctas(int64_t M, int64_t N, int64_t K);

/* The decode kernel's plan for this shape and granularity on a device with
 * `num_sms` streaming multiprocessors; each returns -1 if the arguments do not
 * go to the decode kernel.  Pure and host-only (usable without a GPU).
 *
 * The kernel runs in one of two modes: clusters of S CTAs per 128-row output
 * tile, each CTA taking 1/S of the tile's K range (ctas = ceil(N/128) * S;
 * fp8_decode_split_for_sms returns S), or a persistent stream-K grid of at
 * most two CTAs per SM over which the (tile x 128-wide k-block) units are
 * divided evenly (split returns 0; ctas = min(2 * num_sms, units /
 * ceil(kb/7)) with kb = ceil(K/128), so at most 8 CTAs share a tile).  S =
 * floor(floor(8 * num_sms / 5) / tiles), at least 1 and at most kb, and 1 when
 * K <= 256; clusters when S <= 8, stream-K otherwise.  The plan is the same
 * for every granularity.
 *
 * fp8_decode_exact_for_sms returns 1 when the tile sums are exact (every
 * granularity but blockwise, K <= 262,016): each 128-wide k-block's binary32
 * tensor-core partial is added as an integer multiple of 2^-18, so the result
 * does not depend on how K is divided among CTAs (merged and split
 * projections, and a token alone or in any batch of up to 32, give the same
 * bits); 0 for blockwise scaling (k-block parts added with TwoSum). */
int fp8_decode_ctas_for_sms(int64_t M, int64_t N, int64_t K, int granularity, int num_sms);
int fp8_decode_split_for_sms(int64_t M, int64_t N, int64_t K, int granularity, int num_sms);
int fp8_decode_exact_for_sms(int64_t M, int64_t N, int64_t K, int granularity, int num_sms);

/* Device error word.  Kernels never trap: a bounded wait that runs out sets a
 * bit here and the kernel finishes without waiting further (its outputs are
 * then invalid).  fp8_get_device_error synchronises
 * `stream`, copies the word for the current device into *word (host pointer,
 * may be NULL) and returns FP8_ERR_DEVICE if it is non-zero.  Not for the hot
 * path.  fp8_clear_device_error zeroes the word and the decode GEMM's
 * arrival counters (synchronously). */
fp8_status fp8_get_device_error(void *stream, uint32_t *word);
fp8_status fp8_clear_device_error(void);

/* Self-test of the failure path: launches one thread that waits, with the
 * kernels' own bounded wait, for an mbarrier phase that nothing completes.
 * After timeout_us (1 .. 2,000,000) it gives up, sets bit 13 (0x2000) of the
 * device error word and returns, so the context stays usable; a following
 * fp8_get_device_error reports FP8_ERR_DEVICE with that bit.  No fault, trap
 * or hang is involved.  Errors: FP8_ERR_INVALID_ARG, FP8_ERR_CUDA. */
fp8_status fp8_selftest_bounded_wait(uint32_t timeout_us, void *stream);

/* Makes `device` the current device of this library's CUDA runtime for the
 * calling thread (the library links its own copy of the runtime, so a host
 * program that switches devices through another runtime tells it here).
 * Returns FP8_ERR_INVALID_ARG for a negative index, FP8_ERR_CUDA if the
 * runtime refuses the device. */
fp8_status fp8_set_device(int device);

/* Library version as an integer (major * 10000 + minor * 100 + patch). */
int fp8_library_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8W8A8_H_ */
