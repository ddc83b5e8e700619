// splitk.cuh -- pieces shared by the split-K decode kernels (the W8A8 decode
// GEMM and the weight-only W8A16 one): the stream-K division of units among
// CTAs, the kernel arguments, the bounded CTA-wide wait and the last
// arriver's deterministic sum of a tile's K-range parts.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fp8k {
namespace {

// Units [u0, u1) of CTA c out of U units over G CTAs, and the CTA owning unit u.
__host__ __device__ __forceinline__ int64_t unit_begin(int64_t c, int64_t U, int64_t G) { return (c * U) / G; }
__host__ __device__ __forceinline__ int64_t unit_owner(int64_t u, int64_t U, int64_t G) {
    return ((u + 1) * G - 1) / U;
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// The most CTAs that can share one tile's K range with two CTAs per SM on a
// 152-SM part is ceil(kb_total / units per CTA) + 1; the planner keeps it at
// or below this bound (a fixup reads one slot per sharing CTA at once).
constexpr int kMaxFixupSegs = 8;


struct DecodeArgs {
    const float *scale_a;
    const float *scale_b;
    __nv_bfloat16 *out;
    uint32_t *err;
    uint32_t *counters;
    float *slots;
    int64_t units;
    int gran, M, N, kb_total, n_tiles, stages, weights_static;
    int split;  // cluster mode: CTAs (one cluster) per tile; 0 in stream-K mode
    int tok_rows;     // token rows a token box carries (M); the rest of the token tile stays zero
};

// Cluster mode: at most this many CTAs (parts) per tile.
constexpr int kMaxClusterParts = 8;

// Cluster mode: rows [red_row_begin(q, S), red_row_begin(q + 1, S)) of a tile
// are summed by CTA q of the tile's cluster; at most ceil(128 / S) of them.
__host__ __device__ __forceinline__ int red_row_begin(int q, int S) { return (q * kDecodeRows + S - 1) / S; }

// A bounded wait that gives up at once when the CTA has already given up:
// after one wait times out the kernel keeps its control flow (so barriers stay
// matched) but stops waiting; the error word says the results are invalid.
__device__ __forceinline__ bool cta_wait(uint32_t bar, uint32_t parity, uint32_t *err, uint32_t code,
                                         volatile uint32_t *abort) {
    if (*abort) return false;
    if (mbar_wait(bar, parity, err, code)) return true;
    *abort = 1u;
    return false;
}

// The last-arriving CTA's sum of a tile's K-range parts: every valid entry
// ([token column][weight row] of the tile) summed over the parts in k order
// (TwoSum), scaled, rounded to bf16 and stored.  Thread dt of NT owns VEC
// float4 groups of entries per round, and all SEGS x VEC loads of a round are
// issued before any is used.
template <int SEGS, int VEC, int NT>
__device__ __forceinline__ void fixup_sum(const DecodeArgs &args, const int64_t *slot, int nseg, int entries, int dt,
                                          int n_tile, int m0, bool sa_vec, bool sb_vec, float sa0, float sb0) {
    for (int e0 = 4 * VEC * dt; e0 < entries; e0 += 4 * VEC * NT) {
        float sa_e[4 * VEC], sb_e[4 * VEC];  // the scales, requested before the slots
#pragma unroll
        for (int q = 0; q < 4 * VEC; ++q) {
            const int e = min(e0 + q, entries - 1);
            const int m = e / kDecodeRows, nn = n_tile * kDecodeRows + (e % kDecodeRows);
            sa_e[q] = sa_vec ? __ldg(args.scale_a + m0 + m) : sa0;
            sb_e[q] = (sb_vec && nn < args.N) ? __ldg(args.scale_b + nn) : sb0;
        }
        float4 v[SEGS][VEC];
#pragma unroll
        for (int j = 0; j < SEGS; ++j)
#pragma unroll
            for (int c = 0; c < VEC; ++c)
                if (j < nseg && e0 + 4 * c < entries)
                    v[j][c] = __ldcg(reinterpret_cast<const float4 *>(args.slots + slot[j] + e0 + 4 * c));
        float h[4 * VEC], l[4 * VEC];
#pragma unroll
        for (int q = 0; q < 4 * VEC; ++q) h[q] = l[q] = 0.0f;
#pragma unroll
        for (int j = 0; j < SEGS; ++j) {
            if (j < nseg) {
#pragma unroll
                for (int c = 0; c < VEC; ++c) {
                    if (e0 + 4 * c < entries) {
                        two_sum_acc(h[4 * c + 0], l[4 * c + 0], v[j][c].x);
                        two_sum_acc(h[4 * c + 1], l[4 * c + 1], v[j][c].y);
                        two_sum_acc(h[4 * c + 2], l[4 * c + 2], v[j][c].z);
                        two_sum_acc(h[4 * c + 3], l[4 * c + 3], v[j][c].w);
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 4 * VEC; ++q) {
            const int e = e0 + q;
            const int m = e / kDecodeRows, nn = n_tile * kDecodeRows + (e % kDecodeRows);
            if (e < entries && nn < args.N)
                args.out[static_cast<int64_t>(m0 + m) * args.N + nn] =
                    __float2bfloat16_rn(__fmul_rn(__fmul_rn(__fadd_rn(h[q], l[q]), sa_e[q]), sb_e[q]));
        }
    }
}

}  // namespace
}  // namespace fp8k
