// norm_row.cuh -- the fused RMSNorm -> static E4M3 quantisation of ONE row by
// a group of threads: the row arithmetic of the rmsnorm_quant_fp8 and
// add_rmsnorm_quant_fp8 kernels (a CTA per row).
//
// Source: "We emit F32 where vLLM emits bf16 on the biggest prefill buffers
// ..." (vllm.cpp #417), "Ranked follow-ons from the same audit": the fused
// RMSNorm -> fp8 quant, byte-exact with the unfused norm-then-quant ("quantise
// once").
//
//   q = e4m3( bf16((x * r) * gamma) / s ),   r = 1 / sqrt(ss / K + eps)
//
// The sum of squares ss is formed EXACTLY: every bf16 square is
// m^2 * 2^(2E - 268) with m < 256, so the squares of the row's top 40 binades
// are added as integers into a 128-bit fixed-point accumulator (2^94 per term
// at most, 2^110 for 2^16 terms), and any nonzero smaller term only sets a
// sticky bit.  The smaller terms add up to less than K * 2^14 units of the
// window's lowest bit, far below the rounding position (at least 2^69 units
// once a term lies below the window), so they can change the rounding only by
// a carry through a run of one bits from just below the guard bit down to
// that bound.  That case -- astronomically rare in data, but constructible --
// is detected, and the row is then summed exactly by one thread over the full
// exponent range (sticky_may_carry, exact_row_sum_squares).  The exact sum is
// rounded once to binary32, then mean = ss / K, t = mean + eps, d = sqrt(t), r = 1 / d are
// single IEEE binary32 operations; the two multiplies are separate binary32
// operations (the library is compiled without FMA contraction), bf16 and E4M3
// conversions round to nearest even (the E4M3 one saturating).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace fp8k {
namespace norm {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two values -> two E4M3 codes, `a` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 128-bit unsigned integer as (hi, lo).
struct U128 {
    uint64_t hi, lo;
};

__device__ __forceinline__ U128 add128(U128 a, U128 b) {
    U128 r;
    r.lo = a.lo + b.lo;
    r.hi = a.hi + b.hi + (r.lo < a.lo ? 1u : 0u);
    return r;
}

__device__ __forceinline__ uint64_t shr128(U128 a, int q) {  // low 64 bits of a >> q, 0 <= q < 128
    if (q == 0) return a.lo;
    if (q < 64) return (a.lo >> q) | (a.hi << (64 - q));
    return a.hi >> (q - 64);
}

__device__ __forceinline__ int bit128(U128 a, int i) {
    return static_cast<int>(i < 64 ? (a.lo >> i) & 1u : (a.hi >> (i - 64)) & 1u);
}

__device__ __forceinline__ bool any_below128(U128 a, int i) {  // any set bit at positions < i
    if (i <= 0) return false;
    if (i < 64) return (a.lo & ((1ull << i) - 1)) != 0;
    if (i == 64) return a.lo != 0;
    return a.lo != 0 || (a.hi & ((1ull << (i - 64)) - 1)) != 0;
}

// bf16 bits -> (m, E): x = +-m * 2^(E - 134) with E >= 1 (E = 1 also for subnormals).
__device__ __forceinline__ void bf16_split(uint32_t b, uint32_t &m, int &E) {
    const uint32_t e = (b >> 7) & 0xFFu, mant = b & 0x7Fu;
    m = e ? (128u | mant) : mant;
    E = e ? static_cast<int>(e) : 1;
}

// Shared scratch of one row group's reductions (one entry per warp).
struct RowScratch {
    uint32_t red_limb[5][32];  // per warp: 24-bit limbs of its partial sum
    uint32_t exact[17];        // the exact fallback's limbs (kExactLimbs)
    uint32_t red_a[32], red_b[32], red_f[32];
    float r;
};

// A group of T threads (T a multiple of 32, at most 1024), thread ti of it,
// synchronised by `sync()` (a CTA barrier or a named barrier of exactly the
// group's threads).
struct Group {
    int ti, T;
};

// A 128-bit value below 2^120 as five 24-bit limbs, and back: a sum of up
// to 32 such limbs stays below 2^29, so each limb of a group sum is one
// 32-bit warp reduction (redux.sync), the carries propagated afterwards.
__device__ __forceinline__ void to_limbs(U128 v, uint32_t (&l)[5]) {
    l[0] = static_cast<uint32_t>(v.lo) & 0xFFFFFFu;
    l[1] = static_cast<uint32_t>(v.lo >> 24) & 0xFFFFFFu;
    l[2] = (static_cast<uint32_t>(v.lo >> 48) | (static_cast<uint32_t>(v.hi) << 16)) & 0xFFFFFFu;
    l[3] = static_cast<uint32_t>(v.hi >> 8) & 0xFFFFFFu;
    l[4] = static_cast<uint32_t>(v.hi >> 32) & 0xFFFFFFu;
}

__device__ __forceinline__ void warp_sum_limbs(uint32_t (&l)[5]) {
    uint32_t c = 0;
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const uint32_t t = __reduce_add_sync(0xFFFFFFFFu, l[k]) + c;
        l[k] = k < 4 ? (t & 0xFFFFFFu) : t;
        c = t >> 24;
    }
}

// Sum of a 128-bit value and OR of a flag over the group (one barrier for
// both; the scratch fields it writes are written once per row).  Every partial and the total are below 2^120 (the
// row's sum of squares in window units is below K * 2^94 <= 2^110).
template <class Sync>
__device__ __forceinline__ U128 group_sum_u128_or(U128 v, int &flag, const Group g, RowScratch *sc, Sync sync) {
    uint32_t l[5];
    to_limbs(v, l);
    warp_sum_limbs(l);
    uint32_t f = __reduce_or_sync(0xFFFFFFFFu, static_cast<uint32_t>(flag));
    const int warp = g.ti >> 5, lane = g.ti & 31;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < 5; ++k) sc->red_limb[k][warp] = l[k];
        sc->red_f[warp] = f;
    }
    sync();
    const int nw = g.T >> 5;
#pragma unroll
    for (int k = 0; k < 5; ++k) l[k] = lane < nw ? sc->red_limb[k][lane] : 0u;
    f = lane < nw ? sc->red_f[lane] : 0u;
    warp_sum_limbs(l);
    flag = static_cast<int>(__reduce_or_sync(0xFFFFFFFFu, f));
    U128 r;
    r.lo = static_cast<uint64_t>(l[0]) | (static_cast<uint64_t>(l[1]) << 24) | (static_cast<uint64_t>(l[2]) << 48);
    r.hi = static_cast<uint64_t>(l[2] >> 16) | (static_cast<uint64_t>(l[3]) << 8) | (static_cast<uint64_t>(l[4]) << 32);
    return r;
}

// The exact sum (acc * 2^(2*elo - 268), plus a sticky bit for smaller terms)
// rounded to binary32 at 24 significant bits or the subnormal quantum 2^-149;
// NaN / Inf inputs (special 3 / 2) give NaN / Inf.
__device__ __forceinline__ float round_sum_to_f32(U128 acc, int elo, int sticky, int special) {
    if (special == 3) return __int_as_float(0x7FC00000);
    if (special == 2) return __int_as_float(0x7F800000);
    if (acc.hi == 0 && acc.lo == 0) return 0.0f;
    const int top = acc.hi ? 127 - __clzll(static_cast<long long>(acc.hi)) : 63 - __clzll(static_cast<long long>(acc.lo));
    const int q = max(top - 23, 119 - 2 * elo);
    uint64_t keep;
    if (q <= 0) {
        keep = acc.lo;  // fewer than 24 significant bits: exact
    } else {
        keep = shr128(acc, q);
        const bool half = bit128(acc, q - 1) != 0;
        const bool rest = any_below128(acc, q - 1) || sticky;
        if (half && (rest || (keep & 1u))) keep += 1;
    }
    return ldexpf(static_cast<float>(keep), (q > 0 ? q : 0) + 2 * elo - 268);
}

// True when the squares below the window (sticky set) could carry into the
// rounding of the windowed sum acc: the guard bit is 0 and every bit from
// just below it down to 2^p, p = 14 + bitlen(K), is 1 (the small terms sum to
// less than K * 2^14 < 2^p units, each being m^2 * 4^(E - elo) < 2^16 / 4).
// With the guard bit 1 the windowed sum already rounds up, as the exact sum
// does whether or not a carry reaches it.
__device__ __forceinline__ bool sticky_may_carry(U128 acc, int elo, int K) {
    if (acc.hi == 0 && acc.lo == 0) return true;
    const int top = acc.hi ? 127 - __clzll(static_cast<long long>(acc.hi)) : 63 - __clzll(static_cast<long long>(acc.lo));
    const int q = max(top - 23, 119 - 2 * elo);
    if (q < 2) return true;
    if (bit128(acc, q - 1)) return false;
    const int p = 14 + (32 - __clz(K));
    for (int i = q - 2; i >= p; --i)
        if (!bit128(acc, i)) return false;
    return true;
}

// The exact sum of squares of a finite row by one thread, over the whole
// exponent range: 17 limbs of 32 bits in shared memory (`limb`), bit i worth
// 2^(i - 266) (a square is m^2 * 2^(2E - 2) such units, E >= 1, below 2^522;
// 2^16 of them below 2^538), rounded once to binary32 at 24 significant bits
// or the subnormal quantum 2^-149 (= 2^117 units).  Slow (tens of
// microseconds for K = 5120); taken only when sticky_may_carry says the
// windowed sum cannot decide the rounding.  The limbs live in shared memory so
// that this rare path needs no local-memory frame in the kernel.
constexpr int kExactLimbs = 17;

__device__ __noinline__ float exact_row_sum_squares(const uint4 *row, int nvec, uint32_t *limb) {
    for (int i = 0; i < kExactLimbs; ++i) limb[i] = 0;
    for (int i = 0; i < nvec; ++i) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            uint32_t m;
            int E;
            bf16_split((w[h >> 1] >> (16 * (h & 1))) & 0x7FFFu, m, E);
            if (m == 0) continue;
            const int sh = 2 * E - 2;
            uint64_t add = static_cast<uint64_t>(m * m) << (sh & 31);  // below 2^47
            for (int k = sh >> 5; add != 0 && k < kExactLimbs; ++k) {
                const uint64_t t = static_cast<uint64_t>(limb[k]) + (add & 0xFFFFFFFFull);
                limb[k] = static_cast<uint32_t>(t);
                add = (add >> 32) + (t >> 32);
            }
        }
    }
    int top = -1;
    for (int k = kExactLimbs - 1; k >= 0 && top < 0; --k)
        if (limb[k]) top = 32 * k + 31 - __clz(static_cast<int>(limb[k]));
    if (top < 0) return 0.0f;
    const int q = max(top - 23, 117);
    uint32_t keep = 0;
    for (int i = top; i >= q; --i) keep = (keep << 1) | ((limb[i >> 5] >> (i & 31)) & 1u);
    const uint32_t half = (limb[(q - 1) >> 5] >> ((q - 1) & 31)) & 1u;
    bool rest = false;
    for (int i = q - 2; i >= 0 && !rest; --i) rest = ((limb[i >> 5] >> (i & 31)) & 1u) != 0;
    if (half && (rest || (keep & 1u))) keep += 1;
    return ldexpf(static_cast<float>(keep), q - 266);
}

// Max of two non-negative ints over the group (one barrier for both; the
// scratch fields it writes are written once per row).
template <class Sync>
__device__ __forceinline__ int2 group_max2(int2 v, const Group g, RowScratch *sc, Sync sync) {
    uint32_t a = __reduce_max_sync(0xFFFFFFFFu, static_cast<uint32_t>(v.x));
    uint32_t b = __reduce_max_sync(0xFFFFFFFFu, static_cast<uint32_t>(v.y));
    const int warp = g.ti >> 5, lane = g.ti & 31;
    if (lane == 0) {
        sc->red_a[warp] = a;
        sc->red_b[warp] = b;
    }
    sync();
    const int nw = g.T >> 5;
    a = lane < nw ? sc->red_a[lane] : 0u;
    b = lane < nw ? sc->red_b[lane] : 0u;
    return make_int2(static_cast<int>(__reduce_max_sync(0xFFFFFFFFu, a)),
                     static_cast<int>(__reduce_max_sync(0xFFFFFFFFu, b)));
}

// Exponent field of the largest |element| of a vector of 8 bf16 (0 for zeros
// and subnormals; 0xFF when an Inf or NaN is present), two lanes at a time.
__device__ __forceinline__ uint32_t vec_max_exp(const uint4 v) {
    uint32_t r = __vmaxu2(__vmaxu2(v.x & 0x7F807F80u, v.y & 0x7F807F80u), __vmaxu2(v.z & 0x7F807F80u, v.w & 0x7F807F80u));
    r = max(r & 0xFFFFu, r >> 16);
    return r >> 7;
}

// 3 = some element is a NaN, 2 = some element is an Inf, 0 = neither.
__device__ __forceinline__ int vec_special(const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    int sp = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t b = (w[i >> 1] >> (16 * (i & 1))) & 0x7FFFu;
        if ((b >> 7) == 0xFFu) sp = max(sp, (b & 0x7Fu) ? 3 : 2);
    }
    return sp;
}

// The squares of one vector's elements of binade E >= elo, added exactly as
// integers (element m * 2^(E - 134) contributes m^2 * 2^(2 (E - elo)) units)
// into three 64-bit partial sums at 32-bit offsets (each contribution is
// below 2^47 and a thread adds at most 2^16 of them, so none overflows);
// smaller nonzero elements only set the sticky bit.
__device__ __forceinline__ void vec_sum_squares(const uint4 v, int elo, uint64_t &a0, uint64_t &a1, uint64_t &a2,
                                                int &sticky) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t b = (w[i >> 1] >> (16 * (i & 1))) & 0x7FFFu;
        const uint32_t e = b >> 7, mant = b & 0x7Fu;
        const uint32_t m = e ? (mant | 0x80u) : mant;
        const int E = e ? static_cast<int>(e) : 1;
        const bool nz = b != 0;
        const bool in = nz && E >= elo;
        sticky |= (nz && E < elo) ? 1 : 0;
        const int sh = in ? 2 * (E - elo) : 0;
        const uint64_t c = in ? (static_cast<uint64_t>(m * m) << (sh & 31)) : 0ull;
        const int k = sh >> 5;
        a0 += (k == 0) ? c : 0ull;
        a1 += (k == 1) ? c : 0ull;
        a2 += (k == 2) ? c : 0ull;
    }
}

// One row: xr / gamma / orow hold nvec vectors of 8 elements (K = 8 * nvec);
// thread ti handles vectors ti, ti + T, ... (at most V of them).  Every
// thread of the group must call this (it synchronises the group).
// bf16( fp32(a) + fp32(b) ) for the two bf16 halves of a pair of words.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(bf16_lo(a), bf16_lo(b))));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(bf16_hi(a), bf16_hi(b))));
    return lo | (hi << 16);
}

template <int V, bool kPrefetchGamma, bool kResidual = false, class Sync>
__device__ __forceinline__ void rmsnorm_quant_row(const uint4 *__restrict__ xr, const uint4 *__restrict__ gamma,
                                                  float eps, float s, uint2 *__restrict__ orow, int nvec, int K,
                                                  const Group g, RowScratch *sc, Sync sync,
                                                  uint4 *resid = nullptr) {
    // With kResidual the row is first replaced by h = bf16(fp32(x) + fp32(res))
    // (one binary32 addition, rounded to bf16), which is also written back
    // over the residual row `resid` (each element by the thread that read it).
    uint4 v[V], gm[kPrefetchGamma ? V : 1];
    uint32_t efield = 0;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = g.ti + j * g.T;
        if (idx < nvec) {
            v[j] = ld_stream(xr + idx);
            if (kResidual) {
                const uint4 rv = resid[idx];
                v[j] = make_uint4(add_bf16x2(v[j].x, rv.x), add_bf16x2(v[j].y, rv.y), add_bf16x2(v[j].z, rv.z),
                                  add_bf16x2(v[j].w, rv.w));
                resid[idx] = v[j];
            }
            if (kPrefetchGamma) gm[j] = __ldg(gamma + idx);
            efield = max(efield, vec_max_exp(v[j]));
        }
    }
    int special = 0;  // 3 = a NaN, 2 = an Inf (the max keeps NaN)
    if (efield == 0xFFu) {
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int idx = g.ti + j * g.T;
            if (idx < nvec) special = max(special, vec_special(v[j]));
        }
    }
    const int2 red = group_max2(make_int2(static_cast<int>(efield), special), g, sc, sync);
    special = red.y;
    // The largest binade of a finite element (subnormals count as binade 1;
    // an all-subnormal or all-zero row gives the same window as binade 1).
    const int emax = special ? 0 : red.x;
    const int elo = max(emax - 39, 1);
    uint64_t a0 = 0, a1 = 0, a2 = 0;
    int sticky = 0;
    if (!special) {
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int idx = g.ti + j * g.T;
            if (idx < nvec) vec_sum_squares(v[j], elo, a0, a1, a2, sticky);
        }
    }
    // a0 + a1 * 2^32 + a2 * 2^64 as one 128-bit number
    U128 acc = {a2, a0};
    acc = add128(acc, U128{a1 >> 32, a1 << 32});
    acc = group_sum_u128_or(acc, sticky, g, sc, sync);
    if (g.ti == 0) {
        // (with kResidual the summed row is already in `resid`: every thread
        // wrote its vectors before the group's barriers above)
        const float ss = (!special && sticky && sticky_may_carry(acc, elo, K))
                             ? exact_row_sum_squares(kResidual ? resid : xr, nvec, sc->exact)
                             : round_sum_to_f32(acc, elo, sticky, special);
        const float mean = __fdiv_rn(ss, static_cast<float>(K));
        const float t = __fadd_rn(mean, eps);
        const float d = __fsqrt_rn(t);
        sc->r = __fdiv_rn(1.0f, d);
    }
    sync();
    const float r = sc->r;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = g.ti + j * g.T;
        if (idx < nvec) {
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            const uint4 gv = kPrefetchGamma ? gm[j] : __ldg(gamma + idx);
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
            uint32_t p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float h0 =
                    __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(bf16_lo(w[i]), r), bf16_lo(gw[i]))));
                const float h1 =
                    __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(bf16_hi(w[i]), r), bf16_hi(gw[i]))));
                p[i] = e4m3x2(__fdiv_rn(h0, s), __fdiv_rn(h1, s));
            }
            orow[idx] = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
        }
    }
}

}  // namespace norm
}  // namespace fp8k
