// ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the kernels use:
// mbarriers (with bounded waits), TMA tensor loads, tcgen05 tensor-core MMA /
// TMEM, thread-block-cluster shared memory, and programmatic dependent launch.
//
// Every wait here is bounded: a wait that does not complete within
// kWaitTimeoutNs sets a bit in the caller's device error word and returns
// false, so a broken pipeline ends the kernel with an error status instead of
// hanging the GPU.
#pragma once
#include <cstdint>

namespace fp8k {

constexpr unsigned long long kWaitTimeoutNs = 1000000000ull;  // 1 s

// Error-word bits (OR-ed into the word passed to every kernel).
enum : uint32_t {
    kErrDecodeFullWait = 1u << 0,
    kErrDecodeEmptyWait = 1u << 1,
    kErrDecodeAccumWait = 1u << 2,
    kErrDecodeTmemFullWait = 1u << 3,
    kErrDecodeTmemEmptyWait = 1u << 8,
    kErrDecodeFixup = 1u << 9,
    kErrW16FullWait = 1u << 10,     // weight-only kernel: a stage's TMA loads
    kErrW16AEmptyWait = 1u << 11,   // weight-only kernel: a widened weight tile freed by the MMA
    kErrW16AFullWait = 1u << 12,    // weight-only kernel: a widened weight tile written
    kErrSelfTestWait = 1u << 13,    // fp8_selftest_bounded_wait: the wait nothing completes
    kErrPrefillFullWait = 1u << 4,
    kErrPrefillEmptyWait = 1u << 5,
    kErrPrefillAccumWait = 1u << 6,
    kErrPrefillAccumEmptyWait = 1u << 7,
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (TMA, tcgen05) and
// to the other CTAs of the cluster.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on an mbarrier of any CTA of the cluster (`bar` from map_to_rank),
// releasing this thread's earlier memory operations at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test with a suspend-time hint: the thread sleeps (issuing nothing)
// until the phase completes or about `hint_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and
// sets `code` in *err) if it has not completed after timeout_ns (mbar_wait:
// kWaitTimeoutNs).  Waiting
// threads sleep in the barrier instead of spinning, so they take no issue
// slots from the warps that do the work (the hardware wakes them when the
// phase completes).
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint32_t *err, uint32_t code,
                                              unsigned long long timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) {
            atomicOr(err, code);
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t *err, uint32_t code) {
    return mbar_wait_for(bar, parity, err, code, kWaitTimeoutNs);
}

// --------------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load of one box at (x = innermost coordinate, y) into shared memory;
// completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// The CTA-pair form: the box lands in this CTA's shared memory and its
// completion is signalled on `bar`, which may be the peer CTA's mbarrier (a
// shared::cluster address from map_to_rank), for MMAs issued with
// cta_group::2 by the pair's leader.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *tmap, uint32_t bar, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Same, with an L2 cache-policy hint (from createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void *tmap, uint32_t bar, int32_t x, int32_t y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Bulk tensor store of a 2-D box from this CTA's shared memory to global
// memory, in the calling thread's current bulk group (elements outside the
// tensor are not written).
__device__ __forceinline__ void tma_store_2d(const void *tmap, uint32_t src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the calling thread's bulk groups have finished reading their
// shared-memory sources (the buffers may be written again).
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until the calling thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Barrier `id` (1..15) of `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Orders this thread's earlier generic-proxy writes to shared memory before
// later async-proxy accesses (TMA, tcgen05.mma operand reads) of it.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ----------------------------------------------------------------- tcgen05 --

// Allocates `ncols` TMEM columns (power of two >= 32); must be executed by one
// whole warp.  The TMEM address is written to shared memory at `holder`.
__device__ __forceinline__ void tmem_alloc(uint32_t holder, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// CTA-pair tensor memory (cta_group::2): one warp of each CTA of the pair
// executes these together; the same columns are allocated in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t holder, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row swizzle atoms of 1024 bytes
// (stride-dimension byte offset 1024), a single atom along K (leading offset
// unused), descriptor version 1, swizzle mode 2 (128B).  The tile base must be
// 1024-byte aligned; `addr` may carry a K offset of a multiple of 32 bytes
// inside the 128-byte row.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);           // start address, bits 0-13
    d |= static_cast<uint64_t>(0u) << 16;                         // leading byte offset, bits 16-29
    d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;    // stride byte offset, bits 32-45
    d |= static_cast<uint64_t>(1u) << 46;                         // version, bits 46-47
    d |= static_cast<uint64_t>(2u) << 61;                         // layout: 128-byte swizzle, bits 61-63
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with E4M3 A and B, both
// K-major, an FP32 accumulator, and an M x N tile.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t m, uint32_t n) {
    return (1u << 4)            // D format: F32
           | (0u << 7)          // A format: E4M3
           | (0u << 10)         // B format: E4M3
           | (0u << 15)         // A K-major
           | (0u << 16)         // B K-major
           | ((n >> 3) << 17)   // N / 8, bits 17-22
           | ((m >> 4) << 24);  // M / 16, bits 24-28
}

// Instruction descriptor of tcgen05.mma kind::f16 with BF16 A and B, both
// K-major, an FP32 accumulator, and an M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t m, uint32_t n) {
    return (1u << 4)            // D format: F32
           | (1u << 7)          // A format: BF16
           | (1u << 10)         // B format: BF16
           | (0u << 15)         // A K-major
           | (0u << 16)         // B K-major
           | ((n >> 3) << 17)   // N / 8, bits 17-22
           | ((m >> 4) << 24);  // M / 16, bits 24-28
}

// Each thread of the warp writes 32 consecutive 32-bit TMEM columns of its
// lane (lane = the warp's 32-lane quarter + thread index).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem]^T for BF16 operands (K = 16 per instruction):
// A's 128 rows in the 128 TMEM lanes, two K elements per 32-bit column (the
// lower K index in the low half), 8 columns per instruction.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives (once) on `bar` when every tcgen05.mma this thread issued so far has
// completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T over a CTA pair (cta_group::2), issued by
// one thread of the pair's leader: A's M = 256 rows are the two CTAs' 128-row
// tiles, B's N columns are split between the CTAs' shared memory (first half
// in the leader's), D's rows are in each CTA's TMEM (its 128 lanes).
__device__ __forceinline__ void mma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives (once) on the mbarrier at `bar`'s offset in every CTA of `cta_mask`
// when every cta_group::2 MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(cta_mask)
        : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit TMEM columns of its lane
// (lane = the warp's 32-lane quarter + thread index).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Two binary32 fused multiply-adds in one instruction (Blackwell's paired FP32
// pipe): (y0, y1) = (a0 * s + y0, a1 * s + y1), each rounded once to nearest.
__device__ __forceinline__ void fma2_rn(float &y0, float &y1, float a0, float a1, float s) {
    asm("{\n\t.reg .b64 ra, rs, ry;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rs, {%4, %4};\n\t"
        "mov.b64 ry, {%0, %1};\n\t"
        "fma.rn.f32x2 ry, ra, rs, ry;\n\t"
        "mov.b64 {%0, %1}, ry;\n\t}"
        : "+f"(y0), "+f"(y1)
        : "f"(a0), "f"(a1), "f"(s));
}

// (y0, y1) += (a0, a1), each add rounded once to nearest, in one instruction.
__device__ __forceinline__ void add2_rn(float &y0, float &y1, float a0, float a1) {
    asm("{\n\t.reg .b64 ra, ry;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 ry, {%0, %1};\n\t"
        "add.rn.f32x2 ry, ry, ra;\n\t"
        "mov.b64 {%0, %1}, ry;\n\t}"
        : "+f"(y0), "+f"(y1)
        : "f"(a0), "f"(a1));
}

// ------------------------------------------------------ compensated summation --

// (hi, lo) += v with Knuth's TwoSum: hi + lo represents the running sum with
// the rounding error of every addition kept in lo.  Plain binary32 adds, no
// contraction (the library is compiled with --fmad=false).
__device__ __forceinline__ void two_sum_acc(float &hi, float &lo, float v) {
    const float s = __fadd_rn(hi, v);
    const float bv = __fsub_rn(s, hi);
    const float av = __fsub_rn(s, bv);
    const float err = __fadd_rn(__fsub_rn(hi, av), __fsub_rn(v, bv));
    hi = s;
    lo = __fadd_rn(lo, err);
}

// ----------------------------------------------------------------- cluster --

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Cluster barrier halves: `arrive` (relaxed: orders nothing) and `wait`, for a
// first barrier that only establishes that every CTA of the cluster is running.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// One float from this CTA's shared memory by its shared-window address.
__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Store one float to distributed shared memory (another CTA of the cluster).
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Store to distributed shared memory (another CTA of the cluster).
__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float2 v) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y) : "memory");
}

// One float from distributed shared memory (after the cluster barrier that
// publishes it).
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Loads from distributed shared memory.  Volatile (kept in program order after
// the cluster barrier that publishes the data) but without a memory clobber,
// so several loads can be in flight at once.
__device__ __forceinline__ float2 ld_cluster_f32x2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// ------------------------------------------------ programmatic dependent launch --

// Blocks until the grids this grid depends on have completed and their memory
// is visible (a no-op when the launch had no programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allows the next grid in the stream (if launched with programmatic stream
// serialisation) to start launching.  Called only after grid_dependency_wait():
// a grid that triggered before its own wait would let its successor launch and
// trigger in turn, piling up waiting grids that hold SM resources.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace fp8k
