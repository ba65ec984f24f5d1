// kda_tc.cuh -- Blackwell (sm_103a) building blocks: mbarriers, bulk async
// copies, tcgen05 MMA with TMEM accumulators, shared-memory descriptors.
//
// Every wait is bounded by a clock budget; a wait that runs out returns false
// and the caller records KDA_DEVERR_TIMEOUT and leaves its loop, so no kernel
// of this library can spin forever.  Waits on data that the block itself
// brings in or computes use the fixed budget below; waits on flags that other
// blocks raise, and the decode's waits on its copies, take the budget of the
// launch (kda_set_wait_budget, the same fixed value by default).
#pragma once

#include <stdint.h>

namespace kda {
namespace tc {

// About one second at GB300 clocks.
constexpr long long WAIT_BUDGET_CYCLES = 2000000000ll;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking probe of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity to complete, giving up after
// `budget` clock cycles.  The clock is read before every suspending try_wait
// (which can sleep in hardware until the phase completes), so that a short
// budget, not the hardware's suspend window, bounds the wait.
__device__ __forceinline__ bool mbar_wait_for(uint64_t *bar, uint32_t parity, long long budget) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (clock64() - t0 > budget) return false;
        if (mbar_try_wait(bar, parity)) return true;
    }
}
// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, WAIT_BUDGET_CYCLES);
}
// Bounded wait that also gives up as soon as *abort (a block-local flag in
// shared memory, raised by the part of the block that timed out) is nonzero.
__device__ __forceinline__ bool mbar_wait_ab(uint64_t *bar, uint32_t parity, const volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (clock64() - t0 > WAIT_BUDGET_CYCLES) return false;
    }
    return true;
}

// ---------------------------------------------------------------- bulk copies
// global -> shared, completion counted in bytes on `bar`.  dst, src 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// One tile of a 3-D tensor map into shared memory at dst (16-byte aligned),
// completion counted in bytes on `bar`; coordinates in elements, innermost
// first (x times the element size a multiple of 16 bytes).  `map` is the
// generic address of a __grid_constant__ kernel parameter.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
// shared -> global, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Generic-proxy writes to shared memory become visible to the async proxy
// (tcgen05.mma operand reads, bulk copies) after this fence and a barrier.
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `nthreads` threads (multiple of 32); returns the OR of
// `pred` over the participating threads.
__device__ __forceinline__ bool bar_or(int id, int nthreads, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(out)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return out != 0;
}

// ---------------------------------------------------------------- TMEM
// Allocates ncols TMEM columns (a power of two >= 32).  Unless the block
// allocates again later, it then gives up its permit to allocate.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot_smem, uint32_t ncols, bool last_alloc = true) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
                 "r"(ncols)
                 : "memory");
    if (last_alloc) asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns: thread i of the warp gets row
// (lane base + i), columns col .. col + 15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *out) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 2^x by the hardware approximation (PTX ex2.approx.ftz).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// TMEM lane of row m of an M = 64 accumulator (cta_group::1): rows 16 q .. 16 q + 15
// sit in lanes 32 q .. 32 q + 15 (checked against a host product).
__host__ __device__ constexpr int m64_lane(int m) { return (m >> 4) * 32 + (m & 15); }

// ---------------------------------------------------------------- MMA
// Shared-memory matrix descriptor of a K-major operand with the 128-byte
// swizzle: rows of 128 B, 8-row groups 1024 B apart, base 1024-byte aligned.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);  // start address
    d |= (uint64_t)1 << 16;                   // leading byte offset (unused when swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                   // descriptor version
    d |= (uint64_t)2 << 61;                   // 128-byte swizzle
    return d;
}
// Descriptor of an MN-major operand (rows of the contraction index k, the M or
// N index contiguous within a row):
//   mode SWZ_128B: blocks 64 elements (128 B) wide, 16-byte chunk c of row k
//                  stored at chunk c ^ (k & 7);
//   mode SWZ_32B:  blocks 16 elements (32 B) wide, chunk c stored at
//                  c ^ ((k >> 2) & 1);
// lbo = byte stride between consecutive blocks along M/N, sbo = byte stride
// between consecutive 8-row groups along k.  Checked against a host product
// for both modes, N = 16 .. 128.
constexpr uint32_t SWZ_128B = 2, SWZ_32B = 6;
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t mode) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)mode << 61;
    return d;
}
// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with the B operand MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32_bmn(int M, int N) { return idesc_bf16_f32(M, N) | (1u << 16); }
// D[tmem] (+)= A[smem] * B[smem]^T, one K = 16 step; issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate));
}
// The same with A in TMEM (lane m = row m, K packed two bf16 per 32-bit column,
// 8 columns per K = 16 step).
__device__ __forceinline__ void mma_bf16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
            tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate));
}
// Copy 128 rows x 32 bytes (one K = 16 step of a K-major bf16 A operand,
// described like an MMA operand) from shared memory into TMEM lanes 0-127,
// 8 columns from taddr; it lands in the layout mma_bf16_ta reads (checked
// against a host product).  Ordered with this thread's MMAs.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// Arrive once on `bar` when every previously issued tcgen05.mma / tcgen05.cp of this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Warp-wide forms: every lane of a converged warp calls them with the same
// operands and one lane, picked by elect.sync over the full mask (the same
// lane at every call), issues.  Run by the whole warp, the issue code takes
// about half the time it takes behind a one-lane branch (measured: 8 products
// of M = 128, N = 64 issue in ~206 cycles instead of ~444).  A warp issues
// either only through these or only through the one-thread forms above, so
// that its commits cover its products.
__device__ __forceinline__ void mma_bf16_w(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           bool accumulate) {
    asm volatile(
        "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate));
}
__device__ __forceinline__ void mma_commit_w(uint64_t *bar) {
    asm volatile(
        "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(smem_u32(bar))
        : "memory");
}

}  // namespace tc
}  // namespace kda
