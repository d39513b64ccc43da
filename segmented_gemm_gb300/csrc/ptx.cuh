// Thin inline-PTX wrappers for sm_103a: mbarriers, TMA (tiled and gather4),
// 5th-generation tensor core (tcgen05) MMA / TMEM, proxy fences, and
// bounded waits that never hang the GPU.
#pragma once
#include <cuda.h>
#include <cstdint>

namespace lora {

// ---------------------------------------------------------------------------
// generic helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(int32_t *p, int v)
{
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_relaxed_gpu_add(int32_t *p, int v)
{
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Release only: the thread's earlier accesses are ordered before the add,
// and nothing after it waits for the result.
__device__ __forceinline__ int atom_release_gpu_add(int32_t *p, int v)
{
    int old;
    asm volatile("atom.release.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ int atom_acq_rel_gpu_add(int32_t *p, int v)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Producer side of a named barrier: signal without waiting (the waiting
// side uses bar.sync with the same id and thread count).
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: let the next kernel of the stream start its
// prologue now / wait until the kernels this one depends on have completed
// and their memory is visible (a no-op when launched without the attribute).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
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

// Cycle budgets of the bounded waits: a healthy wait ends in microseconds;
// the long budget (~1 s at 2 GHz) only runs out when something is broken,
// after which every later wait of the CTA uses the short budget so the
// kernel drains quickly instead of hanging.  A kernel may pass a shorter
// long budget of its own (the tiled kernel takes it from its parameters).
constexpr long long kWaitLong = 2000000000ll;
constexpr long long kWaitShort = 200000ll;

__device__ __forceinline__ long long wait_budget(volatile int *abort, long long budget)
{
    return *abort ? (budget < kWaitShort ? budget : kWaitShort) : budget;
}

// Wait for completion of the phase with the given parity.  Returns false
// (and raises *abort + the device status bit) when the budget runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int32_t *status, int32_t timeout_bit, long long long_budget = kWaitLong)
{
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const long long budget = wait_budget(abort, long_budget);
    const long long t0 = clock64();
    while (!mbar_try_wait(a, parity)) {
        if (clock64() - t0 > budget) {
            *abort = 1;
            atomicOr(status, timeout_bit);
            return false;
        }
    }
    return true;
}

// Spin (bounded) until *flag >= target with acquire semantics.
__device__ __forceinline__ bool wait_flag_geq(const int32_t *flag, int target, volatile int *abort,
                                              int32_t *status, int32_t timeout_bit, long long long_budget = kWaitLong)
{
    if (ld_acquire_gpu(flag) >= target) return true;
    const long long budget = wait_budget(abort, long_budget);
    const long long t0 = clock64();
    while (ld_acquire_gpu(flag) < target) {
        if (clock64() - t0 > budget) {
            *abort = 1;
            atomicOr(status, timeout_bit);
            return false;
        }
        __nanosleep(64);
    }
    return true;
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}

// Plain bulk copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) from global to shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// 2-D tiled load of the map's box at (x = inner coordinate, y = row).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *m, uint64_t *bar, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(m), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// Row gather: four arbitrary rows (each one box row high) at inner
// coordinate x, written as four consecutive box rows starting at dst.
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *m, uint64_t *bar, int x, int r0,
                                            int r1, int r2, int r3)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
        "l"(m), "r"(smem_u32(bar)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
        : "memory");
}

// ---------------------------------------------------------------------------
// cp.async (LSU path, 16 bytes per thread; src_bytes < 16 zero-fills the rest)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Arrive on `bar` once all prior cp.async of this thread have completed
// (the arrival is counted in the barrier's expected count: .noinc).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05 ops of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__device__ __forceinline__ uint32_t umma_idesc_bf16(int M, int N)
{
    return (1u << 4)                                  // D format: f32
           | (1u << 7)                                // A format: bf16
           | (1u << 10)                               // B format: bf16
           | ((static_cast<uint32_t>(N) >> 3) << 17)  // N / 8
           | ((static_cast<uint32_t>(M) >> 4) << 24); // M / 16
}

// Shared-memory matrix descriptor for a K-major operand.
//   layout: 2 = 128-byte swizzle (rows of 128 B, 8-row atoms of 1024 B)
//           6 = 32-byte swizzle  (rows of 32 B, 8-row atoms of 256 B)
//   sbo:    byte distance between consecutive 8-row groups
constexpr uint64_t kSwizzle128 = 2;
constexpr uint64_t kSwizzle32 = 6;
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t saddr, uint32_t sbo, uint64_t layout)
{
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFF)          // start address
           | (static_cast<uint64_t>(1) << 16)                      // leading offset (unused here)
           | (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32)    // stride offset
           | (static_cast<uint64_t>(1) << 46)                      // descriptor version
           | (layout << 61);
}

// 32 lanes x 32 bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Wait for outstanding tcgen05.ld; the registers are threaded through so
// no use of them can be scheduled before the wait.
// Ties registers loaded by an earlier tcgen05.ld to a preceding wait::ld (an
// ordered empty asm), so a second batch can share the first one's wait.
__device__ __forceinline__ void tmem_regs_after_wait16(uint32_t (&r)[16])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]));
}
__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// ---------------------------------------------------------------------------
// bf16 packing (round to nearest even, NaN kept quiet)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// e4m3 codes -> bf16, exactly.  An e4m3 code s.eeee.mmm shifted into bf16
// bit positions (sign to bit 15, eeeemmm to bits 10..4) is the bf16 value
// (-1)^s (1.mmm) 2^(e - 127) for e > 0, and (-1)^s (m / 8) 2^-126 for e = 0
// (a bf16 subnormal); both are the e4m3 value times 2^-120.  One bf16
// multiply by 2^120 (exact: at most 4 significant bits) rebases the
// exponent, subnormals included.  The NaN codes (eeee.mmm all ones) become
// the bf16 NaN.
__device__ __forceinline__ uint32_t e4m3_pair_to_bf16x2(uint32_t p)   // codes in bits 0..7 and 16..23
{
    const uint32_t em = p & 0x007F007Fu;
    const uint32_t t = (em << 4) | ((p & 0x00800080u) << 8);
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(0x7B807B80u));   // x 2^120 in both halves
    // em + 1 carries into bit 7 of a half only where em is 0x7F (a NaN code)
    const uint32_t nan = (((em + 0x00010001u) & 0x00800080u) >> 7) * 0xFFFFu;
    return (r & ~nan) | (0x7FC07FC0u & nan);
}

// 16 e4m3 codes (one uint4) -> 16 bf16 values (o[0..3]: codes 0..7, o[4..7]: codes 8..15).
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 c, uint32_t (&o)[8])
{
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        o[2 * k] = e4m3_pair_to_bf16x2(__byte_perm(w[k], 0u, 0x4140));       // codes 4k, 4k + 1
        o[2 * k + 1] = e4m3_pair_to_bf16x2(__byte_perm(w[k], 0u, 0x4342));   // codes 4k + 2, 4k + 3
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

}  // namespace lora
