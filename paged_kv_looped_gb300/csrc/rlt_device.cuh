// Device helpers shared by the sm_103a kernels: bf16 unpacking, mbarrier and
// bulk-copy (TMA, non-tensor) wrappers in inline PTX, bounded waits and the
// device error word.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "rlt.h"

namespace rlt {

constexpr unsigned kFullMask = 0xffffffffu;

// A copy wait gives up after this long (nanoseconds of %globaltimer) and
// records RLT_DEVERR_TIMEOUT instead of spinning forever.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ void record_error(unsigned int *err, unsigned int bits)
{
    if (err != nullptr)
        atomicOr(err, bits);
}

// ---------------------------------------------------------------- bf16 bits
// A bf16 value is the top half of an fp32 with the same bits.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// fp32 -> bf16 bits, round to nearest even (inputs here are finite).
__device__ __forceinline__ uint32_t bf16_bits(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7f800000u) == 0x7f800000u)          // inf / nan: keep, quiet nan
        return (u >> 16) | ((u & 0x007fffffu) ? 0x40u : 0u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return u >> 16;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    return bf16_bits(lo) | (bf16_bits(hi) << 16);
}

// Same rounding (nearest even) in one instruction: hi -> upper half, lo -> lower half.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^x on the special-function unit (flushes denormal results to zero).
__device__ __forceinline__ float fast_exp2(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// ------------------------------------------------------------ shared memory
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking probe: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete; false after the time limit
// (limit_ns of %globaltimer, and at most 2^32 - 1 tries).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1; it != 0; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 255u) == 0u && global_ns() - t0 > limit_ns)
            return false;
    }
    return false;
}

// As mbar_wait, but also gives up as soon as *abort turns non-zero (another
// role of the CTA gave up first).
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity,
                                                   const volatile int *abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1; it != 0; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0u && (*abort != 0 || global_ns() - t0 > kWaitLimitNs))
            return false;
    }
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same buffers.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One contiguous global -> shared bulk copy that completes `bytes` of the
// barrier's transaction count.  dst and src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// The same copy for data read once per call (a request's own K/V rows): its L2 lines are
// marked evict-first, so that what the call reads again soon -- the partials the combine
// merges, q, page tables, plans -- keeps its place in L2.  The policy is made in place (one
// instruction), so no register carries it through a loop.
__device__ __forceinline__ void bulk_load_once(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], pol;\n\t}" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start before the
// kernel ahead of it in the stream has finished.  launch_dependents lets the
// kernel behind this one start (once every CTA has issued it or exited);
// pdl_wait blocks the calling thread until every grid this one depends on has
// completed and its memory writes are visible.  Without such a launch both are
// no-ops.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------- warp helpers
__device__ __forceinline__ float warp_max_xor(float v, int from)
{
    for (int o = from; o < 32; o <<= 1)
        v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum_xor(float v, int from)
{
    for (int o = from; o < 32; o <<= 1)
        v += __shfl_xor_sync(kFullMask, v, o);
    return v;
}

}  // namespace rlt
