// Thin inline-PTX wrappers for sm_103a: mbarriers, bulk (TMA) copies,
// programmatic dependent launch, the global timer, bf16 unpacking.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"

namespace tcl {

// A bounded on-chip wait gives up after this long and reports LORA_DEV_TIMEOUT.
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps in hardware (up to hint_ns) instead of re-issuing the test, so
// waiting warps leave the shared-memory pipe to the warps doing work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Waits for the barrier phase with the given parity, for at most limit_ns
// (WAIT_LIMIT_NS unless a caller passes less); on expiry sets
// LORA_DEV_TIMEOUT in *status and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int32_t *status,
                                                  uint64_t limit_ns = WAIT_LIMIT_NS)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        for (int i = 0; i < 8; ++i)
            if (mbar_try_wait_sleep(bar, parity, 2000))
                return true;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, LORA_DEV_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ unsigned ld_acquire_gpu_u32(const void *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits until the counter *cnt (written by other CTAs) has reached `target`
// -- (int)(*cnt - target) >= 0, so a counter may wrap around --, for at most
// limit_ns; on expiry sets LORA_DEV_TIMEOUT in *status and returns false.
// The read that ends the wait has acquire semantics at GPU scope.
__device__ __forceinline__ bool wait_count_bounded(const void *cnt, unsigned target, int32_t *status,
                                                   uint64_t limit_ns = WAIT_LIMIT_NS)
{
    if ((int)(ld_acquire_gpu_u32(cnt) - target) >= 0)
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        for (int i = 0; i < 16; ++i) {
            if ((int)(ld_acquire_gpu_u32(cnt) - target) >= 0)
                return true;
            __nanosleep(32);
        }
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, LORA_DEV_TIMEOUT);
            return false;
        }
    }
}

// One bulk (non-tensor TMA) copy global -> shared, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only), grouped with commit/wait.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrive on `bar` once all of this thread's earlier cp.async copies have landed
// (the arrival counts against the barrier's initial count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue; wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Thread-block clusters: rank in the cluster, a full cluster barrier, and a
// 16-byte load from the same offset in another CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float4 ld_dsmem_f4(const void *local, uint32_t rank)
{
    uint32_t raddr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_u32(local)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(raddr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint4 lds128(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

// Retained rank of adapter a for this call: -1 unregistered, -2 out of range.
__device__ __forceinline__ int effective_rank(const PoolDev &pool, const int32_t *ranks, int a)
{
    int reg = pool.reg_rank[a];
    if (reg < 0)
        return -1;
    int k = ranks ? ranks[a] : reg;
    if (k < 0 || k > pool.r_max)
        return -2;
    return k;
}

}  // namespace tcl
