// ptx_sync.cuh -- mbarrier, bulk-copy (TMA) and bounded grid-wait helpers for
// sm_103a, written as inline PTX.
//
// Every wait here is bounded by %globaltimer: on expiry it reports failure to
// the caller, which records QMOE_ERR_TIMEOUT in the device status word and
// unwinds without touching further data.
#pragma once
#include <stdint.h>

namespace qmoe {

constexpr int ST_TIMEOUT = 7;
constexpr int ST_DEVICE_CHECK = 8;
constexpr unsigned long long WAIT_LIMIT_NS = 200ull * 1000ull * 1000ull;   // 200 ms

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// make initialised barriers visible to the async (bulk-copy) proxy
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// order this thread's earlier generic-proxy accesses to shared memory before
// its later async-proxy (bulk copy) accesses
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// non-blocking probe of the phase with the given parity
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps in the instruction until
// the phase completes or about hint_ns pass, instead of spinning (spinning
// waiters take issue slots from the warps doing the work)
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
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

// bounded wait for the phase with the given parity; false on timeout
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (globaltimer() - t0 > WAIT_LIMIT_NS) return false;
    }
    return true;
}

// one bulk copy global -> shared, completion counted on bar (bytes % 16 == 0,
// both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// 16 bytes global -> shared through L2 only (no L1 line is filled, so values
// other SMs stored in this launch are seen once their publication was acquired);
// cp_async_wait_all waits for every such copy this thread issued
__device__ __forceinline__ void cp_async_cg16(void* dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// L2 prefetch of `bytes` (multiple of 16) at a 16-byte aligned global address
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Tagged values: a float and the tag of the launch that wrote it, in one
// 64-bit word that is stored and loaded in one access.  A reader that sees its
// own launch's tag has the value itself, so no fence or counter is needed to
// pass single values between CTAs of a co-resident grid.
__device__ __forceinline__ unsigned long long tag_pack(float v, unsigned tag) {
    return ((unsigned long long)tag << 32) | __float_as_uint(v);
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *p carries `tag`; false on timeout (v is then 0).
__device__ __forceinline__ bool poll_tagged(const unsigned long long* p, unsigned tag, float& v) {
    unsigned long long w = ld_relaxed_u64(p);
    if ((unsigned)(w >> 32) != tag) {
        const unsigned long long t0 = globaltimer();
        do {
            if (globaltimer() - t0 > WAIT_LIMIT_NS) {
                v = 0.f;
                return false;
            }
            __nanosleep(32);
            w = ld_relaxed_u64(p);
        } while ((unsigned)(w >> 32) != tag);
    }
    v = __uint_as_float((unsigned)w);
    return true;
}

// Grid-wide arrival: called by one thread of each CTA after its writes.
__device__ __forceinline__ void grid_arrive(unsigned* counter) {
    __threadfence();
    atomicAdd(counter, 1u);
}

// Bounded wait until *counter >= target; false on timeout.
__device__ __forceinline__ bool grid_wait(const unsigned* counter, unsigned target) {
    if (ld_acquire_gpu(counter) >= target) return true;
    const unsigned long long t0 = globaltimer();
    while (ld_acquire_gpu(counter) < target) {
        if (globaltimer() - t0 > WAIT_LIMIT_NS) return false;
        __nanosleep(64);
    }
    return true;
}

__device__ __forceinline__ void named_bar(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace qmoe
