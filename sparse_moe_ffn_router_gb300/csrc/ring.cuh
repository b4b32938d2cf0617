// ring.cuh -- pieces shared by the persistent weight-streaming kernels: 1-D TMA bulk copies,
// programmatic-dependent-launch controls, the consumer-warp barrier, warp-level bf16 MMA
// (m16n8k16, fp32 accumulate) fed by ldmatrix, and gpu-scope release/acquire flags.
#pragma once

#include "launch.h"
#include "sm100.cuh"

namespace moe {

constexpr int kConsumers = 256;         // 8 consumer warps
constexpr int kWarps = kConsumers / 32;
constexpr int kStreamThreads = kConsumers + 32;

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// Barrier of the consumer warps that ANDs a predicate over them, so all consumers take the same
// branch after a bounded wait (none is left behind in a named barrier).
__device__ __forceinline__ bool consumers_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "n"(kConsumers)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------------------------------
// Warp-level bf16 MMA (m16n8k16, fp32 accumulate) fed by ldmatrix from padded rows.

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


// ---------------------------------------------------------------------------------------
// gpu-scope flags between CTAs of one persistent grid

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_acq_rel_add(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ uint32_t atom_release_add(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Generic-proxy writes made visible (acquired) before now become visible to TMA reads issued
// after this fence.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Poll until *p >= target (acquire), backing off from 32 ns to 1 us between polls so that
// many waiters do not hammer one L2 line; false after ~1 s.
__device__ __forceinline__ bool wait_at_least(const uint32_t* p, uint32_t target) {
    if (ld_acquire(p) >= target) return true;
    const uint64_t t0 = global_ns();
    uint32_t ns = 32;
    for (;;) {
        __nanosleep(ns);
        if (ld_acquire(p) >= target) return true;
        if (ns < 1024) ns <<= 1;
        if (global_ns() - t0 > 1000000000ull) return false;
    }
}

}  // namespace moe
