// tma.cuh -- mbarrier, TMA and timer helpers shared by the TMA-fed kernels
// (grouped GEMM, router).  Device code is inline PTX for sm_103a.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// 3-D bf16 tensor map (host; defined in gemm_tc.cu): dims {d0 (contiguous), d1,
// d2}, byte strides {s1, s2}, box {b0, b1, 1}, 128-byte swizzle unless stated.
int encode_bf16_map(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1,
                    CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

constexpr unsigned long long WAIT_NS = 4000000000ull;   // bounded waits give up after 4 s
constexpr unsigned long long DRAIN_NS = 500000000ull;   // draining gives up after 0.5 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// A bounded wait that timed out anywhere on the device (this launch's other
// CTAs, or an earlier launch whose status the host has not read yet) is
// visible in the device status word; waits give up as soon as they see it,
// so one lost arrival costs one time limit, not one per CTA or per launch.
__device__ __forceinline__ bool timeout_pending(const int* status) {
    return status && *reinterpret_cast<const volatile int*>(status) == MOE_ERR_TIMEOUT;
}
// Bounded wait.  Returns false when the wait gave up (timeout, another role's
// abort, or a timeout recorded on the device); the first to time out records
// the status and raises abort.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, unsigned long long limit_ns = WAIT_NS) {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 15) == 0) {
            if (*abort_flag) return false;
            if (timeout_pending(status)) {
                *abort_flag = 1;
                return false;
            }
            if (gtimer() - t0 > limit_ns) {
                set_status(status, MOE_ERR_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}
// Bounded wait used while draining (ignores the abort flag).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = gtimer();
    while (!mbar_try(bar, parity))
        if (gtimer() - t0 > DRAIN_NS) break;
}

// ---- CTA-pair (cluster of 2) helpers ----
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// arrive on an mbarrier in another CTA of the cluster (release at cluster scope)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
// try_wait with cluster-scope acquire (barriers that other CTAs of the cluster arrive on)
__device__ __forceinline__ bool mbar_try_cl(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait, cluster-scope acquire (as mbar_wait)
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             int* status) {
    if (mbar_try_cl(bar, parity)) return true;
    const unsigned long long t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_cl(bar, parity)) return true;
        if ((it & 15) == 0) {
            if (*abort_flag) return false;
            if (timeout_pending(status)) {
                *abort_flag = 1;
                return false;
            }
            if (gtimer() - t0 > WAIT_NS) {
                set_status(status, MOE_ERR_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}
__device__ __forceinline__ void mbar_drain_cl(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = gtimer();
    while (!mbar_try_cl(bar, parity))
        if (gtimer() - t0 > DRAIN_NS) break;
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (bar: a shared::cluster address)
__device__ __forceinline__ void tma_load3_pair(const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                               int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// 4-D TMA load into this CTA's shared memory, completion counted on an mbarrier of
// either CTA of the pair (bar: a shared::cluster address)
__device__ __forceinline__ void tma_load4_pair(const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                               int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load4(const CUtensorMap* map, uint32_t dst, uint32_t bar, int c0,
                                          int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// TMA store of a shared-memory box (bulk-group completion)
__device__ __forceinline__ void tma_store3(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load3(const CUtensorMap* map, uint32_t dst, uint32_t bar, int c0,
                                          int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

}  // namespace moe
