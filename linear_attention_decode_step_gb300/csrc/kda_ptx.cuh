// Thin inline-PTX wrappers for sm_100-class features used by the kernels:
// mbarriers, bulk and tiled-tensor (TMA) copies, named barriers, L2 cache
// policies. Every mbarrier wait is bounded: it gives up after a clock64()
// deadline and reports failure to the caller, which records an error and
// returns instead of spinning forever.
#pragma once

#include <cstdint>

// Budget (clock cycles) of every wait on data or work in flight: about two
// seconds at 2 GHz. A build may lower it (-DKDA_WAIT_BUDGET=...) so that
// waits give up before legitimate copies land, to exercise the exit paths;
// with -DKDA_WAIT_POLL the waits also poll (mbarrier.test_wait) instead of
// letting the hardware suspend the thread, so they give up within the budget.
#ifndef KDA_WAIT_BUDGET
#define KDA_WAIT_BUDGET 4000000000LL
#endif

namespace kda {
namespace ptx {

constexpr long long kWaitBudget = KDA_WAIT_BUDGET;
// Budget of the waits on a kernel's exit path, after a wait gave up: the
// copies and tensor-core products it issued must land before the CTA's
// shared and tensor memory are released. Not lowered by KDA_WAIT_BUDGET.
constexpr long long kDrainBudget = 4000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
#ifdef KDA_WAIT_POLL
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
#else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
#endif
    return ok != 0;
}

// Waits for the phase with the given parity to complete. Returns false if
// `budget` clock cycles pass first.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long budget) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > budget) return false;
    }
    return true;
}

// L2 policy: lines are evicted first (data streamed once per step).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Bulk copy global -> this CTA's shared memory, completing `bytes` of
// transaction count on `bar`. Addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Bulk async-groups of the issuing thread (tensor stores are tracked by them).
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed bulk group of this thread has finished reading
// its shared-memory source (the buffer may then be overwritten).
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Tiled tensor copies (TMA) through a tensor map made on the host with
// cuTensorMapEncodeTiled and passed as a __grid_constant__ kernel parameter
// (`tmap` is its address). Coordinates are element indices, innermost first;
// the innermost one times the element size must be a multiple of 16 bytes,
// and none may be negative for a store. A load always transfers the whole box
// (parts outside the tensor read as zero) and completes the box's bytes on
// `bar`; a store writes only the parts inside the tensor and is tracked by the
// issuing thread's bulk async-groups (bulk_commit / bulk_wait_*).
__device__ __forceinline__ void tma_load_4d(void *dst, const void *tmap, uint64_t *bar, int x, int y,
                                            int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}
__device__ __forceinline__ void tma_load_5d(void *dst, const void *tmap, uint64_t *bar, int x, int y,
                                            int z, int w, int u) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w),
        "r"(u)
        : "memory");
}
__device__ __forceinline__ void tma_store_4d(const void *tmap, const void *src, int x, int y, int z,
                                             int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

// Prefetch [src, src + bytes) into L2 (no shared memory involved).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their memory is visible (no-op without a dependency).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Programmatic dependent launch: allow the next kernel in the stream to start
// launching its CTAs (they still wait in grid_dependency_wait()).
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier over `nthreads` threads (multiple of 32) using hardware barrier `id`.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier over `nthreads` threads (multiple of 32) on hardware barrier `id`
// that also reduces a predicate: every thread gets true only if every
// participating thread passed true. A kernel uses it where a bounded wait
// may have given up in some threads: all of them leave together.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Signals arrival at hardware barrier `id` without waiting (the producer side
// of a named barrier whose consumer calls named_bar_sync with the same count).
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace ptx
}  // namespace kda
