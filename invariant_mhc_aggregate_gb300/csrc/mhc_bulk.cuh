// Bulk asynchronous copies (global -> shared, the copy engine of the SM) and
// the shared-memory transaction barriers that signal their completion, as
// inline PTX for sm_103a.
//
//  * bulk_copy_g2s: one contiguous copy of `bytes` (a multiple of 16, both
//    addresses 16-byte aligned) that counts its bytes on barrier `bar`;
//    tensor_copy_4d: one box of a tensor map (several rows at once).
//  * A stage barrier ("full") is armed by its single producer thread with the
//    number of bytes the stage's copies deliver (arrive_expect_tx); its phase
//    completes once every byte has landed.  A release barrier ("empty") counts
//    one arrival per consumer warp.
//  * Every wait is bounded: mbar_wait gives up after kWaitLimitNs of the
//    global nanosecond timer (or 2^26 polls, whichever comes first) and
//    returns false, so that a kernel whose copies never land ends with an
//    error flag set instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mhc {

constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s: legitimate waits last microseconds

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" : : "r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the copy engine (and the rest of
// the block, after a barrier).
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" : : "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :
                 : "r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t"
        ".reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase of `bar` with the given parity to complete; false if it
// did not within the limit.
static __device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t round = 0; round < (1u << 20); ++round) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
    return false;
}

// mbar_wait with its first poll inline: where the phase has almost always
// completed already, no call is made.
__device__ __forceinline__ bool mbar_wait_fast(uint64_t* bar, uint32_t parity) {
    return mbar_try_wait(bar, parity) || mbar_wait(bar, parity);
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :
        : "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// A tiled copy global -> shared of the box at element coordinates {c0, c1,
// c2, c3} of a 4-D tensor map (a __grid_constant__ kernel parameter),
// counting its bytes on barrier `bar`: the whole box, whose elements past
// the tensor's end read as zero.  c0 (the innermost coordinate) stays a
// multiple of 16 bytes' worth of elements; dst is 128-byte aligned.
__device__ __forceinline__ void tensor_copy_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                               uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];"
        :
        : "r"(smem_addr(dst)), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
        : "memory");
}

// A 4-byte asynchronous copy global -> shared (any 4-byte aligned
// addresses); the issuing thread commits its copies as a group and later
// waits for them (cp_async_wait_all) before a barrier that publishes them.
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" : : "r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Orders this thread's earlier shared-memory accesses (generic proxy) before
// its later bulk copies into shared memory (async proxy).
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The counter of warps that have released a stage: returns the count before
// this arrival and wraps to 0 after `last` (atom.inc), with acquire-release
// ordering at block scope: the warp's earlier shared-memory reads happen
// before it, and the arrival that sees `last` sees every earlier one's.
__device__ __forceinline__ uint32_t release_count(uint32_t* counter, uint32_t last) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.inc.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "r"(smem_addr(counter)), "r"(last)
                 : "memory");
    return old;
}

// Barrier over the first `threads` threads of the block (named barrier `id`,
// 1..15; id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" : : "r"(id), "r"(threads) : "memory");
}

}  // namespace mhc
