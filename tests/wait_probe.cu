// Test support: runs the bounded shared-memory barrier wait of mhc_bulk.cuh
// on a barrier that completes (one arrival) or never completes (nothing
// arrives), and reports the result and the time the wait took.
#include <stdint.h>

#include "mhc_bulk.cuh"

__global__ void wait_probe_kernel(int arrive, unsigned int* result, unsigned long long* elapsed_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mhc::mbar_init(&bar, 1);
        mhc::mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (arrive) mhc::mbar_arrive(&bar);
        const uint64_t t0 = mhc::global_ns();
        const bool done = mhc::mbar_wait(&bar, 0);
        *elapsed_ns = mhc::global_ns() - t0;
        *result = done ? 1u : 0u;
    }
}

extern "C" __attribute__((visibility("default"))) int run_wait_probe(int arrive, void* result, void* elapsed_ns) {
    wait_probe_kernel<<<1, 32>>>(arrive, static_cast<unsigned int*>(result),
                                 static_cast<unsigned long long*>(elapsed_ns));
    if (cudaGetLastError() != cudaSuccess) return 1;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 2;
}
