// Launches the mHC post kernels with post given (PlainCoeffs), for both
// storage types, and owns the bounded-wait flag of the bulk-copy kernels.
#include "mhc_launch_post.cuh"

namespace mhc {

namespace {

// Set to 1 when a bounded wait runs out (see mhc_bulk.cuh); one per device.
__device__ unsigned int g_wait_timeouts;

std::atomic<unsigned int*> g_flag_ptr[post_launch::kMaxDevices];

}  // namespace

cudaError_t wait_flag_ptr(unsigned int** p) {
    const int dev = post_launch::current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    unsigned int* q = g_flag_ptr[dev].load(std::memory_order_acquire);
    if (q == nullptr) {
        const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&q), g_wait_timeouts);
        if (e != cudaSuccess) return e;
        g_flag_ptr[dev].store(q, std::memory_order_release);
    }
    *p = q;
    return cudaSuccess;
}

cudaError_t post_fwd(const PostFwdCall& c, const PlainCoeffs& k, int dtype) {
    return post_launch::fwd(c, k, dtype);
}

cudaError_t post_bwd(const PostBwdCall& c, const PlainCoeffs& k, int dtype) {
    return post_launch::bwd(c, k, dtype);
}

int64_t take_wait_timeouts() {
    unsigned int n = 0;
    const unsigned int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(&n, g_wait_timeouts, sizeof(n)) != cudaSuccess) return -1;
    if (n != 0 && cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(zero)) != cudaSuccess) return -1;
    return int64_t(n);
}

}  // namespace mhc
