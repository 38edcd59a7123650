// Launches the mHC post kernels with post given (PlainCoeffs), for both
// storage types, and owns the bounded-wait flag of the bulk-copy kernels.
#include <cudaTypedefs.h>

#include "mhc_launch_post.cuh"

namespace mhc {

namespace {

// Set to 1 when a bounded wait runs out (see mhc_bulk.cuh); one per device.
__device__ unsigned int g_wait_timeouts;

std::atomic<unsigned int*> g_flag_ptr[kMaxDevices];

}  // namespace

cudaError_t wait_flag_ptr(unsigned int** p) {
    const int dev = current_device();
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

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library does not link the driver library itself); resolved once.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::atomic<void*> fn{nullptr};
    void* p = fn.load(std::memory_order_acquire);
    if (p == nullptr) {
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(p, std::memory_order_release);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
}

cudaError_t encode_rows_map(CUtensorMap* map, const void* base, uint64_t H, uint32_t W, uint32_t rows, uint64_t T) {
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr || W == 0 || H % W != 0) return cudaErrorInvalidValue;
    const cuuint64_t dims[4] = {W, H / W, rows, T};
    const cuuint64_t strides[3] = {uint64_t(W) * 2, H * 2, uint64_t(rows) * H * 2};   // bytes, dimensions 1..3
    const cuuint32_t box[4] = {W, uint32_t(8 * kLanes) / W, rows, 1};
    const cuuint32_t step[4] = {1, 1, 1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(base), dims, strides, box,
                              step, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
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
