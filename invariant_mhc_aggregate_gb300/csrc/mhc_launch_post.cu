// Launches the mHC post kernels (mhc_post.cuh) for both storage types.
#include <atomic>

#include "mhc_launch.cuh"

namespace mhc {

namespace {

// Set to 1 when a bounded wait runs out (see mhc_bulk.cuh); one per device.
__device__ unsigned int g_wait_timeouts;

constexpr int kMaxDevices = 64;
std::atomic<unsigned int*> g_timeouts_ptr[kMaxDevices];

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

cudaError_t timeouts_ptr(unsigned int** p) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    unsigned int* q = g_timeouts_ptr[dev].load(std::memory_order_acquire);
    if (q == nullptr) {
        const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&q), g_wait_timeouts);
        if (e != cudaSuccess) return e;
        g_timeouts_ptr[dev].store(q, std::memory_order_release);
    }
    *p = q;
    return cudaSuccess;
}

// Raises a kernel's dynamic shared-memory limit, once per device (`done`
// holds one bit per device for that kernel).
template <class K>
cudaError_t allow_smem(K kernel, uint32_t bytes, std::atomic<uint64_t>& done) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Vector indices are 32-bit: calls of 2^31 vectors or more run as several
// launches over consecutive token ranges (tokens are independent).
template <int N, int DT, int NW, int U, int MIN_BLOCKS>
cudaError_t post_fwd_vec(const PostFwdCall& c) {
    const uint64_t V = c.H / (2 * NW);
    const uint64_t max_tokens = 0x7FFFFFFFull / V;
    for (uint64_t t0 = 0; t0 < c.T; t0 += max_tokens) {
        const uint64_t nt = (c.T - t0 < max_tokens) ? c.T - t0 : max_tokens;
        const uint32_t n_vec = uint32_t(nt * V);
        const auto* x = static_cast<const Words<NW>*>(c.x) + uint64_t(N) * t0 * V;
        const auto* y = static_cast<const Words<NW>*>(c.y) + t0 * V;
        auto* o = static_cast<Words<NW>*>(c.out) + uint64_t(N) * t0 * V;
        const cudaError_t e =
            launch(post_fwd_vec_kernel<N, DT, NW, U, MIN_BLOCKS>, grid_for(n_vec, kPostBlock * U, ~0u),
                   kPostBlock, c.stream, x, y, c.post + uint64_t(N) * t0, c.res + uint64_t(N) * N * t0, o,
                   n_vec, uint32_t(V), make_fastdiv_u32(uint32_t(V)));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Launch shapes (measured at T = 4096, H = 7168): 16-byte vectors, one per
// thread, with the register budget of 4 blocks per SM (2 at n = 8, whose
// inputs alone take 36 registers); 32-byte vectors, more vectors per thread
// or fewer blocks per SM were slower.
template <int N, int DT>
cudaError_t post_fwd_n(const PostFwdCall& c) {
    if (c.path == kPathVec16) return post_fwd_vec<N, DT, 4, 1, (N >= 8 ? 2 : 4)>(c);
    return launch2d(post_fwd_element_kernel<N, DT>, narrow_grid(c.H, c.T), kNarrowBlock, c.stream,
                    static_cast<const uint16_t*>(c.x), static_cast<const uint16_t*>(c.y), c.post, c.res,
                    static_cast<uint16_t*>(c.out), c.T, c.H);
}

template <int N, int DT, int NW, int BATCH, int MIN_BLOCKS, bool SMEM_COEF>
cudaError_t post_bwd_vec(const PostBwdCall& c) {
    const uint32_t blocks = grid_for(c.T, 1, uint64_t(c.num_sms) * 256);
    return launch(post_bwd_vec_kernel<N, DT, NW, BATCH, MIN_BLOCKS, SMEM_COEF>, blocks, kLanes / (NW / 4), c.stream,
                  static_cast<const Words<NW>*>(c.g), static_cast<const Words<NW>*>(c.x),
                  static_cast<const Words<NW>*>(c.y), c.post, c.res, static_cast<Words<NW>*>(c.grad_x),
                  static_cast<Words<NW>*>(c.grad_y), c.grad_post, c.grad_res, c.T, uint32_t(c.H / (2 * NW)));
}

// Bulk-copy backward: a persistent grid of MIN_BLOCKS blocks per SM, each
// with a STAGES-deep ring of (2n + 1) x 4 KB stages.
template <int N, int DT, int STAGES, int MIN_BLOCKS>
cudaError_t post_bwd_bulk(const PostBwdCall& c) {
    static std::atomic<uint64_t> smem_done{0};
    constexpr uint32_t smem = STAGES * post_bulk_stage_bytes(N);
    auto* kernel = post_bwd_bulk_kernel<N, DT, STAGES, MIN_BLOCKS>;
    cudaError_t e = allow_smem(kernel, smem, smem_done);
    if (e != cudaSuccess) return e;
    unsigned int* timeouts = nullptr;
    if ((e = timeouts_ptr(&timeouts)) != cudaSuccess) return e;
    const uint32_t blocks = grid_for(c.T, 1, uint64_t(c.num_sms) * MIN_BLOCKS);
    return launch_smem(kernel, blocks, kBulkThreads, smem, c.stream, static_cast<const Words<4>*>(c.g),
                       static_cast<const Words<4>*>(c.x), static_cast<const Words<4>*>(c.y), c.post, c.res,
                       static_cast<Words<4>*>(c.grad_x), static_cast<Words<4>*>(c.grad_y), c.grad_post,
                       c.grad_res, c.T, uint32_t(c.H / 8), timeouts);
}

template <int N, int DT>
cudaError_t post_bwd_n(const PostBwdCall& c) {
    // one 16-byte vector per thread and pass; 2 blocks per SM up to n = 4
    // (coefficients in registers), 1 at n = 8 (coefficients in shared memory)
    if (c.path == kPathVec16) {
        if constexpr (N >= 8) return post_bwd_vec<N, DT, 4, 1, 1, true>(c);
        else return post_bwd_bulk<N, DT, 3, 2>(c);
    }
    const uint32_t blocks = grid_for(c.T, 1, uint64_t(c.num_sms) * 256);
    return launch(post_bwd_element_kernel<N, DT>, blocks, kLanes, c.stream,
                  static_cast<const uint16_t*>(c.g), static_cast<const uint16_t*>(c.x),
                  static_cast<const uint16_t*>(c.y), c.post, c.res, static_cast<uint16_t*>(c.grad_x),
                  static_cast<uint16_t*>(c.grad_y), c.grad_post, c.grad_res, c.T, c.H);
}

template <int DT>
cudaError_t post_fwd_dt(const PostFwdCall& c) {
    switch (c.n) {
        case 1: return post_fwd_n<1, DT>(c);
        case 2: return post_fwd_n<2, DT>(c);
        case 4: return post_fwd_n<4, DT>(c);
        default: return post_fwd_n<8, DT>(c);
    }
}

template <int DT>
cudaError_t post_bwd_dt(const PostBwdCall& c) {
    switch (c.n) {
        case 1: return post_bwd_n<1, DT>(c);
        case 2: return post_bwd_n<2, DT>(c);
        case 4: return post_bwd_n<4, DT>(c);
        default: return post_bwd_n<8, DT>(c);
    }
}

}  // namespace

cudaError_t post_fwd(const PostFwdCall& c, int dtype) {
    return dtype == kBF16 ? post_fwd_dt<kBF16>(c) : post_fwd_dt<kF16>(c);
}

cudaError_t post_bwd(const PostBwdCall& c, int dtype) {
    return dtype == kBF16 ? post_bwd_dt<kBF16>(c) : post_bwd_dt<kF16>(c);
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
