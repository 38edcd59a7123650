// Launches the mHC post kernels (mhc_post.cuh) for both storage types.
#include "mhc_launch.cuh"

namespace mhc {

namespace {

// Vector indices are 32-bit: calls of 2^31 vectors or more run as several
// launches over consecutive token ranges (tokens are independent).
template <int N, int DT, int NW>
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
            launch(post_fwd_vec_kernel<N, DT, NW>, grid_for(n_vec, kPostBlock, ~0u), kPostBlock, c.stream,
                   x, y, c.post + uint64_t(N) * t0, c.res + uint64_t(N) * N * t0, o, n_vec, uint32_t(V),
                   make_fastdiv_u32(uint32_t(V)));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int N, int DT>
cudaError_t post_fwd_n(const PostFwdCall& c) {
    switch (c.path) {
        // n = 8 keeps 16-byte vectors on the 32-byte path: 8 x 32-byte
        // vectors and 72 coefficients do not fit the register file.
        case kPathVec32: return post_fwd_vec<N, DT, (N >= 8 ? 4 : 8)>(c);
        case kPathVec16: return post_fwd_vec<N, DT, 4>(c);
        default:
            return launch2d(post_fwd_element_kernel<N, DT>, narrow_grid(c.H, c.T), kNarrowBlock, c.stream,
                            static_cast<const uint16_t*>(c.x), static_cast<const uint16_t*>(c.y), c.post,
                            c.res, static_cast<uint16_t*>(c.out), c.T, c.H);
    }
}

template <int N, int DT>
cudaError_t post_bwd_n(const PostBwdCall& c) {
    const uint32_t blocks = grid_for(c.T, 1, uint64_t(c.num_sms) * 256);
    if (c.path == kPathVec16) {
        return launch(post_bwd_vec_kernel<N, DT>, blocks, kLanes, c.stream,
                      static_cast<const Words<4>*>(c.g), static_cast<const Words<4>*>(c.x),
                      static_cast<const Words<4>*>(c.y), c.post, c.res, static_cast<Words<4>*>(c.grad_x),
                      static_cast<Words<4>*>(c.grad_y), c.grad_post, c.grad_res, c.T, uint32_t(c.H / 8));
    }
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

}  // namespace mhc
