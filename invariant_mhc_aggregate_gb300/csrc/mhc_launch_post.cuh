// Launch shapes of the mHC post kernels (mhc_post.cuh), templated on the
// post coefficient source; instantiated by mhc_launch_post.cu (post given)
// and mhc_launch_post_sigmoid.cu (post from the mix).
#pragma once

#include <atomic>

#include "mhc_launch.cuh"

namespace mhc {

// A tensor map over T tokens of `rows` rows of H 2-byte values (base 16-byte
// aligned) seen as groups of W values (W divides H): boxes of W values x
// 2048 / W groups x `rows` rows x 1 token, i.e. 2048 consecutive values of
// each row, elements past the row's end reading as zero (defined in
// mhc_launch_post.cu; cudaErrorInvalidValue if the driver refuses it).
cudaError_t encode_rows_map(CUtensorMap* map, const void* base, uint64_t H, uint32_t W, uint32_t rows, uint64_t T);

#ifndef MHC_SPLIT_MAX_BOX_ROW
#define MHC_SPLIT_MAX_BOX_ROW 256
#endif

// The widest box row (values) that divides H: the copy engine moves a box
// row by row, so wider rows mean fewer of them for the same bytes.
inline uint32_t split_box_row(uint64_t H) {
    uint32_t W = MHC_SPLIT_MAX_BOX_ROW;
    while (W > 8 && H % W != 0) W /= 2;
    return W;
}

namespace post_launch {

// Vector indices are 32-bit: calls of 2^31 vectors or more run as several
// launches over consecutive token ranges (tokens are independent).
template <int N, int DT, int NW, int U, int MIN_BLOCKS, class Coeffs>
cudaError_t fwd_vec(const PostFwdCall& c, const Coeffs& k) {
    const uint64_t V = c.H / (2 * NW);
    const uint64_t max_tokens = 0x7FFFFFFFull / V;
    for (uint64_t t0 = 0; t0 < c.T; t0 += max_tokens) {
        const uint64_t nt = (c.T - t0 < max_tokens) ? c.T - t0 : max_tokens;
        const uint32_t n_vec = uint32_t(nt * V);
        const auto* x = static_cast<const Words<NW>*>(c.x) + uint64_t(N) * t0 * V;
        const auto* y = static_cast<const Words<NW>*>(c.y) + t0 * V;
        auto* o = static_cast<Words<NW>*>(c.out) + uint64_t(N) * t0 * V;
        const cudaError_t e =
            launch(post_fwd_vec_kernel<N, DT, NW, U, MIN_BLOCKS, Coeffs>, grid_for(n_vec, kPostBlock * U, ~0u),
                   kPostBlock, c.stream, x, y, k.shifted(uint64_t(N) * t0), c.res + uint64_t(N) * N * t0, o,
                   n_vec, uint32_t(V), make_fastdiv_u32(uint32_t(V)));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Launch shapes (measured at T = 4096, H = 7168): 16-byte vectors, one per
// thread, with the register budget of 4 blocks per SM (2 at n = 8, whose
// inputs alone take 36 registers: used for rows of fewer than 64 vectors,
// the split forward takes the longer ones); 32-byte vectors, more vectors
// per thread or fewer blocks per SM were slower.
// Split forward (n = 8, rows of at least 64 vectors): 64 positions per
// block, two threads each.
template <int N, int DT, int MIN_BLOCKS, class Coeffs>
cudaError_t fwd_split(const PostFwdCall& c, const Coeffs& k) {
    const uint64_t V = c.H / 8;
    const uint64_t max_tokens = 0x7FFFFFFFull / V;
    for (uint64_t t0 = 0; t0 < c.T; t0 += max_tokens) {
        const uint64_t nt = (c.T - t0 < max_tokens) ? c.T - t0 : max_tokens;
        const uint32_t n_vec = uint32_t(nt * V);
        const auto* x = static_cast<const Words<4>*>(c.x) + uint64_t(N) * t0 * V;
        const auto* y = static_cast<const Words<4>*>(c.y) + t0 * V;
        auto* o = static_cast<Words<4>*>(c.out) + uint64_t(N) * t0 * V;
        const cudaError_t e =
            launch(post_fwd_split_kernel<N, DT, MIN_BLOCKS, Coeffs>, grid_for(n_vec, kSplitFwdVecs, ~0u), kSplitFwdBlock,
                   c.stream, x, y, k.shifted(uint64_t(N) * t0), c.res + uint64_t(N) * N * t0, o, n_vec, uint32_t(V),
                   make_fastdiv_u32(uint32_t(V)));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int N, int DT, class Coeffs>
cudaError_t fwd_n(const PostFwdCall& c, const Coeffs& k) {
    if constexpr (N >= 8) {
        if (c.path == kPathVec16 && c.H / 8 >= uint64_t(kSplitFwdVecs)) return fwd_split<N, DT, kSplitFwdMinBlocks>(c, k);
    }
    if (c.path == kPathVec16) return fwd_vec<N, DT, 4, 1, (N >= 8 ? 2 : 4)>(c, k);
    return launch2d(post_fwd_element_kernel<N, DT, Coeffs>, narrow_grid(c.H, c.T), kNarrowBlock, c.stream,
                    static_cast<const uint16_t*>(c.x), static_cast<const uint16_t*>(c.y), k, c.res,
                    static_cast<uint16_t*>(c.out), c.T, c.H);
}

// Bulk-copy backward: a persistent grid of MIN_BLOCKS blocks per SM, each
// with a STAGES-deep ring of (2n + 1) x 4 KB stages.  Short rows (NARROW) get
// blocks of only the consumer warps that hold chunks, stages of that width,
// and proportionally more blocks per SM.
template <int N, int DT, int STAGES, int MIN_BLOCKS, class Coeffs, bool NARROW>
cudaError_t bwd_bulk_launch(const PostBwdCall& c, const Coeffs& k, uint32_t consumers) {
    static std::atomic<uint64_t> smem_done{0};
    constexpr uint32_t kMaxSmem = STAGES * post_bulk_stage_bytes(N);
    auto* kernel = post_bwd_bulk_kernel<N, DT, STAGES, MIN_BLOCKS, Coeffs, NARROW>;
    cudaError_t e = allow_smem(kernel, kMaxSmem, smem_done);
    if (e != cudaSuccess) return e;
    unsigned int* flag = nullptr;
    if ((e = wait_flag_ptr(&flag)) != cudaSuccess) return e;
    const uint32_t smem = STAGES * post_bulk_stage_bytes(N, consumers);
    const uint32_t per_sm = MIN_BLOCKS * (uint32_t(kLanes) / consumers);
    const uint32_t blocks = grid_for(c.T, 1, uint64_t(c.num_sms) * per_sm);
    return launch_smem(kernel, blocks, post_bulk_threads<Coeffs>(int(consumers)), smem, c.stream,
                       static_cast<const Words<4>*>(c.g), static_cast<const Words<4>*>(c.x),
                       static_cast<const Words<4>*>(c.y), k, c.res, static_cast<Words<4>*>(c.grad_x),
                       static_cast<Words<4>*>(c.grad_y), c.grad_res, c.T, uint32_t(c.H / 8), flag);
}

// Narrow blocks from rows of at most 128 chunks on, where they let more
// blocks share an SM (measured at n = 4 and about 2^25 values a call:
// H = 512 507 -> 266 us, H = 1024 274 -> 193 us; at H = 1536, 192 consumers
// gained nothing).
template <int N, int DT, int STAGES, int MIN_BLOCKS, class Coeffs>
cudaError_t bwd_bulk(const PostBwdCall& c, const Coeffs& k) {
    const uint64_t V = c.H / 8;
    if (V > uint64_t(kLanes / 2)) return bwd_bulk_launch<N, DT, STAGES, MIN_BLOCKS, Coeffs, false>(c, k, kLanes);
    return bwd_bulk_launch<N, DT, STAGES, MIN_BLOCKS, Coeffs, true>(c, k, uint32_t((V + 31) / 32 * 32));
}

// Split bulk-copy backward (n = 8): one block of 512 consumer threads per SM
// (no producer warp: the warp that frees a stage last refills it), a
// STAGES-deep ring of (2n + 1) x 4 KB stages, each filled by three tiled
// copies through tensor maps of g, x and y encoded for the call.  Tensor
// coordinates are 32-bit signed, so calls of 2^31 tokens or more run as
// several launches over consecutive token ranges (tokens are independent).
template <int N, int DT, int STAGES, class Coeffs>
cudaError_t bwd_split(const PostBwdCall& c, const Coeffs& k) {
    static std::atomic<uint64_t> smem_done{0};
    constexpr uint32_t kSmem = STAGES * post_bulk_stage_bytes(N) + 128;   // + alignment slack
    auto* kernel = post_bwd_split_kernel<N, DT, STAGES, Coeffs>;
    cudaError_t e = allow_smem(kernel, kSmem, smem_done);
    if (e != cudaSuccess) return e;
    unsigned int* flag = nullptr;
    if ((e = wait_flag_ptr(&flag)) != cudaSuccess) return e;
    const uint64_t V = c.H / 8;
    const uint32_t W = split_box_row(c.H);
    constexpr uint64_t kMaxTokens = 0x7FFFFFFFull;
    for (uint64_t t0 = 0; t0 < c.T; t0 += kMaxTokens) {
        const uint64_t nt = (c.T - t0 < kMaxTokens) ? c.T - t0 : kMaxTokens;
        CUtensorMap mg, mx, my;
        if ((e = encode_rows_map(&mg, static_cast<const uint16_t*>(c.g) + uint64_t(N) * t0 * c.H, c.H, W, N, nt)) !=
                cudaSuccess ||
            (e = encode_rows_map(&mx, static_cast<const uint16_t*>(c.x) + uint64_t(N) * t0 * c.H, c.H, W, N, nt)) !=
                cudaSuccess ||
            (e = encode_rows_map(&my, static_cast<const uint16_t*>(c.y) + t0 * c.H, c.H, W, 1, nt)) != cudaSuccess)
            return e;
        const uint32_t blocks = grid_for(nt, 1, uint64_t(c.num_sms));
        e = launch_smem(kernel, blocks, kSplitConsumers, kSmem, c.stream, mg, mx, my, k.shifted(uint64_t(N) * t0),
                        c.res + uint64_t(N) * N * t0, static_cast<Words<4>*>(c.grad_x) + uint64_t(N) * t0 * V,
                        static_cast<Words<4>*>(c.grad_y) + t0 * V, c.grad_res + uint64_t(N) * N * t0, nt, uint32_t(V),
                        W, flag);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int N, int DT, class Coeffs>
cudaError_t bwd_n(const PostBwdCall& c, const Coeffs& k) {
    // 16-byte path: the bulk-copy kernel (2 blocks per SM, a 3-stage ring) up
    // to n = 4; at n = 8 the split kernel (two threads per lane, 1 block per
    // SM, a 3-stage ring of tiled copies: T = 4096, H = 7168 401.5 us with 2
    // stages, 366.1 us with 3)
    if (c.path == kPathVec16) {
        if constexpr (N >= 8) return bwd_split<N, DT, 3>(c, k);
        else return bwd_bulk<N, DT, 3, 2>(c, k);
    }
    const uint32_t blocks = grid_for(c.T, 1, uint64_t(c.num_sms) * 256);
    return launch(post_bwd_element_kernel<N, DT, Coeffs>, blocks, kLanes, c.stream,
                  static_cast<const uint16_t*>(c.g), static_cast<const uint16_t*>(c.x),
                  static_cast<const uint16_t*>(c.y), k, c.res, static_cast<uint16_t*>(c.grad_x),
                  static_cast<uint16_t*>(c.grad_y), c.grad_res, c.T, c.H);
}

template <class Coeffs>
cudaError_t fwd(const PostFwdCall& c, const Coeffs& k, int dtype) {
    const bool bf = dtype == kBF16;
    switch (c.n) {
        case 1: return bf ? fwd_n<1, kBF16>(c, k) : fwd_n<1, kF16>(c, k);
        case 2: return bf ? fwd_n<2, kBF16>(c, k) : fwd_n<2, kF16>(c, k);
        case 4: return bf ? fwd_n<4, kBF16>(c, k) : fwd_n<4, kF16>(c, k);
        default: return bf ? fwd_n<8, kBF16>(c, k) : fwd_n<8, kF16>(c, k);
    }
}

template <class Coeffs>
cudaError_t bwd(const PostBwdCall& c, const Coeffs& k, int dtype) {
    const bool bf = dtype == kBF16;
    switch (c.n) {
        case 1: return bf ? bwd_n<1, kBF16>(c, k) : bwd_n<1, kF16>(c, k);
        case 2: return bf ? bwd_n<2, kBF16>(c, k) : bwd_n<2, kF16>(c, k);
        case 4: return bf ? bwd_n<4, kBF16>(c, k) : bwd_n<4, kF16>(c, k);
        default: return bf ? bwd_n<8, kBF16>(c, k) : bwd_n<8, kF16>(c, k);
    }
}

}  // namespace post_launch
}  // namespace mhc
