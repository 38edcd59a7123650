// Host-side launch layer: picks the launch shape for a validated call and
// launches the kernels of mhc_device.cuh with programmatic stream
// serialization.  Launch shapes never change results.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "mhc_device.cuh"

namespace mhc {

constexpr int kMaxDevices = 64;

inline int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
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

// The device address of the flag that the bulk-copy kernels set when a
// bounded wait runs out (defined in mhc_launch_post.cu), for the current device.
cudaError_t wait_flag_ptr(unsigned int** p);

// Kernel path codes (the values of mhc_path_t).
constexpr int kPathVec16 = 0;
constexpr int kPathPair = 1;
constexpr int kPathElement = 2;
constexpr int kPathVec32 = 3;
constexpr int kPathShift16 = 4;

// The per-token coefficients (pre, or the mix they are computed from) and the
// per-token coefficient gradients travel in a PlainCoeffs / SigmoidCoeffs
// value (mhc_coeffs.cuh) next to these.
struct FwdCall {
    const void* residual;
    void* out;
    uint64_t T, H;
    int n;            // streams: 1, 2, 4 or 8
    int path;         // kPath*
    int num_sms;
    cudaStream_t stream;
};

struct BwdCall {
    const void* g;
    const void* residual;
    void* gres;
    uint64_t T, H;
    int n;
    int path;
    int num_sms;
    cudaStream_t stream;
};

// One translation unit per storage type and coefficient source.
cudaError_t fwd_bf16(const FwdCall& c, const PlainCoeffs& k);
cudaError_t fwd_f16(const FwdCall& c, const PlainCoeffs& k);
cudaError_t bwd_bf16(const BwdCall& c, const PlainCoeffs& k);
cudaError_t bwd_f16(const BwdCall& c, const PlainCoeffs& k);
cudaError_t fwd_bf16(const FwdCall& c, const SigmoidCoeffs& k);
cudaError_t fwd_f16(const FwdCall& c, const SigmoidCoeffs& k);
cudaError_t bwd_bf16(const BwdCall& c, const SigmoidCoeffs& k);
cudaError_t bwd_f16(const BwdCall& c, const SigmoidCoeffs& k);

// mHC post (mhc_post.cuh, launched from mhc_launch_post.cu and
// mhc_launch_post_sigmoid.cu); the post coefficients (given, or from the mix)
// and their gradient travel in the PlainCoeffs / SigmoidCoeffs value.
struct PostFwdCall {
    const void* x;
    const void* y;
    const float* res;
    void* out;
    uint64_t T, H;
    int n;
    int path;
    int num_sms;
    cudaStream_t stream;
};

struct PostBwdCall {
    const void* g;
    const void* x;
    const void* y;
    const float* res;
    void* grad_x;
    void* grad_y;
    float* grad_res;
    uint64_t T, H;
    int n;
    int path;
    int num_sms;
    cudaStream_t stream;
};

cudaError_t post_fwd(const PostFwdCall& c, const PlainCoeffs& k, int dtype);
cudaError_t post_bwd(const PostBwdCall& c, const PlainCoeffs& k, int dtype);
cudaError_t post_fwd(const PostFwdCall& c, const SigmoidCoeffs& k, int dtype);
cudaError_t post_bwd(const PostBwdCall& c, const SigmoidCoeffs& k, int dtype);
// 1 if a bounded wait of the bulk-copy kernels ran out on the current device
// since the last call, else 0 (clears the record; synchronizes the device);
// -1 on a CUDA error.
int64_t take_wait_timeouts();

// The coefficient kernels of their own (mhc_launch_coeffs.cu).
cudaError_t pre_sigmoid(const float* mix, const float* alpha, const float* b, float* pre,
                        uint64_t T, int n, int num_sms, cudaStream_t stream);
cudaError_t sigmoid_param_grad(const float* grad_z, const float* mix, float* grad_b,
                               float* grad_alpha, uint64_t T, int n, bool vec, cudaStream_t stream);

// Launch with programmatic stream serialization (see pdl_enter) and
// `smem` bytes of dynamic shared memory.
template <typename... Params, typename... Args>
cudaError_t launch_smem(void (*kernel)(Params...), uint32_t grid, uint32_t block, uint32_t smem,
                        cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

template <typename... Params, typename... Args>
cudaError_t launch(void (*kernel)(Params...), uint32_t grid, uint32_t block, cudaStream_t stream,
                   Args... args) {
    return launch_smem(kernel, grid, block, 0, stream, args...);
}

inline uint32_t grid_for(uint64_t items, uint32_t per_block, uint64_t cap) {
    uint64_t b = (items + per_block - 1) / per_block;
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return uint32_t(b);
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------

template <int N, int DT, int NW, int BLOCK, int UNROLL, class Coeffs>
cudaError_t launch_fwd_vec(const void* residual, const Coeffs& k, void* out, uint32_t n_vec,
                           uint32_t V, cudaStream_t stream) {
    const uint32_t per_block = uint32_t(BLOCK * UNROLL);
    const uint32_t blocks = uint32_t((uint64_t(n_vec) + per_block - 1) / per_block);
    return launch(agg_fwd_vec_kernel<N, DT, NW, BLOCK, UNROLL, Coeffs>, blocks, BLOCK, stream,
                  static_cast<const Words<NW>*>(residual), k, static_cast<Words<NW>*>(out), n_vec,
                  V, make_fastdiv_u32(V));
}

// Large calls: 256 threads x 1 vector (measured against 64 bytes of
// residual loads per stream pair, i.e. 2 vectors a thread at n = 4 with
// 32-byte vectors: the same cold, and 0.8% / 3.3% faster steady at T = 4096 /
// 1024, H = 7168); calls of at most 8 KiB of output per SM: 128 threads x 1
// vector, to spread a decode-sized call over more SMs.  Vector indices are 32-bit: a call with 2^31 vectors or
// more runs as several launches over consecutive token ranges (tokens are
// independent, so the bytes are the same as one launch).
template <int N, int DT, int NW, class Coeffs>
cudaError_t fwd_vec(const FwdCall& c, const Coeffs& coeffs) {
    const uint64_t V = c.H / (2 * NW);
    const uint64_t max_tokens = 0x7FFFFFFFull / V;
    const uint64_t small_limit = uint64_t(c.num_sms) * (8192 / (4 * NW));
    for (uint64_t t0 = 0; t0 < c.T; t0 += max_tokens) {
        const uint64_t nt = (c.T - t0 < max_tokens) ? c.T - t0 : max_tokens;
        const uint32_t n_vec = uint32_t(nt * V);
        const void* r = static_cast<const char*>(c.residual) + t0 * 2 * N * c.H;
        const Coeffs k = coeffs.shifted(N * t0);
        void* o = static_cast<char*>(c.out) + t0 * 2 * c.H;
        const cudaError_t e =
            n_vec <= small_limit
                ? launch_fwd_vec<N, DT, NW, 128, 1>(r, k, o, n_vec, uint32_t(V), c.stream)
                : launch_fwd_vec<N, DT, NW, 256, 1>(r, k, o, n_vec, uint32_t(V), c.stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Narrow forward paths: one block per (2048-unit row segment, token), with
// at most 65535 token rows of blocks (grid-stride over the rest).
inline dim3 narrow_grid(uint64_t units_per_row, uint64_t T) {
    const uint64_t segs = (units_per_row + kNarrowSeg - 1) / kNarrowSeg;
    return dim3(uint32_t(segs), uint32_t(T < 65535 ? T : 65535));
}

template <typename... Params, typename... Args>
cudaError_t launch2d(void (*kernel)(Params...), dim3 grid, uint32_t block, cudaStream_t stream,
                     Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// The realigned forward: compile-time window offsets (one kernel per H mod 8)
// for the pages' operation (n = 4, BF16, pre given), run-time offsets for
// the others.
template <int N, int DT, int U, class Coeffs>
cudaError_t fwd_shift_launch(dim3 grid, uint32_t block, const FwdCall& c, const uint16_t* r, const Coeffs& k,
                             uint16_t* o) {
    if constexpr (N == 4 && DT == kBF16 && !Coeffs::kBlockTable) {
        switch (c.H & 7u) {
            case 0: return launch2d(agg_fwd_shift_kernel<N, DT, U, 0, Coeffs>, grid, block, c.stream, r, k, o, c.T, c.H);
            case 1: return launch2d(agg_fwd_shift_kernel<N, DT, U, 1, Coeffs>, grid, block, c.stream, r, k, o, c.T, c.H);
            case 2: return launch2d(agg_fwd_shift_kernel<N, DT, U, 2, Coeffs>, grid, block, c.stream, r, k, o, c.T, c.H);
            case 3: return launch2d(agg_fwd_shift_kernel<N, DT, U, 3, Coeffs>, grid, block, c.stream, r, k, o, c.T, c.H);
            case 4: return launch2d(agg_fwd_shift_kernel<N, DT, U, 4, Coeffs>, grid, block, c.stream, r, k, o, c.T, c.H);
            case 5: return launch2d(agg_fwd_shift_kernel<N, DT, U, 5, Coeffs>, grid, block, c.stream, r, k, o, c.T, c.H);
            case 6: return launch2d(agg_fwd_shift_kernel<N, DT, U, 6, Coeffs>, grid, block, c.stream, r, k, o, c.T, c.H);
            default: return launch2d(agg_fwd_shift_kernel<N, DT, U, 7, Coeffs>, grid, block, c.stream, r, k, o, c.T, c.H);
        }
    } else {
        return launch2d(agg_fwd_shift_kernel<N, DT, U, -1, Coeffs>, grid, block, c.stream, r, k, o, c.T, c.H);
    }
}

template <int N, int DT, class Coeffs>
cudaError_t fwd_n(const FwdCall& c, const Coeffs& k) {
    switch (c.path) {
        case kPathVec32: return fwd_vec<N, DT, 8>(c, k);
        case kPathVec16: return fwd_vec<N, DT, 4>(c, k);
        case kPathShift16: {
            // a row's output vectors in nseg equal segments: up to 8 warps x 31 x 2
            // vectors each (U = 2), or, for rows of fewer than 496 vectors, one
            // segment of ceil(vectors / 31) warps (U = 1); blocks of 32 x warps threads
            const uint64_t vecs = shift_row_vectors(c.H);
            const uint32_t tokens = uint32_t(c.T < 65535 ? c.T : 65535);
            const auto* r = static_cast<const uint16_t*>(c.residual);
            auto* o = static_cast<uint16_t*>(c.out);
            constexpr uint64_t kRun2 = 2 * kShiftWarpVectors;
            if (vecs >= 8 * kRun2) {
                const uint64_t nseg = (vecs + 8 * kRun2 - 1) / (8 * kRun2);
                const uint64_t per_seg = (vecs + nseg - 1) / nseg;
                const uint32_t warps = uint32_t((per_seg + kRun2 - 1) / kRun2);
                return fwd_shift_launch<N, DT, 2>(dim3(uint32_t(nseg), tokens), 32 * warps, c, r, k, o);
            }
            const uint32_t warps = uint32_t((vecs + kShiftWarpVectors - 1) / kShiftWarpVectors);
            return fwd_shift_launch<N, DT, 1>(dim3(1, tokens), 32 * warps, c, r, k, o);
        }
        case kPathPair: {
            const uint64_t P = c.H / 2;
            return launch2d(agg_fwd_pair_kernel<N, DT, Coeffs>, narrow_grid(P, c.T), kNarrowBlock, c.stream,
                            static_cast<const uint32_t*>(c.residual), k, static_cast<uint32_t*>(c.out), c.T, P);
        }
        default:
            return launch2d(agg_fwd_element_kernel<N, DT, Coeffs>, narrow_grid(c.H, c.T), kNarrowBlock, c.stream,
                            static_cast<const uint16_t*>(c.residual), k, static_cast<uint16_t*>(c.out), c.T, c.H);
    }
}

template <int DT, class Coeffs>
cudaError_t fwd_dispatch(const FwdCall& c, const Coeffs& k) {
    switch (c.n) {
        case 1: return fwd_n<1, DT>(c, k);
        case 2: return fwd_n<2, DT>(c, k);
        case 4: return fwd_n<4, DT>(c, k);
        default: return fwd_n<8, DT>(c, k);
    }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------

// Rows of fewer vectors than a block has threads get blocks of only the
// warps that hold vectors (the fold adds +0 for the missing lane groups).
template <int N, int DT, int NW, int BATCH, int MIN_BLOCKS, class Coeffs>
cudaError_t launch_bwd_vec(const BwdCall& c, const Coeffs& k, uint32_t V) {
    constexpr uint32_t kThreads = kLanes / (NW / 4);
    const uint32_t threads = V < kThreads ? (V + 31) / 32 * 32 : kThreads;
    const uint32_t blocks = grid_for(c.T, 1, uint64_t(c.num_sms) * 256);
    return launch(agg_bwd_vec_kernel<N, DT, NW, BATCH, MIN_BLOCKS, Coeffs>, blocks, threads, c.stream,
                  static_cast<const Words<NW>*>(c.g), static_cast<const Words<NW>*>(c.residual), k,
                  static_cast<Words<NW>*>(c.gres), c.T, V);
}

// Backward vector launch shapes.  A block holds one token; its threads keep
// BATCH vectors each (g and N residual rows) in registers per pass, with the
// register budget sized for MIN_BLOCKS blocks per SM, so that each SM keeps
// roughly 160 KB of loads in flight.  For the pages' N = 4 with 32-byte
// vectors (128 threads) the batch follows the vectors per thread so that a
// row is covered in one pass: batch 1 / 2 / 4 with 6 / 3 / 2 blocks per SM
// for up to 1 / 2 / more vectors per thread.
template <int N, int DT, class Coeffs>
cudaError_t bwd_vec32(const BwdCall& c, const Coeffs& k) {
    const uint32_t V = uint32_t(c.H / 16);
    if constexpr (N == 4) {
        const uint32_t per_thread = (V + 127) / 128;
        if (per_thread <= 1) return launch_bwd_vec<N, DT, 8, 1, 6>(c, k, V);
        if (per_thread == 2) return launch_bwd_vec<N, DT, 8, 2, 3>(c, k, V);
        return launch_bwd_vec<N, DT, 8, 4, 2>(c, k, V);
    } else if constexpr (N == 1) {
        return launch_bwd_vec<N, DT, 8, 4, 4>(c, k, V);
    } else if constexpr (N == 2) {
        return launch_bwd_vec<N, DT, 8, 4, 3>(c, k, V);
    } else {
        return launch_bwd_vec<N, DT, 8, 2, 2>(c, k, V);
    }
}

template <int N, int DT, class Coeffs>
cudaError_t bwd_vec16(const BwdCall& c, const Coeffs& k) {
    const uint32_t V = uint32_t(c.H / 8);
    if constexpr (N == 1) {
        return launch_bwd_vec<N, DT, 4, 4, 3>(c, k, V);
    } else if constexpr (N == 8) {
        return launch_bwd_vec<N, DT, 4, 1, 2>(c, k, V);
    } else {
        return launch_bwd_vec<N, DT, 4, 2, 3>(c, k, V);
    }
}

// The realigned backward with bulk copies (mhc_shift_bulk.cuh): persistent
// blocks of 256 consumers and a producer warp, two per SM (96 registers a
// thread), each with a ring of 3 stages of 21.1 KB.  Measured at T = 4096,
// H = 7167: 3 stages 84.7 us, 2 stages 91 us, 4 stages 89 us; one block per
// SM with 4 or 6 stages (no register cap) 94-97 us.
template <int N, int DT, class Coeffs>
cudaError_t bwd_shift_bulk(const BwdCall& c, const Coeffs& k) {
    constexpr int S = 3, B = 2;
    constexpr uint32_t kSmem = S * shift_bulk_stage_bytes<N>();
    void (*kernel)(const uint16_t*, const uint16_t*, Coeffs, uint16_t*, uint64_t, uint64_t, unsigned int*);
    switch (c.H & 7u) {
        case 0: kernel = agg_bwd_shift_bulk_kernel<N, DT, 0, S, B, Coeffs>; break;
        case 1: kernel = agg_bwd_shift_bulk_kernel<N, DT, 1, S, B, Coeffs>; break;
        case 2: kernel = agg_bwd_shift_bulk_kernel<N, DT, 2, S, B, Coeffs>; break;
        case 3: kernel = agg_bwd_shift_bulk_kernel<N, DT, 3, S, B, Coeffs>; break;
        case 4: kernel = agg_bwd_shift_bulk_kernel<N, DT, 4, S, B, Coeffs>; break;
        case 5: kernel = agg_bwd_shift_bulk_kernel<N, DT, 5, S, B, Coeffs>; break;
        case 6: kernel = agg_bwd_shift_bulk_kernel<N, DT, 6, S, B, Coeffs>; break;
        default: kernel = agg_bwd_shift_bulk_kernel<N, DT, 7, S, B, Coeffs>; break;
    }
    static std::atomic<uint64_t> smem_done[8];
    cudaError_t e = allow_smem(kernel, kSmem, smem_done[c.H & 7u]);
    if (e != cudaSuccess) return e;
    unsigned int* flag = nullptr;
    if ((e = wait_flag_ptr(&flag)) != cudaSuccess) return e;
    const uint32_t blocks = uint32_t(c.T < uint64_t(c.num_sms) * B ? c.T : uint64_t(c.num_sms) * B);
    return launch_smem(kernel, blocks, uint32_t(kLanes + 32), kSmem, c.stream, static_cast<const uint16_t*>(c.g),
                       static_cast<const uint16_t*>(c.residual), k, static_cast<uint16_t*>(c.gres), c.T, c.H,
                       flag);
}

template <int N, int DT, class Coeffs>
cudaError_t bwd_n(const BwdCall& c, const Coeffs& k) {
    switch (c.path) {
        case kPathVec32: return bwd_vec32<N, DT>(c, k);
        case kPathVec16: return bwd_vec16<N, DT>(c, k);
        case kPathShift16: {
            // rows of fewer than 256 chunks: only the warps that hold chunks
            // (and at least 16n threads for the row-end values)
            const uint64_t chunks = (c.H + 7) / 8;
            uint32_t threads = uint32_t(chunks < uint64_t(kLanes) ? (chunks + 31) / 32 * 32 : kLanes);
            if (threads < uint32_t(16 * N)) threads = uint32_t(16 * N);
            if (threads < 32u) threads = 32u;
            const uint32_t blocks = grid_for(c.T, 1, uint64_t(c.num_sms) * 256);
            if constexpr (N == 4 && DT == kBF16 && !Coeffs::kBlockTable) {
                const bool same_offset =
                    ((reinterpret_cast<uintptr_t>(c.gres) - reinterpret_cast<uintptr_t>(c.residual)) & 15u) == 0;
                if (same_offset && chunks >= uint64_t(kLanes)) return bwd_shift_bulk<N, DT>(c, k);
            }
            if (threads < uint32_t(kLanes))
                return launch(agg_bwd_shift_kernel<N, DT, Coeffs, true>, blocks, threads, c.stream,
                              static_cast<const uint16_t*>(c.g), static_cast<const uint16_t*>(c.residual), k,
                              static_cast<uint16_t*>(c.gres), c.T, c.H);
            return launch(agg_bwd_shift_kernel<N, DT, Coeffs, false>, blocks, threads, c.stream,
                          static_cast<const uint16_t*>(c.g), static_cast<const uint16_t*>(c.residual), k,
                          static_cast<uint16_t*>(c.gres), c.T, c.H);
        }
        case kPathPair: {
            const uint32_t blocks = grid_for(c.T, 1, uint64_t(c.num_sms) * 256);
            return launch(agg_bwd_staged_kernel<N, DT, true, Coeffs>, blocks, kLanes, c.stream,
                          static_cast<const uint16_t*>(c.g), static_cast<const uint16_t*>(c.residual), k,
                          static_cast<uint16_t*>(c.gres), c.T, c.H);
        }
        default: {
            const uint32_t blocks = grid_for(c.T, 1, uint64_t(c.num_sms) * 256);
            return launch(agg_bwd_staged_kernel<N, DT, false, Coeffs>, blocks, kLanes, c.stream,
                          static_cast<const uint16_t*>(c.g), static_cast<const uint16_t*>(c.residual), k,
                          static_cast<uint16_t*>(c.gres), c.T, c.H);
        }
    }
}

template <int DT, class Coeffs>
cudaError_t bwd_dispatch(const BwdCall& c, const Coeffs& k) {
    switch (c.n) {
        case 1: return bwd_n<1, DT>(c, k);
        case 2: return bwd_n<2, DT>(c, k);
        case 4: return bwd_n<4, DT>(c, k);
        default: return bwd_n<8, DT>(c, k);
    }
}

}  // namespace mhc
