// C ABI of the batch-invariant mHC pre "H Aggregate" library for GB300
// (sm_103a): argument validation, kernel-path choice and launch through the
// layer in mhc_launch.cuh.  The kernels are in mhc_device.cuh.
//
// Source: "Add batch-invariant h_aggregate kernel" (RL-Kernel pull request
// 366), Summary and Batch invariance; its reviewer comment for the backward.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "mhc_h_aggregate.h"
#include "mhc_launch.cuh"

namespace {

constexpr int kAbiVersion = 6;

thread_local int32_t g_last_cuda_error = 0;

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

inline Range range_of(const void* p, uint64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + uintptr_t(bytes)};
}

inline bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

inline bool streams_ok(int64_t n) { return n == 1 || n == 2 || n == 4 || n == 8; }

// Rows that no vector path can take use the realigned 16-byte path when they
// hold at least kShiftMinH values (the forward keeps the faster 4-byte pair
// path for even H with 4-byte-aligned buffers); shorter rows the 4- or
// 2-byte paths.
constexpr int64_t kShiftMinH = 64;
constexpr int64_t kShiftMaxH = int64_t(1) << 30;   // row positions are 32-bit there

inline bool dtype_ok(int32_t d) { return d == MHC_DTYPE_BF16 || d == MHC_DTYPE_F16; }

// Sizes are valid and the residual's byte count (2 * n * T * H) fits in int64.
inline bool sizes_ok(int64_t T, int64_t n, int64_t H) {
    if (T < 0 || H <= 0) return false;
    if (T == 0) return true;
    const int64_t lim = INT64_MAX / (2 * n);
    return H <= lim / T;
}

// SM count of the current device, used only to size grids (never the arithmetic).
int num_sms() {
    static std::atomic<int> cached{0};
    int n = cached.load(std::memory_order_relaxed);
    if (n == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            n = 152;
        }
        cached.store(n, std::memory_order_relaxed);
    }
    return n;
}

mhc_path_t fwd_path(const void* residual, const float* pre, const void* out, int64_t T, int64_t n,
                    int64_t H) {
    if (!streams_ok(n) || !sizes_ok(T, n, H) || T == 0) return MHC_PATH_NONE;
    if (!residual || !pre || !out) return MHC_PATH_NONE;
    if (!aligned(residual, 2) || !aligned(out, 2) || !aligned(pre, 4)) return MHC_PATH_NONE;
    const uint64_t res_bytes = uint64_t(T) * 2 * uint64_t(n) * uint64_t(H);
    const Range ro = range_of(out, uint64_t(T) * 2 * uint64_t(H));
    if (overlap(ro, range_of(residual, res_bytes)) ||
        overlap(ro, range_of(pre, uint64_t(T) * 4 * uint64_t(n))))
        return MHC_PATH_NONE;
    if (H % 16 == 0 && aligned(residual, 32) && aligned(out, 32)) return MHC_PATH_VEC32;
    if (H % 8 == 0 && aligned(residual, 16) && aligned(out, 16)) return MHC_PATH_VEC16;
    if (H % 2 == 0 && aligned(residual, 4) && aligned(out, 4)) return MHC_PATH_PAIR;
    if (H >= kShiftMinH && H < kShiftMaxH) return MHC_PATH_SHIFT16;
    return MHC_PATH_ELEMENT;
}

mhc_path_t bwd_path(const void* g, const void* residual, const float* pre, const void* gres,
                    const float* gpre, int64_t T, int64_t n, int64_t H) {
    if (!streams_ok(n) || !sizes_ok(T, n, H) || T == 0) return MHC_PATH_NONE;
    if (!g || !residual || !pre || !gres || !gpre) return MHC_PATH_NONE;
    if (!aligned(g, 2) || !aligned(residual, 2) || !aligned(gres, 2) || !aligned(pre, 4) ||
        !aligned(gpre, 4))
        return MHC_PATH_NONE;
    const uint64_t TH = uint64_t(T) * uint64_t(H);
    const Range rgr = range_of(gres, TH * 2 * uint64_t(n));
    const Range rgp = range_of(gpre, uint64_t(T) * 4 * uint64_t(n));
    const Range ins[3] = {range_of(g, TH * 2), range_of(residual, TH * 2 * uint64_t(n)),
                          range_of(pre, uint64_t(T) * 4 * uint64_t(n))};
    if (overlap(rgr, rgp)) return MHC_PATH_NONE;
    for (const Range& in : ins)
        if (overlap(rgr, in) || overlap(rgp, in)) return MHC_PATH_NONE;
    if (H % 16 == 0 && aligned(g, 32) && aligned(residual, 32) && aligned(gres, 32)) return MHC_PATH_VEC32;
    if (H % 8 == 0 && aligned(g, 16) && aligned(residual, 16) && aligned(gres, 16)) return MHC_PATH_VEC16;
    // the realigned backward is faster than the staged 4-byte one, so it also
    // takes even H
    if (H >= kShiftMinH && H < kShiftMaxH) return MHC_PATH_SHIFT16;
    if (H % 2 == 0 && aligned(g, 4) && aligned(residual, 4) && aligned(gres, 4)) return MHC_PATH_PAIR;
    return MHC_PATH_ELEMENT;
}

// The token's pre (n floats) can be read with float2 / float4 loads.
inline bool pre_vectorizable(const float* pre, int64_t n) {
    return aligned(pre, n >= 4 ? 16 : uintptr_t(4 * n));
}

mhc_status_t finish(cudaError_t launch_error) {
    cudaError_t e = launch_error;
    if (e == cudaSuccess) e = cudaGetLastError();
    g_last_cuda_error = int32_t(e);
    return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA;
}

mhc_status_t aggregate_fwd(const void* residual, const float* pre, void* out, int64_t T, int64_t n,
                           int64_t H, int32_t dtype, mhc_stream_t stream) {
    if (!dtype_ok(dtype)) return MHC_ERR_INVALID_ARG;
    if (!streams_ok(n)) return MHC_ERR_UNSUPPORTED;
    if (!sizes_ok(T, n, H)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    const mhc_path_t path = fwd_path(residual, pre, out, T, n, H);
    if (path == MHC_PATH_NONE) return MHC_ERR_INVALID_ARG;
    if ((path == MHC_PATH_VEC32 || path == MHC_PATH_VEC16) && uint64_t(H) / 8 > 0x7FFFFFFFull)
        return MHC_ERR_UNSUPPORTED;
    const mhc::FwdCall c{residual, out, uint64_t(T), uint64_t(H), int(n), int(path), num_sms(),
                         reinterpret_cast<cudaStream_t>(stream)};
    const mhc::PlainCoeffs k{pre, nullptr, pre_vectorizable(pre, n)};
    return finish(dtype == MHC_DTYPE_BF16 ? mhc::fwd_bf16(c, k) : mhc::fwd_f16(c, k));
}

mhc_status_t aggregate_bwd(const void* grad_out, const void* residual, const float* pre,
                           void* grad_residual, float* grad_pre, int64_t T, int64_t n, int64_t H,
                           int32_t dtype, mhc_stream_t stream) {
    if (!dtype_ok(dtype)) return MHC_ERR_INVALID_ARG;
    if (!streams_ok(n)) return MHC_ERR_UNSUPPORTED;
    if (!sizes_ok(T, n, H)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    const mhc_path_t path = bwd_path(grad_out, residual, pre, grad_residual, grad_pre, T, n, H);
    if (path == MHC_PATH_NONE) return MHC_ERR_INVALID_ARG;
    // vector indices within a row are 32-bit (with headroom for the per-pass stride)
    if ((path == MHC_PATH_VEC32 || path == MHC_PATH_VEC16) && uint64_t(H) / 8 > 0x7FFFFFFFull)
        return MHC_ERR_UNSUPPORTED;
    const mhc::BwdCall c{grad_out, residual, grad_residual, uint64_t(T), uint64_t(H), int(n),
                         int(path), num_sms(), reinterpret_cast<cudaStream_t>(stream)};
    const mhc::PlainCoeffs k{pre, grad_pre, pre_vectorizable(pre, n)};
    return finish(dtype == MHC_DTYPE_BF16 ? mhc::bwd_bf16(c, k) : mhc::bwd_f16(c, k));
}

// ---- the pre coefficients computed from the mix (sigmoid) ----------------

// alpha (one float) and b (n floats) are 4-byte aligned and overlap none of
// the outputs.
bool params_ok(const float* alpha, const float* b, int64_t n, const Range* outs, int n_outs) {
    if (!alpha || !b || !aligned(alpha, 4) || !aligned(b, 4)) return false;
    const Range ra = range_of(alpha, 4), rb = range_of(b, uint64_t(4) * uint64_t(n));
    for (int i = 0; i < n_outs; ++i)
        if (overlap(outs[i], ra) || overlap(outs[i], rb)) return false;
    return true;
}

mhc_status_t aggregate_sigmoid_fwd(const void* residual, const float* mix, const float* alpha,
                                   const float* b, void* out, int64_t T, int64_t n, int64_t H,
                                   int32_t dtype, mhc_stream_t stream) {
    if (!dtype_ok(dtype)) return MHC_ERR_INVALID_ARG;
    if (!streams_ok(n)) return MHC_ERR_UNSUPPORTED;
    if (!sizes_ok(T, n, H)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    const mhc_path_t path = fwd_path(residual, mix, out, T, n, H);
    if (path == MHC_PATH_NONE) return MHC_ERR_INVALID_ARG;
    const Range ro = range_of(out, uint64_t(T) * 2 * uint64_t(H));
    if (!params_ok(alpha, b, n, &ro, 1)) return MHC_ERR_INVALID_ARG;
    if ((path == MHC_PATH_VEC32 || path == MHC_PATH_VEC16) && uint64_t(H) / 8 > 0x7FFFFFFFull)
        return MHC_ERR_UNSUPPORTED;
    const mhc::FwdCall c{residual, out, uint64_t(T), uint64_t(H), int(n), int(path), num_sms(),
                         reinterpret_cast<cudaStream_t>(stream)};
    const mhc::SigmoidCoeffs k{mix, alpha, b, nullptr, nullptr, pre_vectorizable(mix, n)};
    return finish(dtype == MHC_DTYPE_BF16 ? mhc::fwd_bf16(c, k) : mhc::fwd_f16(c, k));
}

mhc_status_t aggregate_sigmoid_bwd(const void* grad_out, const void* residual, const float* mix,
                                   const float* alpha, const float* b, void* grad_residual,
                                   float* grad_z, float* grad_mix, int64_t T, int64_t n, int64_t H,
                                   int32_t dtype, mhc_stream_t stream) {
    if (!dtype_ok(dtype)) return MHC_ERR_INVALID_ARG;
    if (!streams_ok(n)) return MHC_ERR_UNSUPPORTED;
    if (!sizes_ok(T, n, H)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    // grad_z stands in for grad_pre in the path check (same shape and rules)
    const mhc_path_t path = bwd_path(grad_out, residual, mix, grad_residual, grad_z, T, n, H);
    if (path == MHC_PATH_NONE) return MHC_ERR_INVALID_ARG;
    if (!grad_mix || !aligned(grad_mix, 4)) return MHC_ERR_INVALID_ARG;
    const uint64_t TH = uint64_t(T) * uint64_t(H);
    const Range outs[3] = {range_of(grad_residual, TH * 2 * uint64_t(n)),
                           range_of(grad_z, uint64_t(T) * 4 * uint64_t(n)),
                           range_of(grad_mix, uint64_t(T) * 4 * uint64_t(n))};
    const Range ins[3] = {range_of(grad_out, TH * 2), range_of(residual, TH * 2 * uint64_t(n)),
                          range_of(mix, uint64_t(T) * 4 * uint64_t(n))};
    for (const Range& in : ins)
        if (overlap(outs[2], in)) return MHC_ERR_INVALID_ARG;
    if (overlap(outs[2], outs[0]) || overlap(outs[2], outs[1])) return MHC_ERR_INVALID_ARG;
    if (!params_ok(alpha, b, n, outs, 3)) return MHC_ERR_INVALID_ARG;
    if ((path == MHC_PATH_VEC32 || path == MHC_PATH_VEC16) && uint64_t(H) / 8 > 0x7FFFFFFFull)
        return MHC_ERR_UNSUPPORTED;
    const mhc::BwdCall c{grad_out, residual, grad_residual, uint64_t(T), uint64_t(H), int(n),
                         int(path), num_sms(), reinterpret_cast<cudaStream_t>(stream)};
    const mhc::SigmoidCoeffs k{mix, alpha, b, grad_z, grad_mix, pre_vectorizable(mix, n)};
    return finish(dtype == MHC_DTYPE_BF16 ? mhc::bwd_bf16(c, k) : mhc::bwd_f16(c, k));
}

mhc_status_t pre_sigmoid(const float* mix, const float* alpha, const float* b, float* pre,
                         int64_t T, int64_t n, mhc_stream_t stream) {
    if (!streams_ok(n)) return MHC_ERR_UNSUPPORTED;
    if (T < 0 || T > INT64_MAX / (4 * n)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    if (!mix || !pre || !aligned(mix, 4) || !aligned(pre, 4)) return MHC_ERR_INVALID_ARG;
    const Range rp = range_of(pre, uint64_t(T) * 4 * uint64_t(n));
    if (overlap(rp, range_of(mix, uint64_t(T) * 4 * uint64_t(n)))) return MHC_ERR_INVALID_ARG;
    if (!params_ok(alpha, b, n, &rp, 1)) return MHC_ERR_INVALID_ARG;
    return finish(mhc::pre_sigmoid(mix, alpha, b, pre, uint64_t(T), int(n), num_sms(),
                                   reinterpret_cast<cudaStream_t>(stream)));
}

mhc_status_t sigmoid_param_grad(const float* grad_z, const float* mix, float* grad_b,
                                float* grad_alpha, int64_t T, int64_t n, mhc_stream_t stream) {
    if (!streams_ok(n)) return MHC_ERR_UNSUPPORTED;
    if (T < 0 || T > INT64_MAX / (4 * n)) return MHC_ERR_INVALID_ARG;
    if (!grad_b || !grad_alpha || !aligned(grad_b, 4) || !aligned(grad_alpha, 4))
        return MHC_ERR_INVALID_ARG;
    if (T > 0 && (!grad_z || !mix || !aligned(grad_z, 4) || !aligned(mix, 4)))
        return MHC_ERR_INVALID_ARG;
    const Range rb = range_of(grad_b, uint64_t(4) * uint64_t(n)), ra = range_of(grad_alpha, 4);
    if (overlap(rb, ra)) return MHC_ERR_INVALID_ARG;
    if (T > 0) {
        const Range rz = range_of(grad_z, uint64_t(T) * 4 * uint64_t(n));
        const Range rm = range_of(mix, uint64_t(T) * 4 * uint64_t(n));
        if (overlap(rb, rz) || overlap(rb, rm) || overlap(ra, rz) || overlap(ra, rm))
            return MHC_ERR_INVALID_ARG;
    }
    const bool vec = T > 0 && pre_vectorizable(grad_z, n) && pre_vectorizable(mix, n);
    return finish(mhc::sigmoid_param_grad(grad_z, mix, grad_b, grad_alpha, uint64_t(T), int(n), vec,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

// ---- mHC post ---------------------------------------------------------------

// Disjointness of a set of output ranges from each other and from the inputs.
bool disjoint(const Range* outs, int n_outs, const Range* ins, int n_ins) {
    for (int a = 0; a < n_outs; ++a) {
        for (int b = a + 1; b < n_outs; ++b)
            if (overlap(outs[a], outs[b])) return false;
        for (int i = 0; i < n_ins; ++i)
            if (overlap(outs[a], ins[i])) return false;
    }
    return true;
}

mhc_path_t post_fwd_path(const void* x, const void* y, const float* post, const float* res,
                         const void* out, int64_t T, int64_t n, int64_t H) {
    if (!streams_ok(n) || !sizes_ok(T, n, H) || T == 0) return MHC_PATH_NONE;
    if (!x || !y || !post || !res || !out) return MHC_PATH_NONE;
    if (!aligned(x, 2) || !aligned(y, 2) || !aligned(out, 2) || !aligned(post, 4) || !aligned(res, 4))
        return MHC_PATH_NONE;
    const uint64_t TH = uint64_t(T) * uint64_t(H), nu = uint64_t(n);
    const Range outs[1] = {range_of(out, TH * 2 * nu)};
    const Range ins[4] = {range_of(x, TH * 2 * nu), range_of(y, TH * 2),
                          range_of(post, uint64_t(T) * 4 * nu), range_of(res, uint64_t(T) * 4 * nu * nu)};
    if (!disjoint(outs, 1, ins, 4)) return MHC_PATH_NONE;
    if (H % 8 == 0 && aligned(x, 16) && aligned(y, 16) && aligned(out, 16)) return MHC_PATH_VEC16;
    return MHC_PATH_ELEMENT;
}

mhc_path_t post_bwd_path(const void* g, const void* x, const void* y, const float* post,
                         const float* res, const void* grad_x, const void* grad_y,
                         const float* grad_post, const float* grad_res, int64_t T, int64_t n,
                         int64_t H) {
    if (!streams_ok(n) || !sizes_ok(T, n, H) || T == 0) return MHC_PATH_NONE;
    if (!g || !x || !y || !post || !res || !grad_x || !grad_y || !grad_post || !grad_res)
        return MHC_PATH_NONE;
    if (!aligned(g, 2) || !aligned(x, 2) || !aligned(y, 2) || !aligned(grad_x, 2) ||
        !aligned(grad_y, 2) || !aligned(post, 4) || !aligned(res, 4) || !aligned(grad_post, 4) ||
        !aligned(grad_res, 4))
        return MHC_PATH_NONE;
    const uint64_t TH = uint64_t(T) * uint64_t(H), nu = uint64_t(n);
    const Range outs[4] = {range_of(grad_x, TH * 2 * nu), range_of(grad_y, TH * 2),
                           range_of(grad_post, uint64_t(T) * 4 * nu),
                           range_of(grad_res, uint64_t(T) * 4 * nu * nu)};
    const Range ins[5] = {range_of(g, TH * 2 * nu), range_of(x, TH * 2 * nu), range_of(y, TH * 2),
                          range_of(post, uint64_t(T) * 4 * nu), range_of(res, uint64_t(T) * 4 * nu * nu)};
    if (!disjoint(outs, 4, ins, 5)) return MHC_PATH_NONE;
    if (H % 8 == 0 && aligned(g, 16) && aligned(x, 16) && aligned(y, 16) && aligned(grad_x, 16) &&
        aligned(grad_y, 16))
        return MHC_PATH_VEC16;
    return MHC_PATH_ELEMENT;
}

mhc_status_t post_fwd(const void* x, const void* y, const float* post, const float* res, void* out,
                      int64_t T, int64_t n, int64_t H, int32_t dtype, mhc_stream_t stream) {
    if (!dtype_ok(dtype)) return MHC_ERR_INVALID_ARG;
    if (!streams_ok(n)) return MHC_ERR_UNSUPPORTED;
    if (!sizes_ok(T, n, H)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    const mhc_path_t path = post_fwd_path(x, y, post, res, out, T, n, H);
    if (path == MHC_PATH_NONE) return MHC_ERR_INVALID_ARG;
    if (path == MHC_PATH_VEC16 && uint64_t(H) / 8 > 0x7FFFFFFFull) return MHC_ERR_UNSUPPORTED;
    const mhc::PostFwdCall c{x, y, res, out, uint64_t(T), uint64_t(H), int(n), int(path), num_sms(),
                             reinterpret_cast<cudaStream_t>(stream)};
    const mhc::PlainCoeffs k{post, nullptr, false};
    return finish(mhc::post_fwd(c, k, dtype == MHC_DTYPE_BF16 ? mhc::kBF16 : mhc::kF16));
}

mhc_status_t post_bwd(const void* g, const void* x, const void* y, const float* post, const float* res,
                      void* grad_x, void* grad_y, float* grad_post, float* grad_res, int64_t T,
                      int64_t n, int64_t H, int32_t dtype, mhc_stream_t stream) {
    if (!dtype_ok(dtype)) return MHC_ERR_INVALID_ARG;
    if (!streams_ok(n)) return MHC_ERR_UNSUPPORTED;
    if (!sizes_ok(T, n, H)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    const mhc_path_t path =
        post_bwd_path(g, x, y, post, res, grad_x, grad_y, grad_post, grad_res, T, n, H);
    if (path == MHC_PATH_NONE) return MHC_ERR_INVALID_ARG;
    if (path == MHC_PATH_VEC16 && uint64_t(H) / 8 > 0x7FFFFFFFull) return MHC_ERR_UNSUPPORTED;
    const mhc::PostBwdCall c{g, x, y, res, grad_x, grad_y, grad_res, uint64_t(T), uint64_t(H), int(n),
                             int(path), num_sms(), reinterpret_cast<cudaStream_t>(stream)};
    const mhc::PlainCoeffs k{post, grad_post, false};
    return finish(mhc::post_bwd(c, k, dtype == MHC_DTYPE_BF16 ? mhc::kBF16 : mhc::kF16));
}

// ---- mHC post with post = sigmoid(alpha * mix + b) --------------------------

mhc_status_t post_sigmoid_fwd(const void* x, const void* y, const float* mix, const float* alpha,
                              const float* b, const float* res, void* out, int64_t T, int64_t n, int64_t H,
                              int32_t dtype, mhc_stream_t stream) {
    if (!dtype_ok(dtype)) return MHC_ERR_INVALID_ARG;
    if (!streams_ok(n)) return MHC_ERR_UNSUPPORTED;
    if (!sizes_ok(T, n, H)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    // mix stands in for post in the path check (same shape and rules)
    const mhc_path_t path = post_fwd_path(x, y, mix, res, out, T, n, H);
    if (path == MHC_PATH_NONE) return MHC_ERR_INVALID_ARG;
    const Range ro = range_of(out, uint64_t(T) * 2 * uint64_t(n) * uint64_t(H));
    if (!params_ok(alpha, b, n, &ro, 1)) return MHC_ERR_INVALID_ARG;
    if (path == MHC_PATH_VEC16 && uint64_t(H) / 8 > 0x7FFFFFFFull) return MHC_ERR_UNSUPPORTED;
    const mhc::PostFwdCall c{x, y, res, out, uint64_t(T), uint64_t(H), int(n), int(path), num_sms(),
                             reinterpret_cast<cudaStream_t>(stream)};
    const mhc::SigmoidCoeffs k{mix, alpha, b, nullptr, nullptr, false};
    return finish(mhc::post_fwd(c, k, dtype == MHC_DTYPE_BF16 ? mhc::kBF16 : mhc::kF16));
}

mhc_status_t post_sigmoid_bwd(const void* g, const void* x, const void* y, const float* mix,
                              const float* alpha, const float* b, const float* res, void* grad_x,
                              void* grad_y, float* grad_z, float* grad_mix, float* grad_res, int64_t T,
                              int64_t n, int64_t H, int32_t dtype, mhc_stream_t stream) {
    if (!dtype_ok(dtype)) return MHC_ERR_INVALID_ARG;
    if (!streams_ok(n)) return MHC_ERR_UNSUPPORTED;
    if (!sizes_ok(T, n, H)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    // mix and grad_z stand in for post and grad_post in the path check
    const mhc_path_t path = post_bwd_path(g, x, y, mix, res, grad_x, grad_y, grad_z, grad_res, T, n, H);
    if (path == MHC_PATH_NONE) return MHC_ERR_INVALID_ARG;
    if (!grad_mix || !aligned(grad_mix, 4)) return MHC_ERR_INVALID_ARG;
    const uint64_t TH = uint64_t(T) * uint64_t(H), nu = uint64_t(n);
    const Range outs[5] = {range_of(grad_x, TH * 2 * nu), range_of(grad_y, TH * 2),
                           range_of(grad_z, uint64_t(T) * 4 * nu), range_of(grad_res, uint64_t(T) * 4 * nu * nu),
                           range_of(grad_mix, uint64_t(T) * 4 * nu)};
    const Range ins[5] = {range_of(g, TH * 2 * nu), range_of(x, TH * 2 * nu), range_of(y, TH * 2),
                          range_of(mix, uint64_t(T) * 4 * nu), range_of(res, uint64_t(T) * 4 * nu * nu)};
    if (!disjoint(outs, 5, ins, 5)) return MHC_ERR_INVALID_ARG;
    if (!params_ok(alpha, b, n, outs, 5)) return MHC_ERR_INVALID_ARG;
    if (path == MHC_PATH_VEC16 && uint64_t(H) / 8 > 0x7FFFFFFFull) return MHC_ERR_UNSUPPORTED;
    const mhc::PostBwdCall c{g, x, y, res, grad_x, grad_y, grad_res, uint64_t(T), uint64_t(H), int(n),
                             int(path), num_sms(), reinterpret_cast<cudaStream_t>(stream)};
    const mhc::SigmoidCoeffs k{mix, alpha, b, grad_z, grad_mix, false};
    return finish(mhc::post_bwd(c, k, dtype == MHC_DTYPE_BF16 ? mhc::kBF16 : mhc::kF16));
}

}  // namespace

// --------------------------------------------------------------------------
// C ABI
// --------------------------------------------------------------------------

extern "C" {

int32_t mhc_h_aggregate_abi_version(void) { return kAbiVersion; }

const char* mhc_status_string(mhc_status_t status) {
    switch (status) {
        case MHC_OK: return "MHC_OK";
        case MHC_ERR_INVALID_ARG:
            return "MHC_ERR_INVALID_ARG: bad size, dtype, null, misaligned or overlapping buffer";
        case MHC_ERR_UNSUPPORTED:
            return "MHC_ERR_UNSUPPORTED: stream count not in {1,2,4,8}, or H too large for the 32-bit row index";
        case MHC_ERR_CUDA: return "MHC_ERR_CUDA: kernel launch failed (see mhc_h_aggregate_last_cuda_error)";
    }
    return "unknown mhc_status_t";
}

int32_t mhc_h_aggregate_last_cuda_error(void) { return g_last_cuda_error; }

int64_t mhc_h_aggregate_wait_timeouts(void) { return mhc::take_wait_timeouts(); }

mhc_path_t mhc_h_aggregate_fwd_path(const void* residual, const float* pre, const void* out,
                                    int64_t T, int64_t H) {
    return fwd_path(residual, pre, out, T, 4, H);
}

mhc_path_t mhc_h_aggregate_bwd_path(const void* grad_out, const void* residual, const float* pre,
                                    const void* grad_residual, const float* grad_pre, int64_t T,
                                    int64_t H) {
    return bwd_path(grad_out, residual, pre, grad_residual, grad_pre, T, 4, H);
}

mhc_status_t mhc_h_aggregate_fwd(const void* residual, const float* pre, void* out, int64_t T,
                                 int64_t H, mhc_stream_t stream) {
    return aggregate_fwd(residual, pre, out, T, 4, H, MHC_DTYPE_BF16, stream);
}

mhc_status_t mhc_h_aggregate_bwd(const void* grad_out, const void* residual, const float* pre,
                                 void* grad_residual, float* grad_pre, int64_t T, int64_t H,
                                 mhc_stream_t stream) {
    return aggregate_bwd(grad_out, residual, pre, grad_residual, grad_pre, T, 4, H, MHC_DTYPE_BF16,
                         stream);
}

mhc_status_t mhc_aggregate_fwd(const void* residual, const float* pre, void* out, int64_t T,
                               int32_t n, int64_t H, mhc_dtype_t dtype, mhc_stream_t stream) {
    return aggregate_fwd(residual, pre, out, T, n, H, int32_t(dtype), stream);
}

mhc_status_t mhc_aggregate_bwd(const void* grad_out, const void* residual, const float* pre,
                               void* grad_residual, float* grad_pre, int64_t T, int32_t n,
                               int64_t H, mhc_dtype_t dtype, mhc_stream_t stream) {
    return aggregate_bwd(grad_out, residual, pre, grad_residual, grad_pre, T, n, H, int32_t(dtype),
                         stream);
}

mhc_path_t mhc_aggregate_fwd_path(const void* residual, const float* pre, const void* out, int64_t T,
                                  int32_t n, int64_t H) {
    return fwd_path(residual, pre, out, T, n, H);
}

mhc_path_t mhc_aggregate_bwd_path(const void* grad_out, const void* residual, const float* pre,
                                  const void* grad_residual, const float* grad_pre, int64_t T,
                                  int32_t n, int64_t H) {
    return bwd_path(grad_out, residual, pre, grad_residual, grad_pre, T, n, H);
}

mhc_status_t mhc_pre_sigmoid(const float* mix, const float* alpha, const float* b, float* pre,
                             int64_t T, int32_t n, mhc_stream_t stream) {
    return pre_sigmoid(mix, alpha, b, pre, T, n, stream);
}

mhc_status_t mhc_aggregate_sigmoid_fwd(const void* residual, const float* mix, const float* alpha,
                                       const float* b, void* out, int64_t T, int32_t n, int64_t H,
                                       mhc_dtype_t dtype, mhc_stream_t stream) {
    return aggregate_sigmoid_fwd(residual, mix, alpha, b, out, T, n, H, int32_t(dtype), stream);
}

mhc_status_t mhc_aggregate_sigmoid_bwd(const void* grad_out, const void* residual, const float* mix,
                                       const float* alpha, const float* b, void* grad_residual,
                                       float* grad_z, float* grad_mix, int64_t T, int32_t n,
                                       int64_t H, mhc_dtype_t dtype, mhc_stream_t stream) {
    return aggregate_sigmoid_bwd(grad_out, residual, mix, alpha, b, grad_residual, grad_z, grad_mix,
                                 T, n, H, int32_t(dtype), stream);
}

mhc_status_t mhc_sigmoid_param_grad(const float* grad_z, const float* mix, float* grad_b,
                                    float* grad_alpha, int64_t T, int32_t n, mhc_stream_t stream) {
    return sigmoid_param_grad(grad_z, mix, grad_b, grad_alpha, T, n, stream);
}

mhc_status_t mhc_post_fwd(const void* x, const void* y, const float* post, const float* res,
                          void* out, int64_t T, int32_t n, int64_t H, mhc_dtype_t dtype,
                          mhc_stream_t stream) {
    return post_fwd(x, y, post, res, out, T, n, H, int32_t(dtype), stream);
}

mhc_status_t mhc_post_bwd(const void* grad_out, const void* x, const void* y, const float* post,
                          const float* res, void* grad_x, void* grad_y, float* grad_post,
                          float* grad_res, int64_t T, int32_t n, int64_t H, mhc_dtype_t dtype,
                          mhc_stream_t stream) {
    return post_bwd(grad_out, x, y, post, res, grad_x, grad_y, grad_post, grad_res, T, n, H,
                    int32_t(dtype), stream);
}

mhc_status_t mhc_post_sigmoid_fwd(const void* x, const void* y, const float* mix, const float* alpha,
                                  const float* b, const float* res, void* out, int64_t T, int32_t n,
                                  int64_t H, mhc_dtype_t dtype, mhc_stream_t stream) {
    return post_sigmoid_fwd(x, y, mix, alpha, b, res, out, T, n, H, int32_t(dtype), stream);
}

mhc_status_t mhc_post_sigmoid_bwd(const void* grad_out, const void* x, const void* y, const float* mix,
                                  const float* alpha, const float* b, const float* res, void* grad_x,
                                  void* grad_y, float* grad_z, float* grad_mix, float* grad_res,
                                  int64_t T, int32_t n, int64_t H, mhc_dtype_t dtype,
                                  mhc_stream_t stream) {
    return post_sigmoid_bwd(grad_out, x, y, mix, alpha, b, res, grad_x, grad_y, grad_z, grad_mix,
                            grad_res, T, n, H, int32_t(dtype), stream);
}

mhc_path_t mhc_post_fwd_path(const void* x, const void* y, const float* post, const float* res,
                             const void* out, int64_t T, int32_t n, int64_t H) {
    return post_fwd_path(x, y, post, res, out, T, n, H);
}

mhc_path_t mhc_post_bwd_path(const void* grad_out, const void* x, const void* y, const float* post,
                             const float* res, const void* grad_x, const void* grad_y,
                             const float* grad_post, const float* grad_res, int64_t T, int32_t n,
                             int64_t H) {
    return post_bwd_path(grad_out, x, y, post, res, grad_x, grad_y, grad_post, grad_res, T, n, H);
}

}  // extern "C"
