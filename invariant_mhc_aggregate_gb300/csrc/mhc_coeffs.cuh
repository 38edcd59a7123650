// Where a kernel's per-token coefficients come from, and where its per-token
// coefficient gradients go.  The aggregate kernels of mhc_device.cuh are
// templated on one of these "coefficient sources":
//
//  * PlainCoeffs: the pages' op.  pre [T,n] FP32 is an input; the backward
//    writes grad_pre [T,n].
//  * SigmoidCoeffs: the pre coefficients computed in the kernel from the mix,
//      z[t,k] = RN(RN(alpha * mix[t,k]) + b[k]),  pre[t,k] = sigmoid(z[t,k]),
//    and the backward writes grad_z = RN(grad_pre * sigmoid'(z)) and
//    grad_mix = RN(alpha * grad_z) instead of grad_pre.
//
// Source: "perf: fuse mHC coefficient backward epilogue" (Liger-Kernel pull
// request 1402), Summary: the coefficient backward ends in the derivatives of
// the pre / post sigmoids, grad_mix and the gradients of the bias b and the
// scalar alphas.  The page prints no formula; the ones above are this
// library's reading for the pre coefficients, and the binary32 evaluation of
// the sigmoid below is this library's definition, so that every result is a
// fixed function of the input bits on any device:
//
//  exp32(x): argument reduction of W. J. Cody and W. Waite ("Software Manual
//    for the Elementary Functions", 1980), x = k ln2 + r with k the integer
//    nearest x*log2e (ties to even) and r = (x - k*L1) - k*L2, where ln 2 =
//    L1 + L2 and L1 has 15 significant bits (k*L1 exact); e^r by the degree-7
//    Taylor polynomial (coefficients RN(1/i!)) in Horner form from the top
//    term; the result scaled by 2^(k/2) (exact) and then 2^(k - k/2) (one
//    rounding, also into the subnormal range).  NaN -> NaN, x > 89 -> +inf,
//    x < -104 -> +0.  Within 1.2 ulp of e^x on [-104, 0].
//  sigmoid32(z): e = exp32(-|z|), d = 1 + e; for z >= 0 sigmoid = 1/d and
//    1 - sigmoid = e/d, for z < 0 the two swap; sigmoid' = sigmoid *
//    (1 - sigmoid).  Every operation is one RN binary32 operation
//    (__fmul_rn, __fadd_rn, __fdiv_rn, the exact rintf), never contracted.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mhc {

__device__ __forceinline__ float exp32(float x) {
    if (x != x) return x;
    if (x > 89.0f) return __int_as_float(0x7F800000);
    if (x < -104.0f) return 0.0f;
    constexpr float kLog2e = 0x1.715476p+0f;   // RN(log2 e)
    constexpr float kL1 = 0x1.62e4p-1f;        // ln 2, leading 15 bits
    constexpr float kL2 = 0x1.7f7d1cp-20f;     // RN(ln 2 - kL1)
    const float k = rintf(__fmul_rn(x, kLog2e));
    const float r = __fadd_rn(__fadd_rn(x, -__fmul_rn(k, kL1)), -__fmul_rn(k, kL2));
    // Taylor coefficients RN(1/i!), i = 7 .. 2 (1/1! and 1/0! are 1)
    float q = 0x1.a01a02p-13f;
    q = __fadd_rn(0x1.6c16c2p-10f, __fmul_rn(r, q));
    q = __fadd_rn(0x1.111112p-7f, __fmul_rn(r, q));
    q = __fadd_rn(0x1.555556p-5f, __fmul_rn(r, q));
    q = __fadd_rn(0x1.555556p-3f, __fmul_rn(r, q));
    q = __fadd_rn(0x1p-1f, __fmul_rn(r, q));
    q = __fadd_rn(1.0f, __fmul_rn(r, q));
    q = __fadd_rn(1.0f, __fmul_rn(r, q));
    const int ki = static_cast<int>(k);
    const int k1 = ki / 2;
    const float scaled = __fmul_rn(q, __int_as_float((k1 + 127) << 23));
    return __fmul_rn(scaled, __int_as_float((ki - k1 + 127) << 23));
}

// sigmoid(z) in s and 1 - sigmoid(z) in t.
__device__ __forceinline__ void sigmoid32(float z, float& s, float& t) {
    const float a = (z < 0.0f) ? -z : z;
    const float e = exp32(-a);
    const float d = __fadd_rn(1.0f, e);
    const float big = __fdiv_rn(1.0f, d);
    const float small = __fdiv_rn(e, d);
    const bool nonneg = z >= 0.0f;
    s = nonneg ? big : small;
    t = nonneg ? small : big;
}

__device__ __forceinline__ float pre_activation(float alpha, float mix, float b) {
    return __fadd_rn(__fmul_rn(alpha, mix), b);
}

// The N values of a token's [.., N] FP32 row, with float2 / float4 loads when
// `vec` says the row is aligned to min(16, 4N) bytes (read-only, kept in L1:
// every thread of the token reads them).
template <int N>
__device__ __forceinline__ void ld_row(const float* p, bool vec, float (&out)[N]) {
    if (N == 1) {
        out[0] = __ldg(p);
    } else if (vec && N == 2) {
        const float2 v = __ldg(reinterpret_cast<const float2*>(p));
        out[0] = v.x;
        out[N - 1] = v.y;
    } else if (vec) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(p) + i);
            out[4 * i + 0] = v.x;
            out[4 * i + 1] = v.y;
            out[4 * i + 2] = v.z;
            out[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < N; ++k) out[k] = __ldg(p + k);
    }
}

// A kernel either has each thread load (and, for the sigmoid, compute) the
// coefficients it needs (kBlockTable false: load() then to_pre()), or has a
// few threads compute each token's values once into shared memory for the
// whole block (kBlockTable true: mix_at() early, pre_from() later), which is
// what the sigmoid wants: its binary32 evaluation costs about 70
// instructions per value, too many to repeat in every thread of a token.
struct PlainCoeffs {
    const float* pre;   // [T,n]
    float* grad_pre;    // [T,n] (backward only)
    bool vec;           // pre aligned to min(16, 4n) bytes

    static constexpr bool kBlockTable = false;

    // The same source for the tokens from t0 on (offset = n * t0 values).
    __host__ __device__ PlainCoeffs shifted(uint64_t offset) const {
        return PlainCoeffs{pre + offset, grad_pre ? grad_pre + offset : nullptr, vec};
    }

    // Issue the loads of token t's coefficients into p ...
    template <int N>
    __device__ __forceinline__ void load(uint64_t t, float (&p)[N]) const {
        ld_row<N>(pre + uint64_t(N) * t, vec, p);
    }
    // ... and turn what load() left in p into pre, once the kernel has issued
    // its other loads (nothing to do here).
    template <int N>
    __device__ __forceinline__ void to_pre(float (&)[N]) const {}
    // Token t's pre in every lane of a warp (all 32 lanes call it).
    template <int N>
    __device__ __forceinline__ void warp_pre(uint64_t t, float (&p)[N]) const {
        ld_row<N>(pre + uint64_t(N) * t, vec, p);
    }
    // Called by the thread that holds grad_pre[t,k].
    template <int N>
    __device__ __forceinline__ void store_grad(uint64_t t, int k, float gp) const {
        grad_pre[uint64_t(N) * t + k] = gp;
    }
};

struct SigmoidCoeffs {
    const float* mix;   // [T,n]
    const float* alpha; // [1]
    const float* b;     // [n]
    float* grad_z;      // [T,n] (backward only)
    float* grad_mix;    // [T,n] (backward only)
    bool vec;           // mix aligned to min(16, 4n) bytes

    static constexpr bool kBlockTable = true;

    // mix value idx = n*t + k of the [T,n] mix (issued early: the kernels
    // fetch it before their bulk loads and turn it into pre afterwards) ...
    __device__ __forceinline__ float mix_at(uint64_t idx) const { return __ldg(mix + idx); }
    // ... and pre for that value ...
    __device__ __forceinline__ float pre_from(float m, int k) const {
        float s, one_minus;
        sigmoid32(pre_activation(__ldg(alpha), m, __ldg(b + k)), s, one_minus);
        return s;
    }
    // ... or pre and sigmoid' = RN(sigmoid * (1 - sigmoid)) for it (the
    // backward keeps the slope for its epilogue).
    __device__ __forceinline__ void pre_and_slope(float m, int k, float& s, float& slope) const {
        float one_minus;
        sigmoid32(pre_activation(__ldg(alpha), m, __ldg(b + k)), s, one_minus);
        slope = __fmul_rn(s, one_minus);
    }
    // Token t's pre in every lane of a warp (all 32 lanes call it): lanes
    // 0 .. N-1 evaluate one sigmoid each, shuffles broadcast them.
    template <int N>
    __device__ __forceinline__ void warp_pre(uint64_t t, float (&p)[N]) const {
        const uint32_t lane = threadIdx.x & 31u;
        float mine = 0.0f;
        if (lane < uint32_t(N)) mine = pre_from(mix_at(uint64_t(N) * t + lane), int(lane));
#pragma unroll
        for (int k = 0; k < N; ++k) p[k] = __shfl_sync(0xffffffffu, mine, k);
    }

    __host__ __device__ SigmoidCoeffs shifted(uint64_t offset) const {
        return SigmoidCoeffs{mix + offset, alpha, b, grad_z ? grad_z + offset : nullptr,
                             grad_mix ? grad_mix + offset : nullptr, vec};
    }

    // load() leaves mix[t, :] in p; to_pre() replaces it by the sigmoids.
    template <int N>
    __device__ __forceinline__ void load(uint64_t t, float (&p)[N]) const {
        ld_row<N>(mix + uint64_t(N) * t, vec, p);
    }
    template <int N>
    __device__ __forceinline__ void to_pre(float (&p)[N]) const {
        const float a = __ldg(alpha);
#pragma unroll
        for (int k = 0; k < N; ++k) {
            float one_minus;
            sigmoid32(pre_activation(a, p[k], __ldg(b + k)), p[k], one_minus);
        }
    }
    template <int N>
    __device__ __forceinline__ void store_grad(uint64_t t, int k, float gp) const {
        const uint64_t i = uint64_t(N) * t + k;
        float s, slope;
        pre_and_slope(__ldg(mix + i), k, s, slope);
        store_grad_slope<N>(t, k, gp, slope);
    }
    // The same with sigmoid'(z[t,k]) already at hand.
    template <int N>
    __device__ __forceinline__ void store_grad_slope(uint64_t t, int k, float gp, float slope) const {
        const uint64_t i = uint64_t(N) * t + k;
        const float gz = __fmul_rn(gp, slope);
        grad_z[i] = gz;
        grad_mix[i] = __fmul_rn(__ldg(alpha), gz);
    }
};

}  // namespace mhc
