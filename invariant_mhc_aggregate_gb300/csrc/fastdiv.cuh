// Division of 32-bit unsigned integers by a divisor fixed at launch time,
// by multiplication and shift: the round-up method of T. Granlund and
// P. L. Montgomery, "Division by invariant integers using multiplication"
// (PLDI 1994), Theorem 4.2 with a 33-bit multiplier 2^32 + m.
//
// For a divisor d >= 1 let l = ceil(log2 d) and
//   m = floor(2^32 * (2^l - d) / d) + 1          (fits in 32 bits);
// then for every 0 <= n < 2^32
//   n / d = (mulhi32(m, n) + n) >> l,
// where the sum is taken in 64 bits so that it cannot overflow.
//
// Plain C++ when not compiled by nvcc, so that host tests can check it.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define MHC_HD __host__ __device__ __forceinline__
#else
#define MHC_HD inline
#endif

struct FastDivU32 {
    uint32_t d;
    uint32_t m;
    uint32_t l;
};

inline FastDivU32 make_fastdiv_u32(uint32_t d) {
    FastDivU32 f;
    f.d = d;
    uint32_t l = 0;
    while (l < 32 && (uint64_t(1) << l) < d) ++l;
    f.l = l;
    uint64_t two_l = uint64_t(1) << l;
    f.m = uint32_t(((uint64_t(1) << 32) * (two_l - d)) / d + 1);
    return f;
}

MHC_HD uint32_t mulhi_u32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
    return __umulhi(a, b);
#else
    return uint32_t((uint64_t(a) * uint64_t(b)) >> 32);
#endif
}

MHC_HD uint32_t fastdiv_u32(uint32_t n, const FastDivU32& f) {
    return uint32_t((uint64_t(mulhi_u32(f.m, n)) + n) >> f.l);
}
