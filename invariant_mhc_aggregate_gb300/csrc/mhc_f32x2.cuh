// Packed binary32 pairs for sm_100-class GPUs: one instruction rounds two
// independent RN operations (add.rn.f32x2, mul.rn.f32x2), each half
// bit-identical to the scalar __fadd_rn / __fmul_rn on that half.  They halve
// the issue slots of the ALU-heavy kernels (the n = 8 mHC post), whose sums
// and products are otherwise the same scalar RN operations.
//
// One rule keeps them exact: a packed product is never an operand of a
// packed sum.  ptxas merges mul.rn.f32x2 followed by a dependent
// add.rn.f32x2 into one fused multiply-add (measured: about a quarter of the
// results then differ from the two rounded steps), which the no-FMA rule of
// "Add batch-invariant h_aggregate kernel", Batch invariance, forbids.  So
// the halves of a packed product are summed by scalar adds (padd_halves,
// scalar __fadd_rn), and a packed sum only takes values that are themselves
// sums (or loads and shuffles of sums).  Every such combination was measured
// bit-identical to the scalar sequence, and the kernels that use them are
// compared with the CPU oracle byte for byte.

#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mhc {

// Two binary32 values in one 64-bit register pair (lo = first, hi = second).
struct F2 {
    uint64_t v;
};

__device__ __forceinline__ F2 f2(float lo, float hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float f2_lo(F2 a) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
    return lo;
}

__device__ __forceinline__ float f2_hi(F2 a) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
    return hi;
}

// Products of the halves: {a.lo * b.lo, a.hi * b.hi}, each RN.  Its result
// goes to scalar adds only (see above).
__device__ __forceinline__ F2 pmul(F2 a, F2 b) {
    F2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

// Sums of the halves: {a.lo + b.lo, a.hi + b.hi}, each RN.  Its operands are
// sums, never products.
__device__ __forceinline__ F2 padd(F2 a, F2 b) {
    F2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

// The scalar sum of a packed product's two halves, lo + hi (RN).
__device__ __forceinline__ float padd_halves(F2 p) { return __fadd_rn(f2_lo(p), f2_hi(p)); }

// {a.lo + b.lo, a.hi + b.hi} by two scalar adds: the level of a tree whose
// operands are halves of packed products.
__device__ __forceinline__ F2 sadd2(F2 a, F2 b) {
    return f2(__fadd_rn(f2_lo(a), f2_lo(b)), __fadd_rn(f2_hi(a), f2_hi(b)));
}

__device__ __forceinline__ F2 shfl_xor_f2(uint32_t mask, F2 a, int lane_mask) {
    return f2(__shfl_xor_sync(mask, f2_lo(a), lane_mask), __shfl_xor_sync(mask, f2_hi(a), lane_mask));
}

}  // namespace mhc
