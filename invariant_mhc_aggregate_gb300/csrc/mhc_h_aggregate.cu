// Batch-invariant mHC pre "H Aggregate" for GB300 (sm_103a): forward and
// fused backward kernels behind the C ABI declared in mhc_h_aggregate.h.
//
// Source: "Add batch-invariant h_aggregate kernel" (RL-Kernel pull request
// 366).  Summary: residual [T,4,H] BF16, pre [T,4] FP32, out [T,H] BF16,
//   out = bf16((pre0*r0 + pre1*r1) + (pre2*r2 + pre3*r3)).
// Batch invariance: one writer per output, no atomics, FP32 __fmul_rn /
// __fadd_rn, the fixed (0 + 1) + (2 + 3) tree, BF16 only at the boundaries.
// The backward answers that page's reviewer request; its formula is the exact
// derivative of the Summary formula and its grad_pre order (ORDER-256) is
// defined in mhc_h_aggregate.h.
//
// Design (GB300, HBM-bound: about 0.7 FP32 operations per byte moved):
//  * Vector paths move NW 32-bit words per access: NW = 8 uses the 256-bit
//    (32-byte) global loads and stores that sm_100-class GPUs added
//    (ld/st .v8.b32), NW = 4 the 16-byte ones.  One access covers 2*NW BF16
//    values, i.e. NW/4 "chunks" of 8 values.
//  * Forward: a flat grid over output vectors.  A thread loads the four
//    residual vectors feeding its output vector with streaming loads and the
//    token's pre as one 16-byte load, and stores one vector.  Large calls
//    give each thread UNROLL vectors, all loads issued before any arithmetic,
//    to keep enough bytes in flight per SM; decode-sized calls give each
//    thread one vector so the work spreads over as many SMs as possible.  The
//    arithmetic of an element never depends on the grid, the block or T.
//  * Backward: one block per token (grid-stride over tokens) whose threads
//    own the 256 lanes of ORDER-256, NW/4 lanes each: thread j holds the
//    chunks of lanes (NW/4)*j .. (NW/4)*j + NW/4 - 1, which are adjacent, so
//    one vector access serves all of them.  It streams g and the four residual
//    rows, writes grad_residual, and adds the chunk partials of each lane in
//    increasing chunk order.  Groups of 32 lanes fold with warp shuffles (and
//    one in-thread add when a thread holds two lanes), the 8 groups through
//    shared memory.  No atomics, no cross-block traffic.
//  * Narrower paths (H not a multiple of 8, or buffers not 16-byte aligned)
//    run the same per-element arithmetic and the same grad_pre tree with 4- or
//    2-byte accesses, so every path gives the same bytes.
//  * No tensor cores: nothing here is a contraction.
//  * Built without fast math, with --fmad=false and -ftz=false; the
//    intrinsics below already forbid contraction and flushing.

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "mhc_h_aggregate.h"
#include "fastdiv.cuh"

namespace {

constexpr int kAbiVersion = 1;

// --------------------------------------------------------------------------
// memory access helpers
// --------------------------------------------------------------------------

template <int NW>
struct Words {
    uint32_t w[NW];
};

// Vector load of data read exactly once: read-only path, no L1 allocation.
template <int NW>
__device__ __forceinline__ Words<NW> ld_stream(const void* p);

template <>
__device__ __forceinline__ Words<4> ld_stream<4>(const void* p) {
    Words<4> v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
    return v;
}

template <>
__device__ __forceinline__ Words<8> ld_stream<8>(const void* p) {
    Words<8> v;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]),
                   "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
    return v;
}

// Vector store of data written exactly once: streaming (evict-first).
template <int NW>
__device__ __forceinline__ void st_stream(void* p, const Words<NW>& v);

template <>
__device__ __forceinline__ void st_stream<4>(void* p, const Words<4>& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                 :
                 : "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
}

template <>
__device__ __forceinline__ void st_stream<8>(void* p, const Words<8>& v) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :
                 : "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]),
                   "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_stream4(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream4(void* p, uint32_t v) {
    asm volatile("st.global.cs.u32 [%0], %1;" : : "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint16_t ld_stream2(const void* p) {
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream2(void* p, uint16_t v) {
    asm volatile("st.global.cs.u16 [%0], %1;" : : "l"(p), "h"(v) : "memory");
}

// pre[t] is read by every thread of the token: keep it in L1.
__device__ __forceinline__ float4 ld_pre16(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ float4 ld_pre4x(const float* p) {
    return make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
}

template <bool PRE_VEC>
__device__ __forceinline__ float4 ld_pre(const float* p) {
    return PRE_VEC ? ld_pre16(p) : ld_pre4x(p);
}

// Programmatic dependent launch.  Every kernel here is launched so that it may
// become resident while the previous kernel in its stream is still finishing
// (its blocks then wait here, in hardware, until that kernel has completed and
// its memory is visible), and lets the next kernel do the same.  Nothing is
// read or written before the wait, so a producer of any input, or a reader of
// any output, earlier in the stream is always respected.  Outside such a
// launch both instructions do nothing.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

// --------------------------------------------------------------------------
// BF16 <-> FP32 (widening is exact: the BF16 pattern is the upper half)
// --------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_one(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Two FP32 values -> two BF16 values (round to nearest even), lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
    __nv_bfloat16 v = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&v);
}

// --------------------------------------------------------------------------
// the forward element: four RN products, the (0 + 1) + (2 + 3) tree
// --------------------------------------------------------------------------

__device__ __forceinline__ float h_agg(const float4 p, float r0, float r1, float r2, float r3) {
    const float p0 = __fmul_rn(p.x, r0);
    const float p1 = __fmul_rn(p.y, r1);
    const float p2 = __fmul_rn(p.z, r2);
    const float p3 = __fmul_rn(p.w, r3);
    return __fadd_rn(__fadd_rn(p0, p1), __fadd_rn(p2, p3));
}

// Two adjacent elements held as BF16 pairs in one 32-bit word per k.
__device__ __forceinline__ uint32_t h_agg_pair(const float4 p, uint32_t w0, uint32_t w1,
                                               uint32_t w2, uint32_t w3) {
    const float lo = h_agg(p, bf16_lo(w0), bf16_lo(w1), bf16_lo(w2), bf16_lo(w3));
    const float hi = h_agg(p, bf16_hi(w0), bf16_hi(w1), bf16_hi(w2), bf16_hi(w3));
    return pack_bf16x2(lo, hi);
}

template <int NW>
__device__ __forceinline__ Words<NW> h_agg_vec(const float4 p, const Words<NW> (&r)[4]) {
    Words<NW> o;
#pragma unroll
    for (int e = 0; e < NW; ++e) o.w[e] = h_agg_pair(p, r[0].w[e], r[1].w[e], r[2].w[e], r[3].w[e]);
    return o;
}

// --------------------------------------------------------------------------
// forward kernels
// --------------------------------------------------------------------------

// Vector path.  Output vector i (i = t*V + v, V = H / (2*NW) vectors per row)
// is out[i]; the residual vector of row k is res[t*4V + k*V + v] =
// res[i + 3tV + kV].
template <int NW, int BLOCK, int UNROLL, bool PRE_VEC>
__global__ void __launch_bounds__(BLOCK)
h_agg_fwd_vec_kernel(const Words<NW>* __restrict__ res, const float* __restrict__ pre,
                     Words<NW>* __restrict__ out, uint32_t n_vec, uint32_t V, FastDivU32 divV) {
    pdl_enter();
    const uint32_t first = blockIdx.x * uint32_t(BLOCK * UNROLL) + threadIdx.x;
    Words<NW> r[UNROLL][4];
    float4 p[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const uint32_t i = first + uint32_t(u * BLOCK);
        if (i < n_vec) {
            const uint32_t t = fastdiv_u32(i, divV);
            const Words<NW>* src = res + (uint64_t(i) + 3ull * uint64_t(t) * V);
#pragma unroll
            for (int k = 0; k < 4; ++k) r[u][k] = ld_stream<NW>(src + uint64_t(k) * V);
            p[u] = ld_pre<PRE_VEC>(pre + 4ull * t);
        }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const uint32_t i = first + uint32_t(u * BLOCK);
        if (i < n_vec) st_stream<NW>(out + i, h_agg_vec<NW>(p[u], r[u]));
    }
}

// 4-byte path (H even): pair i = t*P + c, P = H/2.
__global__ void __launch_bounds__(256)
h_agg_fwd_pair_kernel(const uint32_t* __restrict__ res2, const float* __restrict__ pre,
                      uint32_t* __restrict__ out2, uint64_t n_pairs, uint64_t P) {
    pdl_enter();
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_pairs; i += stride) {
        const uint64_t t = i / P;
        const uint32_t* src = res2 + (i + 3 * t * P);
        const uint32_t w0 = ld_stream4(src);
        const uint32_t w1 = ld_stream4(src + P);
        const uint32_t w2 = ld_stream4(src + 2 * P);
        const uint32_t w3 = ld_stream4(src + 3 * P);
        st_stream4(out2 + i, h_agg_pair(ld_pre4x(pre + 4 * t), w0, w1, w2, w3));
    }
}

// 2-byte path (any H, any 2-byte alignment): element i = t*H + h.
__global__ void __launch_bounds__(256)
h_agg_fwd_element_kernel(const uint16_t* __restrict__ res, const float* __restrict__ pre,
                         uint16_t* __restrict__ out, uint64_t n, uint64_t H) {
    pdl_enter();
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint64_t t = i / H;
        const uint16_t* src = res + (i + 3 * t * H);
        const float r0 = bf16_one(ld_stream2(src));
        const float r1 = bf16_one(ld_stream2(src + H));
        const float r2 = bf16_one(ld_stream2(src + 2 * H));
        const float r3 = bf16_one(ld_stream2(src + 3 * H));
        st_stream2(out + i, to_bf16(h_agg(ld_pre4x(pre + 4 * t), r0, r1, r2, r3)));
    }
}

// --------------------------------------------------------------------------
// backward
// --------------------------------------------------------------------------

constexpr int kLanes = 256;   // lanes of ORDER-256
constexpr int kGroups = 8;    // groups of 32 lanes

// grad_residual for two adjacent elements: bf16(RN(pre_k * g)).
__device__ __forceinline__ uint32_t scale_pair(float pk, uint32_t gw) {
    return pack_bf16x2(__fmul_rn(pk, bf16_lo(gw)), __fmul_rn(pk, bf16_hi(gw)));
}

template <int NW>
__device__ __forceinline__ Words<NW> scale_vec(float pk, const Words<NW>& g) {
    Words<NW> o;
#pragma unroll
    for (int e = 0; e < NW; ++e) o.w[e] = scale_pair(pk, g.w[e]);
    return o;
}

// ((q0+q1)+(q2+q3)) + ((q4+q5)+(q6+q7)) of q_e = g_e * r_e (exact products)
// for the chunk held in words w0 .. w0+3 of g and r.
template <int NW>
__device__ __forceinline__ float chunk_partial(const Words<NW>& g, const Words<NW>& r, int w0) {
    const float q0 = __fmul_rn(bf16_lo(g.w[w0 + 0]), bf16_lo(r.w[w0 + 0]));
    const float q1 = __fmul_rn(bf16_hi(g.w[w0 + 0]), bf16_hi(r.w[w0 + 0]));
    const float q2 = __fmul_rn(bf16_lo(g.w[w0 + 1]), bf16_lo(r.w[w0 + 1]));
    const float q3 = __fmul_rn(bf16_hi(g.w[w0 + 1]), bf16_hi(r.w[w0 + 1]));
    const float q4 = __fmul_rn(bf16_lo(g.w[w0 + 2]), bf16_lo(r.w[w0 + 2]));
    const float q5 = __fmul_rn(bf16_hi(g.w[w0 + 2]), bf16_hi(r.w[w0 + 2]));
    const float q6 = __fmul_rn(bf16_lo(g.w[w0 + 3]), bf16_lo(r.w[w0 + 3]));
    const float q7 = __fmul_rn(bf16_hi(g.w[w0 + 3]), bf16_hi(r.w[w0 + 3]));
    return __fadd_rn(__fadd_rn(__fadd_rn(q0, q1), __fadd_rn(q2, q3)),
                     __fadd_rn(__fadd_rn(q4, q5), __fadd_rn(q6, q7)));
}

__device__ __forceinline__ float chunk_partial8(const float q[8]) {
    return __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                     __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
}

// Steps 4 and 5 of ORDER-256 for a block of 256/LPT threads, thread j holding
// lanes LPT*j + l (l < LPT) in acc[l][k].  A group of 32 lanes is 32/LPT
// adjacent threads: lane strides 16 .. LPT are thread strides 16/LPT .. 1
// (xor shuffles), lane stride 1 (when LPT == 2) is the add of a thread's own
// two lanes.  The 8 group values then fold with strides 4, 2, 1 in shared
// memory, and grad_pre[t, 0..3] is written.  All threads of the block call it.
template <int LPT>
__device__ __forceinline__ void fold_lanes_and_store(float (&acc)[LPT][4], float (*red)[4],
                                                     float* __restrict__ grad_pre_t) {
    constexpr int kThreadsPerGroup = 32 / LPT;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int s = kThreadsPerGroup / 2; s >= 1; s >>= 1) {
#pragma unroll
            for (int l = 0; l < LPT; ++l)
                acc[l][k] = __fadd_rn(acc[l][k], __shfl_xor_sync(0xffffffffu, acc[l][k], s));
        }
        if (LPT == 2) acc[0][k] = __fadd_rn(acc[0][k], acc[LPT - 1][k]);
    }
    if ((threadIdx.x % kThreadsPerGroup) == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) red[threadIdx.x / kThreadsPerGroup][k] = acc[0][k];
    }
    __syncthreads();
    if (threadIdx.x < 4) {
        const int k = threadIdx.x;
        float w[kGroups];
#pragma unroll
        for (int i = 0; i < kGroups; ++i) w[i] = red[i][k];
#pragma unroll
        for (int s = kGroups / 2; s >= 1; s >>= 1) {
#pragma unroll
            for (int i = 0; i < s; ++i) w[i] = __fadd_rn(w[i], w[i + s]);
        }
        grad_pre_t[k] = w[0];
    }
    __syncthreads();  // red[] is reused by the next token of this block
}

// Vector path: H % (2*NW) == 0 and g / residual / grad_residual aligned to
// 4*NW bytes.  V = H / (2*NW) vectors per row; thread j handles vectors
// j, j + B, j + 2B, ... (B = 256/LPT threads), i.e. for lane LPT*j + l the
// chunks LPT*(j + mB) + l = (LPT*j + l) + 256m: exactly that lane's chunks,
// in increasing order.  Up to BATCH vectors per thread are held in registers
// per pass.
template <int NW, int BATCH, int MIN_BLOCKS, bool PRE_VEC>
__global__ void __launch_bounds__(kLanes / (NW / 4), MIN_BLOCKS)
h_agg_bwd_vec_kernel(const Words<NW>* __restrict__ g, const Words<NW>* __restrict__ res,
                     const float* __restrict__ pre, Words<NW>* __restrict__ gres,
                     float* __restrict__ grad_pre, uint64_t T, uint32_t V) {
    pdl_enter();
    constexpr int LPT = NW / 4;
    constexpr uint32_t B = kLanes / LPT;
    __shared__ float red[kGroups][4];
    const uint32_t j = threadIdx.x;
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const float4 p4 = ld_pre<PRE_VEC>(pre + 4 * t);
        const float pk[4] = {p4.x, p4.y, p4.z, p4.w};
        const Words<NW>* gt = g + t * V;
        const Words<NW>* rt = res + 4 * t * V;
        Words<NW>* grt = gres + 4 * t * V;
        float acc[LPT][4];
#pragma unroll
        for (int l = 0; l < LPT; ++l)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[l][k] = 0.0f;
        for (uint32_t v0 = j; v0 < V; v0 += B * BATCH) {
            Words<NW> gv[BATCH];
            Words<NW> rv[BATCH][4];
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const uint32_t v = v0 + uint32_t(b) * B;
                if (v < V) {
                    gv[b] = ld_stream<NW>(gt + v);
#pragma unroll
                    for (int k = 0; k < 4; ++k) rv[b][k] = ld_stream<NW>(rt + uint64_t(k) * V + v);
                }
            }
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const uint32_t v = v0 + uint32_t(b) * B;
                if (v < V) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        st_stream<NW>(grt + uint64_t(k) * V + v, scale_vec<NW>(pk[k], gv[b]));
#pragma unroll
                        for (int l = 0; l < LPT; ++l)
                            acc[l][k] = __fadd_rn(acc[l][k], chunk_partial<NW>(gv[b], rv[b][k], 4 * l));
                    }
                }
            }
        }
        fold_lanes_and_store<LPT>(acc, red, grad_pre + 4 * t);
    }
}

// 2-byte path: any H and any 2-byte alignment; same lanes, chunks and tree,
// with positions past H contributing +0.0.  256 threads, one lane each.
__global__ void __launch_bounds__(kLanes)
h_agg_bwd_element_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ res,
                         const float* __restrict__ pre, uint16_t* __restrict__ gres,
                         float* __restrict__ grad_pre, uint64_t T, uint64_t H) {
    pdl_enter();
    __shared__ float red[kGroups][4];
    const uint64_t C = (H + 7) / 8;
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const float4 p = ld_pre4x(pre + 4 * t);
        const float pk[4] = {p.x, p.y, p.z, p.w};
        const uint16_t* gt = g + t * H;
        const uint16_t* rt = res + 4 * t * H;
        uint16_t* grt = gres + 4 * t * H;
        float acc[1][4] = {{0.0f, 0.0f, 0.0f, 0.0f}};
        for (uint64_t c = threadIdx.x; c < C; c += kLanes) {
            float gf[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint64_t h = 8 * c + e;
                gf[e] = (h < H) ? bf16_one(ld_stream2(gt + h)) : 0.0f;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint64_t h = 8 * c + e;
                    if (h < H) {
                        q[e] = __fmul_rn(gf[e], bf16_one(ld_stream2(rt + uint64_t(k) * H + h)));
                        st_stream2(grt + uint64_t(k) * H + h, to_bf16(__fmul_rn(pk[k], gf[e])));
                    } else {
                        q[e] = 0.0f;
                    }
                }
                acc[0][k] = __fadd_rn(acc[0][k], chunk_partial8(q));
            }
        }
        fold_lanes_and_store<1>(acc, red, grad_pre + 4 * t);
    }
}

// --------------------------------------------------------------------------
// host side: validation, path choice, launch
// --------------------------------------------------------------------------

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

// Byte counts of [T,4,H] BF16 etc., or false when they overflow int64.
inline bool sizes_ok(int64_t T, int64_t H) {
    if (T < 0 || H <= 0) return false;
    if (T == 0) return true;
    const int64_t lim = INT64_MAX / 8;  // residual bytes = 8 * T * H
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

// Status of the launches since begin_launches(): a failed cudaLaunchKernelEx
// is recorded by launch(), anything else by cudaGetLastError().
void begin_launches() { g_last_cuda_error = 0; }

mhc_status_t finish_launch() {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) g_last_cuda_error = int32_t(e);
    return g_last_cuda_error != 0 ? MHC_ERR_CUDA : MHC_OK;
}

mhc_path_t fwd_path(const void* residual, const float* pre, const void* out, int64_t T, int64_t H) {
    if (!sizes_ok(T, H) || T == 0) return MHC_PATH_NONE;
    if (!residual || !pre || !out) return MHC_PATH_NONE;
    if (!aligned(residual, 2) || !aligned(out, 2) || !aligned(pre, 4)) return MHC_PATH_NONE;
    const uint64_t res_bytes = uint64_t(T) * 8 * uint64_t(H);
    const Range ro = range_of(out, uint64_t(T) * 2 * uint64_t(H));
    if (overlap(ro, range_of(residual, res_bytes)) || overlap(ro, range_of(pre, uint64_t(T) * 16)))
        return MHC_PATH_NONE;
    if (H % 16 == 0 && aligned(residual, 32) && aligned(out, 32)) return MHC_PATH_VEC32;
    if (H % 8 == 0 && aligned(residual, 16) && aligned(out, 16)) return MHC_PATH_VEC16;
    if (H % 2 == 0 && aligned(residual, 4) && aligned(out, 4)) return MHC_PATH_PAIR;
    return MHC_PATH_ELEMENT;
}

mhc_path_t bwd_path(const void* g, const void* residual, const float* pre, const void* gres,
                    const float* gpre, int64_t T, int64_t H) {
    if (!sizes_ok(T, H) || T == 0) return MHC_PATH_NONE;
    if (!g || !residual || !pre || !gres || !gpre) return MHC_PATH_NONE;
    if (!aligned(g, 2) || !aligned(residual, 2) || !aligned(gres, 2) || !aligned(pre, 4) ||
        !aligned(gpre, 4))
        return MHC_PATH_NONE;
    const uint64_t TH = uint64_t(T) * uint64_t(H);
    const Range rgr = range_of(gres, TH * 8);
    const Range rgp = range_of(gpre, uint64_t(T) * 16);
    const Range ins[3] = {range_of(g, TH * 2), range_of(residual, TH * 8), range_of(pre, uint64_t(T) * 16)};
    if (overlap(rgr, rgp)) return MHC_PATH_NONE;
    for (const Range& in : ins)
        if (overlap(rgr, in) || overlap(rgp, in)) return MHC_PATH_NONE;
    if (H % 16 == 0 && aligned(g, 32) && aligned(residual, 32) && aligned(gres, 32)) return MHC_PATH_VEC32;
    if (H % 8 == 0 && aligned(g, 16) && aligned(residual, 16) && aligned(gres, 16)) return MHC_PATH_VEC16;
    return MHC_PATH_ELEMENT;
}

// Launch with programmatic stream serialization (see pdl_enter).
template <typename... Params, typename... Args>
void launch(void (*kernel)(Params...), uint32_t grid, uint32_t block, cudaStream_t stream,
            Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
    if (e != cudaSuccess) g_last_cuda_error = int32_t(e);
}

inline uint32_t grid_for(uint64_t items, uint32_t per_block, uint64_t cap) {
    uint64_t b = (items + per_block - 1) / per_block;
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return uint32_t(b);
}

template <int NW, int BLOCK, int UNROLL>
void launch_fwd_vec(const void* residual, const float* pre, void* out, uint32_t n_vec, uint32_t V,
                    bool pre_vec, cudaStream_t stream) {
    const uint32_t per_block = uint32_t(BLOCK * UNROLL);
    const uint32_t blocks = uint32_t((uint64_t(n_vec) + per_block - 1) / per_block);
    const FastDivU32 divV = make_fastdiv_u32(V);
    const Words<NW>* r = static_cast<const Words<NW>*>(residual);
    Words<NW>* o = static_cast<Words<NW>*>(out);
    if (pre_vec)
        launch(h_agg_fwd_vec_kernel<NW, BLOCK, UNROLL, true>, blocks, BLOCK, stream, r, pre, o, n_vec, V, divV);
    else
        launch(h_agg_fwd_vec_kernel<NW, BLOCK, UNROLL, false>, blocks, BLOCK, stream, r, pre, o, n_vec, V, divV);
}

// Launch shapes of the vector forward (launch-time only; results do not
// depend on them).  Large calls: 256 threads, 64 bytes of output each
// (2 vectors of 32 bytes or 4 of 16); calls of at most 8 KiB of output per
// SM: 128 threads x 1 vector, to spread a decode-sized call over more SMs.
template <int NW>
void fwd_vec(const void* residual, const float* pre, void* out, uint64_t T, uint64_t H,
             bool pre_vec, cudaStream_t stream) {
    constexpr uint64_t kElemsPerVec = 2 * NW;
    const uint64_t V = H / kElemsPerVec;
    // Vector indices are 32-bit: a call with 2^31 vectors or more runs as
    // several launches over consecutive token ranges.  Tokens are
    // independent, so the bytes are the same as one launch.
    const uint64_t max_tokens = 0x7FFFFFFFull / V;
    const uint64_t small_limit = uint64_t(num_sms()) * (8192 / (4 * NW));
    for (uint64_t t0 = 0; t0 < T; t0 += max_tokens) {
        const uint64_t nt = (T - t0 < max_tokens) ? T - t0 : max_tokens;
        const uint32_t n_vec = uint32_t(nt * V);
        const void* r = static_cast<const char*>(residual) + t0 * 8 * H;
        const float* p = pre + 4 * t0;
        void* o = static_cast<char*>(out) + t0 * 2 * H;
        if (n_vec <= small_limit)
            launch_fwd_vec<NW, 128, 1>(r, p, o, n_vec, uint32_t(V), pre_vec, stream);
        else
            launch_fwd_vec<NW, 256, 16 / NW>(r, p, o, n_vec, uint32_t(V), pre_vec, stream);
    }
}

// Backward vector launch shapes (launch-time only; the sums do not depend on
// them).  A block holds one token; its threads keep BATCH vectors each in
// registers per pass, and the register budget is sized for MIN_BLOCKS blocks
// per SM.  The batch is chosen from the vectors per thread so that a row is
// covered in one pass where possible and each SM keeps roughly 160 KB of loads
// in flight: 32-byte vectors (128 threads) use batch 1 / 2 / 4 with 6 / 3 / 2
// blocks per SM for up to 1 / 2 / more vectors per thread; 16-byte vectors
// (256 threads) use batch 2 with 3 blocks per SM.
template <int NW, int BATCH, int MIN_BLOCKS>
void launch_bwd_vec(const void* g, const void* residual, const float* pre, void* gres, float* gpre,
                    uint64_t T, uint32_t V, cudaStream_t stream) {
    constexpr int kThreads = kLanes / (NW / 4);
    const uint32_t blocks = grid_for(T, 1, uint64_t(num_sms()) * 256);
    const Words<NW>* gv = static_cast<const Words<NW>*>(g);
    const Words<NW>* rv = static_cast<const Words<NW>*>(residual);
    Words<NW>* grv = static_cast<Words<NW>*>(gres);
    if (aligned(pre, 16))
        launch(h_agg_bwd_vec_kernel<NW, BATCH, MIN_BLOCKS, true>, blocks, kThreads, stream, gv, rv, pre, grv,
               gpre, T, V);
    else
        launch(h_agg_bwd_vec_kernel<NW, BATCH, MIN_BLOCKS, false>, blocks, kThreads, stream, gv, rv, pre, grv,
               gpre, T, V);
}

void bwd_vec32(const void* g, const void* residual, const float* pre, void* gres, float* gpre,
               uint64_t T, uint64_t H, cudaStream_t stream) {
    const uint32_t V = uint32_t(H / 16);
    const uint32_t per_thread = (V + 127) / 128;
    if (per_thread <= 1)
        launch_bwd_vec<8, 1, 6>(g, residual, pre, gres, gpre, T, V, stream);
    else if (per_thread == 2)
        launch_bwd_vec<8, 2, 3>(g, residual, pre, gres, gpre, T, V, stream);
    else
        launch_bwd_vec<8, 4, 2>(g, residual, pre, gres, gpre, T, V, stream);
}

void bwd_vec16(const void* g, const void* residual, const float* pre, void* gres, float* gpre,
               uint64_t T, uint64_t H, cudaStream_t stream) {
    launch_bwd_vec<4, 2, 3>(g, residual, pre, gres, gpre, T, uint32_t(H / 8), stream);
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
        case MHC_ERR_INVALID_ARG: return "MHC_ERR_INVALID_ARG: bad size, null, misaligned or overlapping buffer";
        case MHC_ERR_UNSUPPORTED: return "MHC_ERR_UNSUPPORTED: H too large for the 32-bit row index";
        case MHC_ERR_CUDA: return "MHC_ERR_CUDA: kernel launch failed (see mhc_h_aggregate_last_cuda_error)";
    }
    return "unknown mhc_status_t";
}

int32_t mhc_h_aggregate_last_cuda_error(void) { return g_last_cuda_error; }

mhc_path_t mhc_h_aggregate_fwd_path(const void* residual, const float* pre, const void* out,
                                    int64_t T, int64_t H) {
    return fwd_path(residual, pre, out, T, H);
}

mhc_path_t mhc_h_aggregate_bwd_path(const void* grad_out, const void* residual, const float* pre,
                                    const void* grad_residual, const float* grad_pre, int64_t T,
                                    int64_t H) {
    return bwd_path(grad_out, residual, pre, grad_residual, grad_pre, T, H);
}

mhc_status_t mhc_h_aggregate_fwd(const void* residual, const float* pre, void* out, int64_t T,
                                 int64_t H, mhc_stream_t stream_) {
    if (!sizes_ok(T, H)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    const mhc_path_t path = fwd_path(residual, pre, out, T, H);
    if (path == MHC_PATH_NONE) return MHC_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    begin_launches();
    const bool pre_vec = aligned(pre, 16);
    const uint64_t cap = uint64_t(num_sms()) * 1024;
    if ((path == MHC_PATH_VEC32 || path == MHC_PATH_VEC16) && uint64_t(H) / 8 > 0x7FFFFFFFull)
        return MHC_ERR_UNSUPPORTED;

    if (path == MHC_PATH_VEC32) {
        fwd_vec<8>(residual, pre, out, uint64_t(T), uint64_t(H), pre_vec, stream);
    } else if (path == MHC_PATH_VEC16) {
        fwd_vec<4>(residual, pre, out, uint64_t(T), uint64_t(H), pre_vec, stream);
    } else if (path == MHC_PATH_PAIR) {
        const uint64_t P = uint64_t(H) / 2;
        const uint64_t n = uint64_t(T) * P;
        launch(h_agg_fwd_pair_kernel, grid_for(n, 256, cap), 256, stream,
               static_cast<const uint32_t*>(residual), pre, static_cast<uint32_t*>(out), n, P);
    } else {
        const uint64_t n = uint64_t(T) * uint64_t(H);
        launch(h_agg_fwd_element_kernel, grid_for(n, 256, cap), 256, stream,
               static_cast<const uint16_t*>(residual), pre, static_cast<uint16_t*>(out), n, uint64_t(H));
    }
    return finish_launch();
}

mhc_status_t mhc_h_aggregate_bwd(const void* grad_out, const void* residual, const float* pre,
                                 void* grad_residual, float* grad_pre, int64_t T, int64_t H,
                                 mhc_stream_t stream_) {
    if (!sizes_ok(T, H)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    const mhc_path_t path = bwd_path(grad_out, residual, pre, grad_residual, grad_pre, T, H);
    if (path == MHC_PATH_NONE) return MHC_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if ((path == MHC_PATH_VEC32 || path == MHC_PATH_VEC16) && uint64_t(H) / 8 > 0xFFFFFFFFull)
        return MHC_ERR_UNSUPPORTED;
    begin_launches();

    if (path == MHC_PATH_VEC32) {
        bwd_vec32(grad_out, residual, pre, grad_residual, grad_pre, uint64_t(T), uint64_t(H), stream);
    } else if (path == MHC_PATH_VEC16) {
        bwd_vec16(grad_out, residual, pre, grad_residual, grad_pre, uint64_t(T), uint64_t(H), stream);
    } else {
        const uint32_t blocks = grid_for(uint64_t(T), 1, uint64_t(num_sms()) * 256);
        launch(h_agg_bwd_element_kernel, blocks, kLanes, stream, static_cast<const uint16_t*>(grad_out),
               static_cast<const uint16_t*>(residual), pre, static_cast<uint16_t*>(grad_residual), grad_pre,
               uint64_t(T), uint64_t(H));
    }
    return finish_launch();
}

}  // extern "C"
