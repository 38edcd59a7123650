// Device code of the mHC "H Aggregate" library for GB300 (sm_103a): the
// forward and fused backward kernels, templated on the stream count N, the
// storage type DT and the access width.
//
// Source: "Add batch-invariant h_aggregate kernel" (RL-Kernel pull request
// 366).  Summary: residual [T,4,H] BF16, pre [T,4] FP32, out [T,H] BF16,
//   out = bf16((pre0*r0 + pre1*r1) + (pre2*r2 + pre3*r3)).
// Batch invariance: one writer per output, no atomics, FP32 __fmul_rn /
// __fadd_rn in the fixed (0 + 1) + (2 + 3) tree; inputs widened exactly,
// one rounding to BF16 per output.
// The backward answers that page's reviewer request; its formula is the exact
// derivative of the Summary formula and its grad_pre order (ORDER-256) is
// defined in mhc_h_aggregate.h.  N = 4 with BF16 storage is the pages' op;
// N in {1, 2, 8} (balanced pairwise tree) and FP16 storage are this library's
// widening of it, keeping every rule above.
//
// Design (GB300, HBM-bound: about 0.7 FP32 operations per byte moved):
//  * Vector paths move NW 32-bit words per access: NW = 8 uses the 256-bit
//    (32-byte) global loads and stores that sm_100-class GPUs added
//    (ld/st .v8.b32), NW = 4 the 16-byte ones.  One access covers 2*NW
//    stored values, i.e. NW/4 "chunks" of 8 values.
//  * Forward: a flat grid over output vectors.  A thread loads the N residual
//    vectors feeding its output vector with streaming loads and the token's
//    pre, and stores one vector.  Large calls give each thread UNROLL
//    vectors, all loads issued before any arithmetic, to keep enough bytes
//    in flight per SM; decode-sized calls give each thread one vector so the
//    work spreads over as many SMs as possible.  The arithmetic of an element
//    never depends on the grid, the block or T.
//  * Backward: one block per token (grid-stride over tokens) whose threads
//    own the 256 lanes of ORDER-256, NW/4 lanes each: thread j holds the
//    chunks of lanes (NW/4)*j .. (NW/4)*j + NW/4 - 1, which are adjacent, so
//    one vector access serves all of them.  It streams g and the N residual
//    rows, writes grad_residual, and adds the chunk partials of each lane in
//    increasing chunk order.  Groups of 32 lanes fold with warp shuffles (and
//    one in-thread add when a thread holds two lanes), the 8 groups through
//    shared memory.  No atomics, no cross-block traffic.
//  * Narrower paths (H not a multiple of 8, or buffers not 16-byte aligned)
//    run the same per-element arithmetic and the same grad_pre tree: even H
//    with 4-byte-aligned buffers with 4-byte coalesced accesses (the backward
//    stages row segments in shared memory so that each lane still sees its
//    own 8-value chunks), other rows of H >= 64 (odd H) with aligned 16-byte
//    accesses realigned in registers (mhc_shift.cuh), and short rows with
//    2-byte accesses.  Every path gives the same bytes.
//  * Every kernel is launched with programmatic stream serialization and
//    waits for its predecessor before touching memory (pdl_enter).
//  * No tensor cores: nothing here is a contraction.
//  * Built without fast math, with --fmad=false and -ftz=false; the
//    intrinsics below already forbid contraction and flushing.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "fastdiv.cuh"
#include "mhc_coeffs.cuh"

namespace mhc {

constexpr int kBF16 = 0;
constexpr int kF16 = 1;

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
// storage <-> FP32: BF16 widening is exact (the pattern is the upper half of
// the binary32 one), binary16 widening is exact too (cvt.f32.f16); narrowing
// rounds to nearest even in both.
// --------------------------------------------------------------------------

template <int DT>
struct Elem;

template <>
struct Elem<kBF16> {
    static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
    static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
    static __device__ __forceinline__ float one(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    static __device__ __forceinline__ uint16_t cvt(float x) {
        __nv_bfloat16 v = __float2bfloat16_rn(x);
        return *reinterpret_cast<uint16_t*>(&v);
    }
};

template <>
struct Elem<kF16> {
    static __device__ __forceinline__ float lo(uint32_t w) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
    }
    static __device__ __forceinline__ float hi(uint32_t w) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
    }
    static __device__ __forceinline__ float one(uint16_t b) { return __half2float(__ushort_as_half(b)); }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    static __device__ __forceinline__ uint16_t cvt(float x) { return __half_as_ushort(__float2half_rn(x)); }
};

// --------------------------------------------------------------------------
// the forward element: N RN products and the balanced pairwise tree of RN
// sums (N = 4: (p0 + p1) + (p2 + p3))
// --------------------------------------------------------------------------

template <int N>
__device__ __forceinline__ float tree_sum(float (&p)[N]) {
#pragma unroll
    for (int width = N; width > 1; width /= 2) {
#pragma unroll
        for (int i = 0; i < width / 2; ++i) p[i] = __fadd_rn(p[2 * i], p[2 * i + 1]);
    }
    return p[0];
}

// Two adjacent elements held as a pair in word `e` of each of the N inputs.
template <int N, int DT>
__device__ __forceinline__ uint32_t agg_pair(const float (&pre)[N], const uint32_t (&w)[N]) {
    float lo[N], hi[N];
#pragma unroll
    for (int k = 0; k < N; ++k) {
        lo[k] = __fmul_rn(pre[k], Elem<DT>::lo(w[k]));
        hi[k] = __fmul_rn(pre[k], Elem<DT>::hi(w[k]));
    }
    return Elem<DT>::pack(tree_sum<N>(lo), tree_sum<N>(hi));
}

// --------------------------------------------------------------------------
// forward kernels
// --------------------------------------------------------------------------

// Vector path.  Output vector i (i = t*V + v, V = H / (2*NW) vectors per row)
// is out[i]; the residual vector of row k is res[t*N*V + k*V + v] =
// res[i + (N-1)tV + kV].
template <int N, int DT, int NW, int BLOCK, int UNROLL, class Coeffs>
__global__ void __launch_bounds__(BLOCK)
agg_fwd_vec_kernel(const Words<NW>* __restrict__ res, Coeffs coeffs, Words<NW>* __restrict__ out,
                   uint32_t n_vec, uint32_t V, FastDivU32 divV) {
    pdl_enter();
    const uint32_t first = blockIdx.x * uint32_t(BLOCK * UNROLL) + threadIdx.x;
    Words<NW> r[UNROLL][N];
    float p[UNROLL][N];
    uint32_t tok[UNROLL];
    // kBlockTable: the coefficients of the (at most BLOCK*UNROLL + 1) tokens
    // the block touches, each computed once, by the first threads, before
    // their residual loads (the sigmoid's temporaries and the loaded vectors
    // are then never live together, which keeps the register count, and so
    // the occupancy, of the plain kernel).
    __shared__ float table[Coeffs::kBlockTable ? (BLOCK * UNROLL + 1) * N : 1];
    uint32_t t0 = 0;
    if constexpr (Coeffs::kBlockTable) {
        const uint32_t b0 = blockIdx.x * uint32_t(BLOCK * UNROLL);
        const uint32_t b1 = min(b0 + uint32_t(BLOCK * UNROLL), n_vec) - 1;
        t0 = fastdiv_u32(b0, divV);
        const uint32_t count = (fastdiv_u32(b1, divV) - t0 + 1) * uint32_t(N);
        for (uint32_t j = threadIdx.x; j < count; j += BLOCK)
            table[j] = coeffs.pre_from(coeffs.mix_at(uint64_t(t0) * N + j), int(j % N));
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const uint32_t i = first + uint32_t(u * BLOCK);
        if (i < n_vec) {
            const uint32_t t = fastdiv_u32(i, divV);
            tok[u] = t;
            const Words<NW>* src = res + (uint64_t(i) + uint64_t(N - 1) * uint64_t(t) * V);
#pragma unroll
            for (int k = 0; k < N; ++k) r[u][k] = ld_stream<NW>(src + uint64_t(k) * V);
            if constexpr (!Coeffs::kBlockTable) coeffs.template load<N>(t, p[u]);
        }
    }
    if constexpr (Coeffs::kBlockTable) {
        __syncthreads();
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (first + uint32_t(u * BLOCK) < n_vec) {
#pragma unroll
                for (int k = 0; k < N; ++k) p[u][k] = table[(tok[u] - t0) * N + k];
            }
        }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const uint32_t i = first + uint32_t(u * BLOCK);
        if (i < n_vec) {
            if constexpr (!Coeffs::kBlockTable) coeffs.template to_pre<N>(p[u]);
            Words<NW> o;
#pragma unroll
            for (int e = 0; e < NW; ++e) {
                uint32_t w[N];
#pragma unroll
                for (int k = 0; k < N; ++k) w[k] = r[u][k].w[e];
                o.w[e] = agg_pair<N, DT>(p[u], w);
            }
            st_stream<NW>(out + i, o);
        }
    }
}

// Narrow forward paths: a 2-D grid of (row segment, token) blocks, grid-stride
// over tokens.  A block of 256 threads covers 2048 units of one output row
// (unit = a 4-byte pair of values when H is even and the buffers are 4-byte
// aligned, else one 2-byte value); thread j takes units e*256 + j (e < 8), so
// consecutive threads touch consecutive units (coalesced), and all its loads
// are issued before any arithmetic.  The token's pre is loaded once.
constexpr int kNarrowBlock = 256;
constexpr int kNarrowPerThread = 8;
constexpr int kNarrowSeg = kNarrowBlock * kNarrowPerThread;

// Token t's pre in p, for a block whose threads all run the same token loop,
// once the token's loads are issued.  With a block table, threads 0..N-1
// compute the N values into table[parity] and the block reads them after a
// barrier (the two halves alternate, so one barrier per token suffices);
// otherwise every thread finishes what load() fetched.
template <int N, class Coeffs>
__device__ __forceinline__ void token_pre(const Coeffs& coeffs, uint64_t t, float (&p)[N],
                                          float (*table)[N], int& parity) {
    if constexpr (Coeffs::kBlockTable) {
        if (threadIdx.x < N)
            table[parity][threadIdx.x] =
                coeffs.pre_from(coeffs.mix_at(uint64_t(N) * t + threadIdx.x), int(threadIdx.x));
        __syncthreads();
#pragma unroll
        for (int k = 0; k < N; ++k) p[k] = table[parity][k];
        parity ^= 1;
    } else {
        coeffs.template to_pre<N>(p);
    }
}

// 4-byte path: P = H/2 pairs per row.
template <int N, int DT, class Coeffs>
__global__ void __launch_bounds__(kNarrowBlock)
agg_fwd_pair_kernel(const uint32_t* __restrict__ res2, Coeffs coeffs, uint32_t* __restrict__ out2,
                    uint64_t T, uint64_t P) {
    __shared__ float table[2][N];   // kBlockTable: the token's pre, by loop parity
    pdl_enter();
    const uint64_t base = uint64_t(blockIdx.x) * kNarrowSeg + threadIdx.x;
    int parity = 0;
    for (uint64_t t = blockIdx.y; t < T; t += gridDim.y) {
        float p[N];
        if constexpr (!Coeffs::kBlockTable) coeffs.template load<N>(t, p);
        const uint32_t* src = res2 + uint64_t(N) * t * P;
        uint32_t w[kNarrowPerThread][N];
#pragma unroll
        for (int e = 0; e < kNarrowPerThread; ++e) {
            const uint64_t c = base + uint64_t(e) * kNarrowBlock;
            if (c < P) {
#pragma unroll
                for (int k = 0; k < N; ++k) w[e][k] = ld_stream4(src + uint64_t(k) * P + c);
            }
        }
        token_pre<N>(coeffs, t, p, table, parity);
#pragma unroll
        for (int e = 0; e < kNarrowPerThread; ++e) {
            const uint64_t c = base + uint64_t(e) * kNarrowBlock;
            if (c < P) st_stream4(out2 + t * P + c, agg_pair<N, DT>(p, w[e]));
        }
    }
}

// 2-byte path: any H and any 2-byte alignment.
template <int N, int DT, class Coeffs>
__global__ void __launch_bounds__(kNarrowBlock)
agg_fwd_element_kernel(const uint16_t* __restrict__ res, Coeffs coeffs, uint16_t* __restrict__ out,
                       uint64_t T, uint64_t H) {
    __shared__ float table[2][N];
    pdl_enter();
    const uint64_t base = uint64_t(blockIdx.x) * kNarrowSeg + threadIdx.x;
    int parity = 0;
    for (uint64_t t = blockIdx.y; t < T; t += gridDim.y) {
        float p[N];
        if constexpr (!Coeffs::kBlockTable) coeffs.template load<N>(t, p);
        const uint16_t* src = res + uint64_t(N) * t * H;
        uint16_t v[kNarrowPerThread][N];
#pragma unroll
        for (int e = 0; e < kNarrowPerThread; ++e) {
            const uint64_t h = base + uint64_t(e) * kNarrowBlock;
            if (h < H) {
#pragma unroll
                for (int k = 0; k < N; ++k) v[e][k] = ld_stream2(src + uint64_t(k) * H + h);
            }
        }
        token_pre<N>(coeffs, t, p, table, parity);
#pragma unroll
        for (int e = 0; e < kNarrowPerThread; ++e) {
            const uint64_t h = base + uint64_t(e) * kNarrowBlock;
            if (h < H) {
                float q[N];
#pragma unroll
                for (int k = 0; k < N; ++k) q[k] = __fmul_rn(p[k], Elem<DT>::one(v[e][k]));
                st_stream2(out + t * H + h, Elem<DT>::cvt(tree_sum<N>(q)));
            }
        }
    }
}

// --------------------------------------------------------------------------
// backward
// --------------------------------------------------------------------------

constexpr int kLanes = 256;   // lanes of ORDER-256
constexpr int kGroups = 8;    // groups of 32 lanes

// grad_residual for two adjacent elements: cvt(RN(pre_k * g)).
template <int DT>
__device__ __forceinline__ uint32_t scale_pair(float pk, uint32_t gw) {
    return Elem<DT>::pack(__fmul_rn(pk, Elem<DT>::lo(gw)), __fmul_rn(pk, Elem<DT>::hi(gw)));
}

template <int DT, int NW>
__device__ __forceinline__ Words<NW> scale_vec(float pk, const Words<NW>& g) {
    Words<NW> o;
#pragma unroll
    for (int e = 0; e < NW; ++e) o.w[e] = scale_pair<DT>(pk, g.w[e]);
    return o;
}

// ((q0+q1)+(q2+q3)) + ((q4+q5)+(q6+q7)) of q_e = g_e * r_e (exact products)
// for the chunk held in words w0 .. w0+3 of g and r.
template <int DT, int NW>
__device__ __forceinline__ float chunk_partial(const Words<NW>& g, const Words<NW>& r, int w0) {
    float q[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        q[2 * i] = __fmul_rn(Elem<DT>::lo(g.w[w0 + i]), Elem<DT>::lo(r.w[w0 + i]));
        q[2 * i + 1] = __fmul_rn(Elem<DT>::hi(g.w[w0 + i]), Elem<DT>::hi(r.w[w0 + i]));
    }
    return __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                     __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
}

// Steps 4 and 5 of ORDER-256 for a block of 256/LPT threads, thread j holding
// lanes LPT*j + l (l < LPT) in acc[l][k].  A group of 32 lanes is 32/LPT
// adjacent threads: lane strides 16 .. LPT are thread strides 16/LPT .. 1
// (xor shuffles), lane stride 1 (when LPT == 2) is the add of a thread's own
// two lanes.  The 8 group values then fold with strides 4, 2, 1 in shared
// memory, and grad_pre[t, 0..N-1] goes to the coefficient source (which
// stores it, or the gradients derived from it).  All threads of the block call it.
//
// A block of fewer than 256/LPT threads (`groups` groups of 32 lanes) stands
// for the full 256 lanes whose higher lanes hold +0: their group values are
// +0 in the cross-group fold.  `sync` is the barrier over the folding
// threads (the whole block, or the consumer threads of a block with a
// producer warp), and `tid` the thread's index among them (threadIdx.x if
// negative).
// The barrier of the threads that fold a token's lane sums or share its
// shared-memory tables: the whole block, or (bulk-copy kernels) its consumer
// threads.
struct BlockSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

template <int N, int LPT, class Coeffs, class Sync = BlockSync>
__device__ __forceinline__ void fold_lanes_and_store(float (&acc)[LPT][N], float (*red)[N],
                                                     const Coeffs& coeffs, uint64_t t,
                                                     const float* slope, int groups = kGroups,
                                                     Sync sync = Sync{}, int tid = -1) {
    const int x = tid < 0 ? int(threadIdx.x) : tid;   // the thread's index among the folding threads
    constexpr int kThreadsPerGroup = 32 / LPT;
#pragma unroll
    for (int k = 0; k < N; ++k) {
#pragma unroll
        for (int s = kThreadsPerGroup / 2; s >= 1; s >>= 1) {
#pragma unroll
            for (int l = 0; l < LPT; ++l)
                acc[l][k] = __fadd_rn(acc[l][k], __shfl_xor_sync(0xffffffffu, acc[l][k], s));
        }
        if (LPT == 2) acc[0][k] = __fadd_rn(acc[0][k], acc[LPT - 1][k]);
    }
    if ((x % kThreadsPerGroup) == 0) {
#pragma unroll
        for (int k = 0; k < N; ++k) red[x / kThreadsPerGroup][k] = acc[0][k];
    }
    sync();
    if (x < N) {
        const int k = x;
        float w[kGroups];
#pragma unroll
        for (int i = 0; i < kGroups; ++i) w[i] = (i < groups) ? red[i][k] : 0.0f;
#pragma unroll
        for (int s = kGroups / 2; s >= 1; s >>= 1) {
#pragma unroll
            for (int i = 0; i < s; ++i) w[i] = __fadd_rn(w[i], w[i + s]);
        }
        if constexpr (Coeffs::kBlockTable) {
            coeffs.template store_grad_slope<N>(t, k, w[0], slope[k]);
        } else {
            coeffs.template store_grad<N>(t, k, w[0]);
        }
    }
    sync();  // red[] (and the slope table) are reused by the next token of this block
}

// Vector path: H % (2*NW) == 0 and g / residual / grad_residual aligned to
// 4*NW bytes.  V = H / (2*NW) vectors per row; thread j handles vectors
// j, j + B, j + 2B, ... (B = 256/LPT threads), i.e. for lane LPT*j + l the
// chunks LPT*(j + mB) + l = (LPT*j + l) + 256m: exactly that lane's chunks,
// in increasing order.  Up to BATCH vectors per thread are held in registers
// per pass.
template <int N, int DT, int NW, int BATCH, int MIN_BLOCKS, class Coeffs>
__global__ void __launch_bounds__(kLanes / (NW / 4), MIN_BLOCKS)
agg_bwd_vec_kernel(const Words<NW>* __restrict__ g, const Words<NW>* __restrict__ res,
                   Coeffs coeffs, Words<NW>* __restrict__ gres, uint64_t T, uint32_t V) {
    constexpr int LPT = NW / 4;
    constexpr uint32_t B = kLanes / LPT;
    __shared__ float red[kGroups][N];
    __shared__ float table[N];   // kBlockTable: the token's pre ...
    __shared__ float slope[N];   // ... and sigmoid' (for the epilogue)
    pdl_enter();
    const uint32_t j = threadIdx.x;
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
        float pk[N];
        float m_own = 0.0f;   // kBlockTable: thread j < N fetches mix[t, j] first
        if constexpr (Coeffs::kBlockTable) {
            if (j < N) m_own = coeffs.mix_at(uint64_t(N) * t + j);
        } else {
            coeffs.template load<N>(t, pk);
        }
        bool pk_ready = false;
        const Words<NW>* gt = g + t * V;
        const Words<NW>* rt = res + uint64_t(N) * t * V;
        Words<NW>* grt = gres + uint64_t(N) * t * V;
        float acc[LPT][N];
#pragma unroll
        for (int l = 0; l < LPT; ++l)
#pragma unroll
            for (int k = 0; k < N; ++k) acc[l][k] = 0.0f;
        // With a block table the first pass runs in every thread (its loads
        // are guarded), so that all of them meet the barrier that publishes
        // the table; the fold's barriers keep the table until the next token.
        for (uint32_t v0 = j; Coeffs::kBlockTable ? (v0 < V || !pk_ready) : (v0 < V);
             v0 += B * BATCH) {
            Words<NW> gv[BATCH];
            Words<NW> rv[BATCH][N];
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const uint32_t v = v0 + uint32_t(b) * B;
                if (v < V) {
                    gv[b] = ld_stream<NW>(gt + v);
#pragma unroll
                    for (int k = 0; k < N; ++k) rv[b][k] = ld_stream<NW>(rt + uint64_t(k) * V + v);
                }
            }
            if (!pk_ready) {
                if constexpr (Coeffs::kBlockTable) {
                    if (j < N) coeffs.pre_and_slope(m_own, int(j), table[j], slope[j]);
                    __syncthreads();
#pragma unroll
                    for (int k = 0; k < N; ++k) pk[k] = table[k];
                } else {
                    coeffs.template to_pre<N>(pk);
                }
                pk_ready = true;
            }
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const uint32_t v = v0 + uint32_t(b) * B;
                if (v < V) {
#pragma unroll
                    for (int k = 0; k < N; ++k) {
                        st_stream<NW>(grt + uint64_t(k) * V + v, scale_vec<DT, NW>(pk[k], gv[b]));
#pragma unroll
                        for (int l = 0; l < LPT; ++l)
                            acc[l][k] = __fadd_rn(acc[l][k], chunk_partial<DT, NW>(gv[b], rv[b][k], 4 * l));
                    }
                }
            }
        }
        fold_lanes_and_store<N, LPT>(acc, red, coeffs, t, slope, int(blockDim.x * LPT / 32));
    }
}

// Narrow backward paths: any H; same lanes, chunks and tree.  256 threads,
// one lane each.  A token's rows are processed in segments of 2048 values =
// 256 chunks, so segment m holds exactly chunk 256m + j of lane j.  Each
// segment of g and of the N residual rows is loaded with coalesced accesses
// into shared memory (values past H are +0), lane j reads its chunk there,
// adds its partial and writes its grad_residual chunk back in place, and the
// segment's grad_residual rows are then stored with coalesced accesses.
// PAIRS: 4-byte accesses (H even, buffers 4-byte aligned); else 2-byte.
template <int N, int DT, bool PAIRS, class Coeffs>
__global__ void __launch_bounds__(kLanes)
agg_bwd_staged_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ res,
                      Coeffs coeffs, uint16_t* __restrict__ gres, uint64_t T, uint64_t H) {
    constexpr int kSeg = 8 * kLanes;                 // values per segment
    constexpr int kUnit = PAIRS ? 2 : 1;             // values per access
    constexpr int kPer = kSeg / (kUnit * kLanes);    // accesses per thread per row
    __shared__ float red[kGroups][N];
    __shared__ float table[N];   // kBlockTable: the token's pre ...
    __shared__ float slope[N];   // ... and sigmoid' (for the epilogue)
    __shared__ __align__(16) uint16_t sg[kSeg];
    __shared__ __align__(16) uint16_t sr[N][kSeg];
    pdl_enter();
    const uint32_t j = threadIdx.x;
    const uint64_t C = (H + 7) / 8;
    const uint64_t U = H / kUnit;                    // units per row
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
        float pk[N];
        float m_own = 0.0f;   // kBlockTable: thread j < N fetches mix[t, j] first
        if constexpr (Coeffs::kBlockTable) {
            if (j < N) m_own = coeffs.mix_at(uint64_t(N) * t + j);
        } else {
            coeffs.template load<N>(t, pk);
        }
        bool pk_ready = false;
        const uint16_t* gt = g + t * H;
        const uint16_t* rt = res + uint64_t(N) * t * H;
        uint16_t* grt = gres + uint64_t(N) * t * H;
        float acc[1][N];
#pragma unroll
        for (int k = 0; k < N; ++k) acc[0][k] = 0.0f;
        for (uint64_t base = 0; base < H; base += kSeg) {
            const uint64_t ubase = base / kUnit;
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const uint32_t s = e * kLanes + j;   // unit index within the segment
                const uint64_t u = ubase + s;
                if (PAIRS) {
                    reinterpret_cast<uint32_t*>(sg)[s] =
                        (u < U) ? ld_stream4(reinterpret_cast<const uint32_t*>(gt) + u) : 0u;
#pragma unroll
                    for (int k = 0; k < N; ++k)
                        reinterpret_cast<uint32_t*>(sr[k])[s] =
                            (u < U) ? ld_stream4(reinterpret_cast<const uint32_t*>(rt + uint64_t(k) * H) + u) : 0u;
                } else {
                    sg[s] = (u < U) ? ld_stream2(gt + u) : uint16_t(0);
#pragma unroll
                    for (int k = 0; k < N; ++k)
                        sr[k][s] = (u < U) ? ld_stream2(rt + uint64_t(k) * H + u) : uint16_t(0);
                }
            }
            if constexpr (Coeffs::kBlockTable) {
                if (!pk_ready && j < N) coeffs.pre_and_slope(m_own, int(j), table[j], slope[j]);
            }
            __syncthreads();
            if (!pk_ready) {
                if constexpr (Coeffs::kBlockTable) {
#pragma unroll
                    for (int k = 0; k < N; ++k) pk[k] = table[k];
                } else {
                    coeffs.template to_pre<N>(pk);
                }
                pk_ready = true;
            }
            if (base / 8 + j < C) {
                Words<4> gv;
                *reinterpret_cast<uint4*>(gv.w) = *reinterpret_cast<const uint4*>(sg + 8 * j);
#pragma unroll
                for (int k = 0; k < N; ++k) {
                    Words<4> rv;
                    *reinterpret_cast<uint4*>(rv.w) = *reinterpret_cast<const uint4*>(&sr[k][8 * j]);
                    acc[0][k] = __fadd_rn(acc[0][k], chunk_partial<DT, 4>(gv, rv, 0));
                    const Words<4> o = scale_vec<DT, 4>(pk[k], gv);
                    *reinterpret_cast<uint4*>(&sr[k][8 * j]) = *reinterpret_cast<const uint4*>(o.w);
                }
            }
            __syncthreads();
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const uint32_t s = e * kLanes + j;
                const uint64_t u = ubase + s;
                if (u < U) {
#pragma unroll
                    for (int k = 0; k < N; ++k) {
                        if (PAIRS)
                            st_stream4(reinterpret_cast<uint32_t*>(grt + uint64_t(k) * H) + u,
                                       reinterpret_cast<const uint32_t*>(sr[k])[s]);
                        else
                            st_stream2(grt + uint64_t(k) * H + u, sr[k][s]);
                    }
                }
            }
            __syncthreads();  // the next segment overwrites the staging buffers
        }
        fold_lanes_and_store<N, 1>(acc, red, coeffs, t, slope);
    }
}

// --------------------------------------------------------------------------
// the pre coefficients on their own, and the gradients of alpha and b
// --------------------------------------------------------------------------

// pre[i] = sigmoid(alpha * mix[i] + b[i mod N]) over the T*N values (flat,
// grid-stride; the same binary32 sequence as the fused kernels).
constexpr int kCoeffBlock = 256;

template <int N>
__global__ void __launch_bounds__(kCoeffBlock)
pre_sigmoid_kernel(const float* __restrict__ mix, const float* __restrict__ alpha,
                   const float* __restrict__ b, float* __restrict__ pre, uint64_t count) {
    pdl_enter();
    const float a = __ldg(alpha);
    const uint64_t stride = uint64_t(gridDim.x) * kCoeffBlock;
    for (uint64_t i = uint64_t(blockIdx.x) * kCoeffBlock + threadIdx.x; i < count; i += stride) {
        float s, one_minus;
        sigmoid32(pre_activation(a, __ldg(mix + i), __ldg(b + (i % N))), s, one_minus);
        pre[i] = s;
    }
}

// Thread-block cluster helpers (inline PTX): this CTA's rank in its cluster,
// the cluster-wide barrier (release / acquire: shared-memory writes made
// before it, to any CTA of the cluster, are visible after it), and a store
// into another CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_shared_cluster(const float* local, uint32_t rank, float v) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" : : "r"(remote), "f"(v) : "memory");
}

// grad_b[k] = sum over t of grad_z[t,k] and grad_alpha = sum over t of
// tree_N(grad_z[t,k] * mix[t,k]), both in ORDER-256 with tokens in place of h:
// chunk c = tokens 8c .. 8c+7 (+0 past T) summed by the chunk tree; lane j
// adds the partials of chunks j, j + 256, ... in increasing order from +0;
// groups of 32 lanes fold with strides 16 .. 1, the 8 groups with 4, 2, 1.
//
// One cluster of 8 CTAs, CTA w owning the lanes 32w .. 32w+31 of group w: its
// chunks are 256m + 32w + i (i < 32), i.e. the 256 consecutive tokens
// 8(256m + 32w) .. + 255 of every "m-block" m.  Each round, warp q of the CTA
// takes m-block m0 + q: lane l loads tokens 32e + l (e < 8) of it (32
// consecutive rows per warp load), and xor shuffles over 8 lanes build the
// chunk trees, leaving chunk 4e + l/8 in lane l (l % 8 == 0); the partials
// go to shared memory, and warp 0, lane i, adds those of chunk i for the
// round's m-blocks in increasing m.  Warp 0 then folds the group with xor
// shuffles, lane 0 stores the group value into CTA 0's shared memory, and
// after a cluster barrier CTA 0 folds the 8 group values and writes the
// result.  No global scratch, no atomics; the exchange uses two hardware
// cluster barriers (all 8 CTAs are resident together by construction).
constexpr int kParamClusterCtas = kGroups;   // 8
constexpr int kParamWarps = 8;
constexpr int kParamThreads = 32 * kParamWarps;

template <int N>
__global__ void __launch_bounds__(kParamThreads)
sigmoid_param_grad_kernel(const float* __restrict__ grad_z, const float* __restrict__ mix,
                          float* __restrict__ grad_b, float* __restrict__ grad_alpha, uint64_t T,
                          bool vec) {
    constexpr int M = N + 1;   // grad_b[0 .. N-1], grad_alpha
    __shared__ float part[kParamWarps][32][M];
    __shared__ float groups[kParamClusterCtas][M];   // used in CTA 0
    pdl_enter();
    const uint32_t w = cluster_rank();
    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint64_t n_mblocks = ((T + 7) / 8 + 255) / 256;
    float acc[M];
#pragma unroll
    for (int k = 0; k < M; ++k) acc[k] = 0.0f;
    for (uint64_t m0 = 0; m0 < n_mblocks; m0 += kParamWarps) {
        const uint64_t m = m0 + warp;
        const uint64_t tbase = 8 * (256 * m + 32 * uint64_t(w));
        float gz[8][N], mx[8][N];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint64_t t = tbase + 32 * e + lane;
            if (m < n_mblocks && t < T) {
                ld_row<N>(grad_z + uint64_t(N) * t, vec, gz[e]);
                ld_row<N>(mix + uint64_t(N) * t, vec, mx[e]);
            } else {
#pragma unroll
                for (int k = 0; k < N; ++k) gz[e][k] = mx[e][k] = 0.0f;
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float v[M];
            float prod[N];
#pragma unroll
            for (int k = 0; k < N; ++k) {
                v[k] = gz[e][k];
                prod[k] = __fmul_rn(gz[e][k], mx[e][k]);
            }
            v[N] = tree_sum<N>(prod);
#pragma unroll
            for (int sh = 1; sh <= 4; sh <<= 1) {
#pragma unroll
                for (int k = 0; k < M; ++k) v[k] = __fadd_rn(v[k], __shfl_xor_sync(0xffffffffu, v[k], sh));
            }
            if ((lane % 8) == 0) {
#pragma unroll
                for (int k = 0; k < M; ++k) part[warp][4 * e + lane / 8][k] = v[k];
            }
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int q = 0; q < kParamWarps; ++q) {
                if (m0 + q < n_mblocks) {
#pragma unroll
                    for (int k = 0; k < M; ++k) acc[k] = __fadd_rn(acc[k], part[q][lane][k]);
                }
            }
        }
        __syncthreads();   // part[] is refilled by the next round
    }
    // every CTA of the cluster is running (and CTA 0's shared memory live)
    // before any of them writes into CTA 0's shared memory
    cluster_barrier();
    if (warp == 0) {
#pragma unroll
        for (int k = 0; k < M; ++k) {
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1)
                acc[k] = __fadd_rn(acc[k], __shfl_xor_sync(0xffffffffu, acc[k], sh));
        }
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < M; ++k) st_shared_cluster(&groups[w][k], 0, acc[k]);
        }
    }
    cluster_barrier();
    if (w == 0 && threadIdx.x < uint32_t(M)) {
        const uint32_t k = threadIdx.x;
        float g[kParamClusterCtas];
#pragma unroll
        for (int i = 0; i < kParamClusterCtas; ++i) g[i] = groups[i][k];
#pragma unroll
        for (int s2 = kParamClusterCtas / 2; s2 >= 1; s2 >>= 1) {
#pragma unroll
            for (int i = 0; i < s2; ++i) g[i] = __fadd_rn(g[i], g[i + s2]);
        }
        if (k < uint32_t(N)) grad_b[k] = g[0];
        else grad_alpha[0] = g[0];
    }
}

}  // namespace mhc

#include "mhc_shift.cuh"
#include "mhc_post.cuh"
#include "mhc_shift_bulk.cuh"
