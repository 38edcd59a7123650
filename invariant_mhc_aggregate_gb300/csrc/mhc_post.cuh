// mHC post: the layer output y expanded back onto the n residual streams,
//
//   out[t,k,h] = cvt( tree_n( res[t,k,j] * x[t,j,h] ) + post[t,k] * y[t,h] )
//
// and its backward
//
//   grad_x[t,j,h]   = cvt( tree_n over k of res[t,k,j] * g[t,k,h] )
//   grad_y[t,h]     = cvt( tree_n over k of post[t,k] * g[t,k,h] )
//   grad_res[t,k,j] = sum over h of g[t,k,h] * x[t,j,h]      (ORDER-256)
//   grad_post[t,k]  = sum over h of g[t,k,h] * y[t,h]        (ORDER-256)
//
// Source: "Add batch-invariant h_aggregate kernel", Summary, names the stage
// ("MHC Post") without defining it; "perf: fuse mHC coefficient backward
// epilogue", Summary, names its post coefficients and the residual-mixing
// (n*n) coefficients.  The formula is this library's reading (the
// hyper-connection update), with the pre aggregate's rules: RN binary32
// products and sums, the balanced pairwise tree over the n mixing terms, the
// post term added last, conversion to the storage type only at the output.
//
// Layout: x, g, out, grad_x [T,n,H]; y, grad_y [T,H]; post, grad_post [T,n];
// res, grad_res [T,n,n] (row k: output stream k, column j: input stream j).
//
// The post coefficients come from a coefficient source (mhc_coeffs.cuh):
// PlainCoeffs reads post and writes grad_post; SigmoidCoeffs computes
// post = sigmoid(alpha * mix + b) in the kernel and writes grad_z and
// grad_mix in place of grad_post.
//
// Kernels (HBM-bound at n <= 4: the forward moves (4n + 2) H bytes a token,
// the backward (6n + 4) H):
//  * forward, 16-byte path: a flat grid over the [T,H] plane, one vector per
//    thread; a thread loads the n x vectors and the y vector of its position
//    and writes the n output vectors (n = 8, rows of 128+ vectors: two
//    threads per position, 4 of its 8 values each).
//  * backward, 16-byte path, n <= 4: the bulk-copy kernel below (rows
//    streamed through a shared-memory ring, one producer warp, 256 consumer
//    lanes); n = 8: the split kernel (the same ring, each lane served by two
//    threads that take half of each chunk's positions).  Either way lane j
//    writes grad_x and grad_y for its chunks and adds their partials to the
//    n*n + n sums, which fold like grad_pre's.
//  * other shapes and alignments: the same arithmetic with 2-byte accesses.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mhc_bulk.cuh"
#include "mhc_f32x2.cuh"

namespace mhc {

// The n*n mixing and n post coefficients of token t, in registers.
template <int N>
__device__ __forceinline__ void ld_post_coeffs(const float* post, const float* res, uint64_t t,
                                               float (&pk)[N], float (&rk)[N][N]) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
        pk[k] = __ldg(post + uint64_t(N) * t + k);
#pragma unroll
        for (int j = 0; j < N; ++j) rk[k][j] = __ldg(res + (uint64_t(N) * t + k) * N + j);
    }
}

// The coefficients of the token a backward block works on (bulk and 2-byte
// kernels).  Up to n = 4 they sit in registers (loaded from global memory,
// or copied from the token table); at n = 8 (72 values, next to 72 lane
// sums) they stay in the token table in shared memory, read where they are
// used.
template <int N, bool kShared = (N >= 8)>
struct PostCoeffs {
    float pk[N], rk[N][N];
    template <class Sync = BlockSync>
    __device__ __forceinline__ void load(const float* post, const float* res, uint64_t t, float*,
                                         Sync = Sync()) {
        ld_post_coeffs<N>(post, res, t, pk, rk);
    }
    // ... or res alone (post set by the caller) ...
    __device__ __forceinline__ void load_res(const float* res, uint64_t t) {
#pragma unroll
        for (int k = 0; k < N; ++k)
#pragma unroll
            for (int j = 0; j < N; ++j) rk[k][j] = __ldg(res + (uint64_t(N) * t + k) * N + j);
    }
    // ... or from a token table in shared memory (post_fill_table)
    __device__ __forceinline__ void from_table(const float* tab) {
#pragma unroll
        for (int k = 0; k < N; ++k) {
            pk[k] = tab[N * N + k];
#pragma unroll
            for (int j = 0; j < N; ++j) rk[k][j] = tab[k * N + j];
        }
    }
    __device__ __forceinline__ float r(int k, int j) const { return rk[k][j]; }
    __device__ __forceinline__ float p(int k) const { return pk[k]; }
};

template <int N>
struct PostCoeffs<N, true> {
    const float* s;   // the token table (post_fill_table): res row-major, then post
    __device__ __forceinline__ void from_table(const float* tab) { s = tab; }
    __device__ __forceinline__ float r(int k, int j) const { return s[k * N + j]; }
    __device__ __forceinline__ float p(int k) const { return s[N * N + k]; }
};

// Token t's table in shared memory, written by threads j < n*n + n of the
// group that shares it: res[t] row-major (n*n), post[t] (n), and, when post
// is computed from the mix (Coeffs::kBlockTable), sigmoid'(z[t]) (n) for the
// backward's epilogue.  Ends with the group's barrier.
template <int N>
constexpr int kPostTable = N * N + 2 * N;

template <int N, class Coeffs, class Sync>
__device__ __forceinline__ void post_fill_table(const Coeffs& c, const float* __restrict__ res, uint64_t t,
                                                uint32_t j, float* tab, Sync sync) {
    if (j < uint32_t(N * N)) {
        tab[j] = __ldg(res + uint64_t(N) * N * t + j);
    } else if (j < uint32_t(N * N + N)) {
        const int k = int(j) - N * N;
        if constexpr (Coeffs::kBlockTable) {
            c.pre_and_slope(c.mix_at(uint64_t(N) * t + k), k, tab[j], tab[j + N]);
        } else {
            tab[j] = __ldg(c.pre + uint64_t(N) * t + k);
        }
    }
    sync();
}

// Token t's coefficients into cf: straight from global memory (post given,
// registers), else through the token table.  Every thread of the group
// calls it; the previous token's readers have passed the fold's closing
// barrier.
template <int N, bool SMEM, class Coeffs, class Sync>
__device__ __forceinline__ void post_load_token(const Coeffs& c, const float* __restrict__ res, uint64_t t,
                                                uint32_t j, float* tab, PostCoeffs<N, SMEM>& cf, Sync sync) {
    if constexpr (Coeffs::kBlockTable || SMEM) {
        post_fill_table<N>(c, res, t, j, tab, sync);
        cf.from_table(tab);
    } else {
        cf.load(c.pre, res, t, tab, sync);
    }
}

// The gradient of post[t,k] (the lane sum w) through the coefficient source:
// grad_post itself, or grad_z and grad_mix with sigmoid'(z[t,k]) = slope[k].
template <int N, class Coeffs>
__device__ __forceinline__ void post_store_grad(const Coeffs& c, uint64_t t, int k, float w, const float* slope) {
    if constexpr (Coeffs::kBlockTable) {
        c.template store_grad_slope<N>(t, k, w, slope[k]);
    } else {
        c.template store_grad<N>(t, k, w);
    }
}

// One output value of stream k from the n input values xs and y, given row
// k of res (rk) and post[t,k] (pk).
template <int N>
__device__ __forceinline__ float post_value(const float (&rk)[N], float pk, const float (&xs)[N], float ys) {
    float p[N];
#pragma unroll
    for (int j = 0; j < N; ++j) p[j] = __fmul_rn(rk[j], xs[j]);
    return __fadd_rn(tree_sum<N>(p), __fmul_rn(pk, ys));
}

// Row k of res for token t (read-only cache: every thread of a token reads
// the same values).
template <int N>
__device__ __forceinline__ void ld_res_row(const float* res, uint64_t t, int k, float (&rk)[N]) {
#pragma unroll
    for (int j = 0; j < N; ++j) rk[j] = __ldg(res + (uint64_t(N) * t + k) * N + j);
}

// --------------------------------------------------------------------------
// forward
// --------------------------------------------------------------------------

constexpr int kPostBlock = 256;

// Vector path: the [T, V] plane of vectors (V = H / (2*NW) per row), block
// b taking vectors b*BLOCK*U + u*BLOCK + threadIdx (u < U): each thread loads
// the n x vectors and the y vector of its U positions, then writes their n
// output vectors.
//
// With post computed from the mix (Coeffs::kBlockTable) the sigmoids are
// evaluated once the thread's own loads are issued: per warp for rows of 32
// vectors or more, else into a block table published by one barrier.
template <int N, int DT, int NW, int U, int MIN_BLOCKS, class Coeffs>
__global__ void __launch_bounds__(kPostBlock, MIN_BLOCKS)
post_fwd_vec_kernel(const Words<NW>* __restrict__ x, const Words<NW>* __restrict__ y, Coeffs coeffs,
                    const float* __restrict__ res, Words<NW>* __restrict__ out, uint32_t n_vec, uint32_t V,
                    FastDivU32 divV) {
    __shared__ float table[Coeffs::kBlockTable ? (kPostBlock * U + 1) * N : 1];
    pdl_enter();
    const uint32_t i0 = blockIdx.x * (kPostBlock * U) + threadIdx.x;
    Words<NW> xv[U][N], yv[U];
    uint32_t tok[U];
    uint64_t row0[U];   // x / out vector of stream 0
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint32_t i = i0 + uint32_t(u) * kPostBlock;
        if (i < n_vec) {
            tok[u] = fastdiv_u32(i, divV);
            row0[u] = uint64_t(N) * tok[u] * V + (i - tok[u] * V);
#pragma unroll
            for (int j = 0; j < N; ++j) xv[u][j] = ld_stream<NW>(x + row0[u] + uint64_t(j) * V);
            yv[u] = ld_stream<NW>(y + i);
        }
    }
    // post from the mix, evaluated while the loads above are in flight: for
    // rows of 32 vectors or more (one vector per thread) a warp spans at most
    // two tokens, whose 2n sigmoids its first lanes evaluate and shuffles
    // hand out, with no barrier; else the block's table and one barrier.
    const bool warp_coeffs = (U == 1) && V >= 32;
    uint32_t t_first = 0;
    float pkw[N];
    if constexpr (Coeffs::kBlockTable) {
        if (warp_coeffs) {
            const uint32_t lane = threadIdx.x & 31u;
            const uint32_t wbase = blockIdx.x * kPostBlock + (threadIdx.x & ~31u);
            uint32_t wt = 0;
            float mine = 0.0f;
            if (wbase < n_vec) {
                wt = fastdiv_u32(wbase, divV);
                const uint32_t tt = wt + lane / N;
                if (lane < uint32_t(2 * N) && uint64_t(tt) * V < n_vec)
                    mine = coeffs.pre_from(coeffs.mix_at(uint64_t(N) * tt + lane % N), int(lane % N));
            }
            const uint32_t sel = (i0 < n_vec) ? tok[0] - wt : 0u;
#pragma unroll
            for (int k = 0; k < N; ++k) pkw[k] = __shfl_sync(0xffffffffu, mine, int(sel) * N + k);
        } else {
            const uint32_t first = blockIdx.x * (kPostBlock * U);
            const uint32_t last =
                (n_vec - first > uint32_t(kPostBlock * U)) ? first + kPostBlock * U - 1 : n_vec - 1;
            t_first = fastdiv_u32(first, divV);
            const uint32_t count = (fastdiv_u32(last, divV) - t_first + 1) * N;
            for (uint32_t q = threadIdx.x; q < count; q += kPostBlock)
                table[q] = coeffs.pre_from(coeffs.mix_at(uint64_t(N) * t_first + q), int(q % N));
            __syncthreads();
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint32_t i = i0 + uint32_t(u) * kPostBlock;
        if (i < n_vec) {
#pragma unroll
            for (int k = 0; k < N; ++k) {
                float rk[N];
                ld_res_row<N>(res, tok[u], k, rk);
                float pk;
                if constexpr (Coeffs::kBlockTable) pk = warp_coeffs ? pkw[k] : table[(tok[u] - t_first) * N + k];
                else pk = __ldg(coeffs.pre + uint64_t(N) * tok[u] + k);
                Words<NW> o;
#pragma unroll
                for (int e = 0; e < NW; ++e) {
                    float xl[N], xh[N];
#pragma unroll
                    for (int j = 0; j < N; ++j) {
                        xl[j] = Elem<DT>::lo(xv[u][j].w[e]);
                        xh[j] = Elem<DT>::hi(xv[u][j].w[e]);
                    }
                    o.w[e] = Elem<DT>::pack(post_value<N>(rk, pk, xl, Elem<DT>::lo(yv[u].w[e])),
                                            post_value<N>(rk, pk, xh, Elem<DT>::hi(yv[u].w[e])));
                }
                st_stream<NW>(out + row0[u] + uint64_t(k) * V, o);
            }
        }
    }
}

// Split forward (n = 8, 16-byte path, rows of at least kSplitFwdVecs
// vectors): two threads per 16-byte position, thread half e taking its
// positions 4e .. 4e + 3 (8 bytes of each of the n x vectors and of y), so
// that a thread's unpacked inputs (4n + 4 values) and one output's
// coefficients fit in few registers and more blocks share an SM: blocks of
// 128 threads (64 positions), 8 per SM at 64 registers (256-thread blocks
// 0.6% slower at T = 4096, H = 7168, 512-thread blocks 12%).  A block's
// positions span at most two tokens (rows of at least 64 vectors), whose
// coefficients (res row-major, then post, computed when post comes from the
// mix) the block puts in a shared table while its loads are in flight: with
// post given, 4-byte asynchronous copies issued before the x loads, so that
// no thread waits for a coefficient before issuing them (169.6 -> 167.8 us);
// with post from the mix, computed after them.  Each output value is
// post_value's: the n-term tree, then the post term.
constexpr int kSplitFwdBlock = 128;
constexpr int kSplitFwdMinBlocks = 8;
constexpr int kSplitFwdVecs = kSplitFwdBlock / 2;

// The 4 values of 8 bytes of a 2-byte row (2 words, low half first).
template <int DT>
__device__ __forceinline__ void unpack_half(uint2 w, float (&f)[4]) {
    f[0] = Elem<DT>::lo(w.x);
    f[1] = Elem<DT>::hi(w.x);
    f[2] = Elem<DT>::lo(w.y);
    f[3] = Elem<DT>::hi(w.y);
}

// An 8-byte streaming store.
__device__ __forceinline__ void st_stream_half(void* p, uint32_t a, uint32_t b) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" : : "l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ uint2 ld_stream_half(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// The block table of the split forward, per token: res[t] row-major (n*n),
// then post[t,k] twice for each k (a packed pair).
template <int N>
constexpr int kSplitFwdTable = N * N + 2 * N;

template <int N, int DT, int MIN_BLOCKS, class Coeffs>
__global__ void __launch_bounds__(kSplitFwdBlock, MIN_BLOCKS)
post_fwd_split_kernel(const Words<4>* __restrict__ x, const Words<4>* __restrict__ y, Coeffs coeffs,
                      const float* __restrict__ res, Words<4>* __restrict__ out, uint32_t n_vec, uint32_t V,
                      FastDivU32 divV) {
    static_assert(N == 8, "the packed split forward is written for n = 8");
    constexpr int M = kSplitFwdTable<N>;
    constexpr int JP = N / 2;   // input stream pairs
    __shared__ __align__(16) float tab[2][M];
    pdl_enter();
    const uint32_t e = threadIdx.x & 1u;
    const uint32_t first = blockIdx.x * uint32_t(kSplitFwdVecs);
    const uint32_t i = first + (threadIdx.x >> 1);
    const bool mine = i < n_vec;
    // the block's tokens' coefficients (V >= kSplitFwdVecs: at most two tokens)
    const uint32_t last = (n_vec - first > uint32_t(kSplitFwdVecs)) ? first + kSplitFwdVecs - 1 : n_vec - 1;
    const uint32_t t_first = fastdiv_u32(first, divV);
    const uint32_t count = (fastdiv_u32(last, divV) - t_first + 1) * uint32_t(M);
    if constexpr (!Coeffs::kBlockTable) {
        for (uint32_t q = threadIdx.x; q < count; q += kSplitFwdBlock) {
            const uint32_t tt = q / uint32_t(M), m = q - tt * uint32_t(M);
            const uint64_t t = uint64_t(t_first) + tt;
            if (m < uint32_t(N * N)) cp_async4(&tab[tt][m], res + uint64_t(N) * N * t + m);
            else cp_async4(&tab[tt][m], coeffs.pre + uint64_t(N) * t + int(m - N * N) / 2);
        }
        cp_async_commit();
    }
    uint32_t tok = 0;
    uint64_t row0 = 0;   // x / out vector of stream 0
    // x paired across input streams, xp[jp][p] = {x[2jp](p), x[2jp+1](p)},
    // and y at positions (0, 1), (2, 3)
    F2 xp[JP][4], yp[2];
    if (mine) {
        tok = fastdiv_u32(i, divV);
        row0 = uint64_t(N) * tok * V + (i - tok * V);
        uint2 xw[N];
#pragma unroll
        for (int j = 0; j < N; ++j) xw[j] = ld_stream_half(reinterpret_cast<const uint2*>(x + row0 + uint64_t(j) * V) + e);
        const uint2 yw = ld_stream_half(reinterpret_cast<const uint2*>(y + i) + e);
#pragma unroll
        for (int jp = 0; jp < JP; ++jp) {
            float a[4], b[4];
            unpack_half<DT>(xw[2 * jp], a);
            unpack_half<DT>(xw[2 * jp + 1], b);
#pragma unroll
            for (int p = 0; p < 4; ++p) xp[jp][p] = f2(a[p], b[p]);
        }
        float yf[4];
        unpack_half<DT>(yw, yf);
        yp[0] = f2(yf[0], yf[1]);
        yp[1] = f2(yf[2], yf[3]);
    }
    if constexpr (Coeffs::kBlockTable) {
        // post from the mix: the sigmoids are computed once the loads are issued
        for (uint32_t q = threadIdx.x; q < count; q += kSplitFwdBlock) {
            const uint32_t tt = q / uint32_t(M), m = q - tt * uint32_t(M);
            const uint64_t t = uint64_t(t_first) + tt;
            tab[tt][m] = (m < uint32_t(N * N)) ? __ldg(res + uint64_t(N) * N * t + m)
                                               : coeffs.pre_from(coeffs.mix_at(uint64_t(N) * t + (m - N * N) / 2),
                                                                 int(m - N * N) / 2);
        }
    } else {
        cp_async_wait_all();
    }
    __syncthreads();
    if (!mine) return;
    const float* ct = tab[tok - t_first];
#pragma unroll
    for (int k = 0; k < N; ++k) {
        // {res[k][2jp], res[k][2jp+1]} and {post[k], post[k]}
        F2 c[JP];
#pragma unroll
        for (int jp = 0; jp < JP; jp += 2) {
            const ulonglong2 r = *reinterpret_cast<const ulonglong2*>(ct + k * N + 2 * jp);
            c[jp].v = r.x, c[jp + 1].v = r.y;
        }
        F2 pk;
        pk.v = *reinterpret_cast<const uint64_t*>(ct + N * N + 2 * k);
        // post_value at positions (0, 1) and (2, 3): the tree's first level by
        // scalar adds of each packed product's halves, its upper levels
        // packed over the position pair, then the post term added by halves
        F2 o[2];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            F2 l1[JP];
#pragma unroll
            for (int jp = 0; jp < JP; ++jp)
                l1[jp] = f2(padd_halves(pmul(c[jp], xp[jp][2 * pp])), padd_halves(pmul(c[jp], xp[jp][2 * pp + 1])));
            o[pp] = sadd2(padd(padd(l1[0], l1[1]), padd(l1[2], l1[3])), pmul(pk, yp[pp]));
        }
        st_stream_half(reinterpret_cast<uint2*>(out + row0 + uint64_t(k) * V) + e,
                       Elem<DT>::pack(f2_lo(o[0]), f2_hi(o[0])), Elem<DT>::pack(f2_lo(o[1]), f2_hi(o[1])));
    }
}

// 2-byte path: a 2-D grid of (2048-value row segment, token) blocks,
// grid-stride over tokens; thread j takes values e*256 + j (e < 8).  With
// post computed from the mix, the token's n sigmoids go through shared
// memory (threads 0 .. n-1, one barrier before and after their use).
template <int N, int DT, class Coeffs>
__global__ void __launch_bounds__(kNarrowBlock)
post_fwd_element_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ y, Coeffs coeffs,
                        const float* __restrict__ res, uint16_t* __restrict__ out, uint64_t T, uint64_t H) {
    __shared__ float table[N];
    pdl_enter();
    const uint64_t base = uint64_t(blockIdx.x) * kNarrowSeg + threadIdx.x;
    for (uint64_t t = blockIdx.y; t < T; t += gridDim.y) {
        if constexpr (Coeffs::kBlockTable) {
            if (threadIdx.x < uint32_t(N))
                table[threadIdx.x] = coeffs.pre_from(coeffs.mix_at(uint64_t(N) * t + threadIdx.x), int(threadIdx.x));
            __syncthreads();
        }
#pragma unroll 2
        for (int e = 0; e < kNarrowPerThread; ++e) {
            const uint64_t h = base + uint64_t(e) * kNarrowBlock;
            if (h < H) {
                float xs[N];
#pragma unroll
                for (int j = 0; j < N; ++j) xs[j] = Elem<DT>::one(ld_stream2(x + (uint64_t(N) * t + j) * H + h));
                const float ys = Elem<DT>::one(ld_stream2(y + t * H + h));
#pragma unroll
                for (int k = 0; k < N; ++k) {
                    float rk[N];
                    ld_res_row<N>(res, t, k, rk);
                    float pk;
                    if constexpr (Coeffs::kBlockTable) pk = table[k];
                    else pk = __ldg(coeffs.pre + uint64_t(N) * t + k);
                    st_stream2(out + (uint64_t(N) * t + k) * H + h, Elem<DT>::cvt(post_value<N>(rk, pk, xs, ys)));
                }
            }
        }
        if constexpr (Coeffs::kBlockTable) __syncthreads();   // table[] is rewritten for the next token
    }
}

// --------------------------------------------------------------------------
// backward
// --------------------------------------------------------------------------

// One level of a warp reduce-scatter: the lane holds C values (indices
// base .. base + C - 1, the first `real` of them real, the rest +0 padding)
// and, with its partner lane ^ S, splits them: the lower lane keeps the first
// ceil(C/2), the upper one the rest, each adding the partner's copies of the
// values it keeps.  Every value is summed over exactly the lane pairs of the
// xor butterfly (lane i with i ^ S), and IEEE addition is commutative bit
// for bit, so each value's sum is the butterfly's, in fewer shuffles (at
// n = 4, 21 instead of 100 for 20 values).
template <int C, int S>
__device__ __forceinline__ void rs_level(const float (&v)[C], float (&out)[(C + 1) / 2], int& base, int& real,
                                         uint32_t lane) {
    constexpr int H = (C + 1) / 2;
    const bool upper = (lane & uint32_t(S)) != 0u;
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const float lo = v[i];
        const float hi = (H + i < C) ? v[H + i] : 0.0f;
        const float recv = __shfl_xor_sync(0xffffffffu, upper ? lo : hi, S);
        out[i] = __fadd_rn(upper ? hi : lo, recv);
    }
    if (upper) {
        base += H;
        real = real > H ? real - H : 0;
    } else {
        real = real < H ? real : H;
    }
}

// The warp sums of M values (the xor butterfly over 32 lanes), scattered:
// each lane hands the values it ends with to put(index, sum) ...
template <int M, class Put>
__device__ __forceinline__ void warp_sums_put(const float (&acc)[M], uint32_t lane, Put put) {
    constexpr int C1 = (M + 1) / 2, C2 = (C1 + 1) / 2, C3 = (C2 + 1) / 2, C4 = (C3 + 1) / 2, C5 = (C4 + 1) / 2;
    int base = 0, real = M;
    float a1[C1], a2[C2], a3[C3], a4[C4], a5[C5];
    rs_level<M, 16>(acc, a1, base, real, lane);
    rs_level<C1, 8>(a1, a2, base, real, lane);
    rs_level<C2, 4>(a2, a3, base, real, lane);
    rs_level<C3, 2>(a3, a4, base, real, lane);
    rs_level<C4, 1>(a4, a5, base, real, lane);
#pragma unroll
    for (int i = 0; i < C5; ++i)
        if (i < real) put(base + i, a5[i]);
}

// ... or writes them into row[index]
template <int M>
__device__ __forceinline__ void warp_sums_to(const float (&acc)[M], float* row, uint32_t lane) {
    warp_sums_put<M>(acc, lane, [row](int i, float v) { row[i] = v; });
}

// The cross-group step of the fold below: once the block's group values are
// in shared memory (group_value(g, m) for g < groups), value m folds over the
// 8 groups with strides 4, 2, 1 (a missing group counts +0) and is stored.
// Opens and closes with the group's barrier.
template <int N, class Coeffs, class Sync, class GroupValue>
__device__ __forceinline__ void post_fold_groups(GroupValue group_value, const Coeffs& coeffs, const float* slope,
                                                 float* __restrict__ grad_res, uint64_t t, Sync sync,
                                                 int groups, uint32_t thread) {
    constexpr int M = N * N + N;
    sync();
    if (thread < uint32_t(M)) {
        const int m = int(thread);
        float w[kGroups];
#pragma unroll
        for (int i = 0; i < kGroups; ++i) w[i] = (i < groups) ? group_value(i, m) : 0.0f;
#pragma unroll
        for (int s = kGroups / 2; s >= 1; s >>= 1) {
#pragma unroll
            for (int i = 0; i < s; ++i) w[i] = __fadd_rn(w[i], w[i + s]);
        }
        if (m < N * N) grad_res[uint64_t(N) * N * t + m] = w[0];
        else post_store_grad<N>(coeffs, t, m - N * N, w[0], slope);
    }
    sync();   // red[] (and the coefficient table) are reused by the next token
}

// The ORDER-256 fold of M = n*n + n lane sums of a 256-lane block (LPT lanes
// per thread: lanes LPT*thread + l): xor shuffles over each group of 32 lanes,
// the 8 group values through shared memory; grad_res[t,k,j] = value k*n + j,
// and value n*n + k, the gradient of post[t,k], goes to the coefficient
// source (post_store_grad; `slope` holds the token's sigmoid' when post comes
// from the mix).  All threads of the block call it.
//
// `groups`: the lane groups of 32 that have threads; the lanes of the others
// hold +0 and their group values are +0 in the cross-group fold.
template <int N, int LPT, class Coeffs, class Sync = BlockSync>
__device__ __forceinline__ void post_fold_and_store(float (&acc)[LPT][N * N + N], float (*red)[N * N + N],
                                                    const Coeffs& coeffs, const float* slope,
                                                    float* __restrict__ grad_res, uint64_t t,
                                                    Sync sync = Sync(), int groups = kGroups) {
    constexpr int M = N * N + N;
    constexpr int kThreadsPerGroup = 32 / LPT;
    if constexpr (LPT == 1) {
        // one lane per thread: the warp's sums by reduce-scatter
        warp_sums_to<M>(acc[0], red[threadIdx.x / 32], threadIdx.x & 31u);
    } else {
#pragma unroll
        for (int m = 0; m < M; ++m) {
#pragma unroll
            for (int s = kThreadsPerGroup / 2; s >= 1; s >>= 1) {
#pragma unroll
                for (int l = 0; l < LPT; ++l)
                    acc[l][m] = __fadd_rn(acc[l][m], __shfl_xor_sync(0xffffffffu, acc[l][m], s));
            }
            acc[0][m] = __fadd_rn(acc[0][m], acc[LPT - 1][m]);
        }
        if ((threadIdx.x % kThreadsPerGroup) == 0) {
#pragma unroll
            for (int m = 0; m < M; ++m) red[threadIdx.x / kThreadsPerGroup][m] = acc[0][m];
        }
    }
    post_fold_groups<N>([red](int i, int m) { return red[i][m]; }, coeffs, slope, grad_res, t, sync, groups,
                        threadIdx.x);
}

// The grad_x vector of input stream j (j < n) or the grad_y vector (j == n)
// from the n g vectors of one position: coefficient column j of res, or post.
template <int N, int DT, int NW, class C>
__device__ __forceinline__ Words<NW> post_chunk_grad(const C& cf, const Words<NW> (&gv)[N], int j) {
    Words<NW> o;
#pragma unroll
    for (int e = 0; e < NW; ++e) {
        float ql[N], qh[N];
#pragma unroll
        for (int k = 0; k < N; ++k) {
            const float c = j < N ? cf.r(k, j) : cf.p(k);
            ql[k] = __fmul_rn(c, Elem<DT>::lo(gv[k].w[e]));
            qh[k] = __fmul_rn(c, Elem<DT>::hi(gv[k].w[e]));
        }
        o.w[e] = Elem<DT>::pack(tree_sum<N>(ql), tree_sum<N>(qh));
    }
    return o;
}

// One position (NW/4 chunks) of a token: writes its grad_x and grad_y vectors
// and adds each chunk's partials to its lane's n*n + n sums.  Stream by
// stream, so that one gradient vector is live at a time.
template <int N, int DT, int NW, class C, class StX, class StY>
__device__ __forceinline__ void post_chunk(const C& cf, const Words<NW> (&gv)[N], const Words<NW> (&xv)[N],
                                           const Words<NW>& yv, float (&acc)[NW / 4][N * N + N], StX st_x,
                                           StY st_y) {
#pragma unroll
    for (int j = 0; j < N; ++j) {
        st_x(j, post_chunk_grad<N, DT, NW>(cf, gv, j));
#pragma unroll
        for (int k = 0; k < N; ++k) {
#pragma unroll
            for (int l = 0; l < NW / 4; ++l)
                acc[l][k * N + j] = __fadd_rn(acc[l][k * N + j], chunk_partial<DT, NW>(gv[k], xv[j], 4 * l));
        }
    }
    st_y(post_chunk_grad<N, DT, NW>(cf, gv, N));
#pragma unroll
    for (int k = 0; k < N; ++k) {
#pragma unroll
        for (int l = 0; l < NW / 4; ++l)
            acc[l][N * N + k] = __fadd_rn(acc[l][N * N + k], chunk_partial<DT, NW>(gv[k], yv, 4 * l));
    }
}

// Bulk-copy path (H % 8 == 0, the 2-byte buffers 16-byte aligned): the
// token's rows stream through shared memory.  A persistent block of 256
// consumer threads (ORDER-256 lane j = thread j) and one producer warp walks
// its tokens t = blockIdx, blockIdx + gridDim, ...; each token in segments of
// 256 chunks (4 KB of each row).  One producer thread copies a segment's
// 2n + 1 input row pieces (g, x, y) into a free stage of a STAGES-deep ring
// with bulk copies that complete on the stage's "full" barrier; each
// consumer thread then takes chunk j of the segment from shared memory,
// writes its grad_x and grad_y vectors, adds its partials, and its warp
// releases the stage on the "empty" barrier.  The loads thus stay in flight
// without holding registers.  After a token's last segment the consumers
// fold the lane sums (named barrier 1 over the 256 consumers).
//
// A wait that runs out (no copy should ever take that long) sets *timeouts
// to 1 (a plain store: every writer writes the same value); the thread then
// stops waiting, the block still runs to its end
// on whatever the stage holds, and the producer waits (bounded) for the
// copies it issued before it exits.
// A stage holds `width` chunks (16 bytes) of each of the 2n + 1 rows: 256,
// or for rows of fewer than 256 chunks the block's consumer threads.
__host__ __device__ constexpr uint32_t post_bulk_stage_bytes(int n, uint32_t width = kLanes) {
    return uint32_t(2 * n + 1) * width * 16u;
}

//
// With post computed from the mix (Coeffs::kBlockTable) a helper warp
// evaluates each token's sigmoids and slopes (lanes 0 .. n-1) into a ring of
// kPostSlots token slots, ahead of the consumers: slot i % kPostSlots is
// published by its "ready" barrier (the consumers wait on it before a
// token's first chunk) and handed back by its "free" barrier (consumer
// thread 0, after the token's fold), which the helper waits on before
// writing it again.  Neither the producer nor the consumers evaluate a
// sigmoid.
constexpr int kPostSlots = 3;

// The producer's check before it fills stage `st` for the `round`-th time:
// the consumers have released the stage's previous contents ("empty") and
// every byte of its previous copies has landed ("full"; the consumers waited
// for that phase already, so in a normal run this costs one poll).  If
// either wait runs out, the producer issues no further copy: re-arming a
// transaction barrier whose previous phase is still open, or writing into a
// stage that copies are still filling, is never done.
__device__ __forceinline__ bool stage_reusable(uint64_t* full, uint64_t* empty, uint32_t st, uint32_t round) {
    return mbar_wait(&empty[st], (round - 1) & 1u) && mbar_wait_fast(&full[st], (round - 1) & 1u);
}

// Threads of a block with `consumers` consumer threads (256, or for rows of
// fewer than 256 chunks the warps that hold chunks): then the producer warp,
// then (post from the mix) the helper warp.
template <class Coeffs>
__host__ __device__ constexpr int post_bulk_threads(int consumers = kLanes) {
    return consumers + 32 + (Coeffs::kBlockTable ? 32 : 0);
}

template <int N, int DT, int STAGES, int MIN_BLOCKS, class Coeffs, bool NARROW>
__global__ void __launch_bounds__(post_bulk_threads<Coeffs>(), MIN_BLOCKS)
post_bwd_bulk_kernel(const Words<4>* __restrict__ g, const Words<4>* __restrict__ x,
                     const Words<4>* __restrict__ y, Coeffs coeffs, const float* __restrict__ res,
                     Words<4>* __restrict__ grad_x, Words<4>* __restrict__ grad_y,
                     float* __restrict__ grad_res, uint64_t T, uint32_t V,
                     unsigned int* __restrict__ timeouts) {
    static_assert(N <= 4, "the bulk-copy kernel keeps its coefficients in registers");
    constexpr bool kSig = Coeffs::kBlockTable;
    constexpr int R = 2 * N + 1;   // staged rows: g (N), x (N), y
    constexpr int M = N * N + N;
    constexpr int kNS = kSig ? kPostSlots : 1;
    extern __shared__ __align__(128) unsigned char stage_mem[];   // STAGES * R * 4 KB
    __shared__ __align__(8) uint64_t full[STAGES];
    __shared__ __align__(8) uint64_t empty[STAGES];
    __shared__ __align__(8) uint64_t ready[kNS];
    __shared__ __align__(8) uint64_t freed[kNS];
    __shared__ float red[kGroups][M];
    __shared__ float slots[kNS][2 * N];   // post, then sigmoid'
    // consumer threads: 256, or (NARROW: rows of fewer than 256 chunks) a
    // multiple of 32 set by the launch; a stage row holds `width` chunks (256,
    // or all of a shorter row's)
    const uint32_t consumers = NARROW ? blockDim.x - 32u - (kSig ? 32u : 0u) : uint32_t(kLanes);
    const uint32_t width = consumers;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], consumers / 32u);
        }
#pragma unroll
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&ready[s], 1);
            mbar_init(&freed[s], 1);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_enter();
    const uint32_t nseg = (V + kLanes - 1) / kLanes;

    if (threadIdx.x >= consumers + 32u) {
        // helper warp (post from the mix): the block's tokens' sigmoids, in order
        if constexpr (kSig) {
            const uint32_t lane = threadIdx.x - (consumers + 32u);
            bool ok = true;
            uint32_t tok = 0;
            for (uint64_t t = blockIdx.x; t < T; t += gridDim.x, ++tok) {
                const uint32_t sl = tok % kNS;
                if (tok >= uint32_t(kNS) && lane == 0 && ok) ok = mbar_wait(&freed[sl], (tok / kNS - 1) & 1u);
                __syncwarp();
                if (lane < uint32_t(N)) {
                    coeffs.pre_and_slope(coeffs.mix_at(uint64_t(N) * t + lane), int(lane), slots[sl][lane],
                                         slots[sl][N + lane]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ready[sl]);
            }
            if (lane == 0 && !ok) *timeouts = 1u;
        }
        return;
    }

    if (threadIdx.x >= consumers) {
        // producer warp: one thread issues the copies
        if (threadIdx.x != consumers) return;
        bool ok = true;
        uint32_t item = 0, issued = 0;
        for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
            for (uint32_t s = 0; s < nseg; ++s, ++item) {
                const uint32_t st = item % STAGES, round = item / STAGES;
                if (round > 0 && ok) ok = stage_reusable(full, empty, st, round);
                if (!ok) continue;   // after a wait ran out, no copy is issued
                const uint32_t c0 = s * kLanes;
                const uint32_t bytes = (V - c0 < uint32_t(kLanes) ? V - c0 : uint32_t(kLanes)) * 16u;
                unsigned char* dst = stage_mem + size_t(st) * post_bulk_stage_bytes(N, width);
                mbar_arrive_expect_tx(&full[st], bytes * R);
#pragma unroll
                for (int k = 0; k < N; ++k) {
                    bulk_copy_g2s(dst + size_t(k) * width * 16, g + (uint64_t(N) * t + k) * V + c0, bytes, &full[st]);
                    bulk_copy_g2s(dst + size_t(N + k) * width * 16, x + (uint64_t(N) * t + k) * V + c0, bytes,
                                  &full[st]);
                }
                bulk_copy_g2s(dst + size_t(2 * N) * width * 16, y + t * V + c0, bytes, &full[st]);
                issued = item + 1;
            }
        }
        // every copy issued has landed before the block's shared memory goes
        for (uint32_t i = issued > uint32_t(STAGES) ? issued - STAGES : 0; i < issued; ++i)
            if (!mbar_wait(&full[i % STAGES], (i / STAGES) & 1u)) ok = false;
        if (!ok) *timeouts = 1u;
        return;
    }

    // consumers
    const uint32_t j = threadIdx.x;
    const auto sync = [consumers] { named_sync(1, consumers); };
    bool ok = true;
    uint32_t item = 0, tok = 0;
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x, ++tok) {
        const uint32_t sl = tok % kNS;
        PostCoeffs<N> cf;
        if constexpr (kSig) {
            cf.load_res(res, t);
            if (ok) ok = mbar_wait(&ready[sl], (tok / kNS) & 1u);
#pragma unroll
            for (int k = 0; k < N; ++k) cf.pk[k] = slots[sl][k];
        } else {
            cf.load(coeffs.pre, res, t, nullptr, sync);
        }
        float acc[1][M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[0][m] = 0.0f;
#pragma unroll 1
        for (uint32_t s = 0; s < nseg; ++s, ++item) {
            const uint32_t st = item % STAGES;
            if (ok) ok = mbar_wait(&full[st], (item / STAGES) & 1u);
            const uint32_t c = s * kLanes + j;
            if (c < V) {
                const Words<4>* sm =
                    reinterpret_cast<const Words<4>*>(stage_mem + size_t(st) * post_bulk_stage_bytes(N, width)) + j;
                Words<4> gv[N], xv[N];
#pragma unroll
                for (int k = 0; k < N; ++k) {
                    gv[k] = sm[k * width];
                    xv[k] = sm[(N + k) * width];
                }
                const Words<4> yv = sm[2 * N * width];
                post_chunk<N, DT, 4>(
                    cf, gv, xv, yv, acc,
                    [&](int k, const Words<4>& o) { st_stream<4>(grad_x + (uint64_t(N) * t + k) * V + c, o); },
                    [&](const Words<4>& o) { st_stream<4>(grad_y + t * V + c, o); });
            }
            __syncwarp();
            if ((j & 31u) == 0) mbar_arrive(&empty[st]);
        }
        post_fold_and_store<N, 1>(acc, red, coeffs, slots[sl] + N, grad_res, t, sync, int(consumers / 32u));
        // the fold's closing barrier: every consumer is done with the slot
        if (kSig && j == 0) mbar_arrive(&freed[sl]);
    }
    if (!ok) *timeouts = 1u;
}

// Split bulk-copy path for n = 8 (H % 8 == 0, the 2-byte buffers 16-byte
// aligned).  A lane's 72 sums do not fit one thread's registers beside its
// chunk's 17 input vectors, so each ORDER-256 lane is served by two consumer
// threads that split the chunk's 8 positions: thread half e takes positions
// 4e .. 4e + 3 (words 2e, 2e + 1 of each 16-byte vector).
//
//  * grad_x, grad_y: each thread writes its 8 bytes of every output vector;
//    the n-term tree is (k < n/2 terms) + (k >= n/2 terms), and a thread
//    holds the g values of "its" n/2 streams k (4e .. 4e + 3) and of the
//    other n/2 in separate arrays, so the two subtrees come out in either
//    order and add commutatively.
//  * a chunk's partial for stream pair (k, j) is chunk_partial's tree,
//    (positions 0-3) + (positions 4-7): each thread forms its half for
//    every k, keeps the sum of k in its own range and sends the other
//    half to its partner (shfl_xor 1), which adds it to its own.  Thread e
//    thus keeps the lane sums of grad_res[k][j] and grad_post[k] for
//    k in 4e .. 4e + 3 (36 values).
//  * lanes: warps 2q and 2q + 1 hold the lanes of group q with lane bit 0
//    equal to 0 and 1 (lane 32q + 2i + b in thread 2i + e of warp 2q + b).
//    The in-group fold's strides 16, 8, 4, 2 are thread strides 16 .. 2
//    (reduce-scatter), stride 1 adds the two warps' values in shared
//    memory, then the groups fold with strides 4, 2, 1: ORDER-256's pairs
//    and order.
//
// The rows stream through shared memory as in the bulk kernel above (one
// producer warp, a STAGES-deep ring of (2n + 1) x 4 KB stages, "full" and
// "empty" barriers, bounded waits and the same timeout flag).  The token's
// coefficients sit in a shared table (split_prefetch_table).
constexpr int kSplitConsumers = 2 * kLanes;

template <int N>
constexpr int kSplitSums = N * N / 2 + N / 2;

// warp_sums_put's reduce-scatter over thread strides 16, 8, 4, 2 only
// (thread bit 0, the position half, stays apart): each thread hands the
// sums it ends with to put(index, sum).
template <int M, class Put>
__device__ __forceinline__ void pair_sums_put(const float (&acc)[M], uint32_t lane, Put put) {
    constexpr int C1 = (M + 1) / 2, C2 = (C1 + 1) / 2, C3 = (C2 + 1) / 2, C4 = (C3 + 1) / 2;
    int base = 0, real = M;
    float a1[C1], a2[C2], a3[C3], a4[C4];
    rs_level<M, 16>(acc, a1, base, real, lane);
    rs_level<C1, 8>(a1, a2, base, real, lane);
    rs_level<C2, 4>(a2, a3, base, real, lane);
    rs_level<C3, 2>(a3, a4, base, real, lane);
#pragma unroll
    for (int i = 0; i < C4; ++i)
        if (i < real) put(base + i, a4[i]);
}

// Sum i of position half e is value m of the fold (k*n + j: grad_res;
// n*n + k: grad_post): i < n*n/2 is k = e n/2 + i / n, j = i % n; the rest
// grad_post[e n/2 + i - n*n/2].
template <int N>
__device__ __forceinline__ int split_sum_index(uint32_t e, int i) {
    constexpr int NH = N / 2;
    return i < N * NH ? int(e) * NH * N + i : N * N + int(e) * NH + (i - N * NH);
}

// One chunk, position half e, in packed pairs (mhc_f32x2.cuh).  sm = the
// stage's row 0 at this thread's 8 bytes (row r at sm[r * 2 * kLanes]);
// tab = the token table (tab[j*n + k] = res[t,k,j], tab[n*n + k] =
// post[t,k]); gx = grad_x row 0 at this thread's 8 bytes (row j at
// gx[j * rs]); gy likewise for grad_y; `live` = the warp's threads that run
// it (both threads of each lane).
//
// The g values are paired across streams: go[i][p] = {g[ko + 2i](p),
// g[ko + 2i + 1](p)} for this thread's own streams ko = n/2 e ..., gt[i][p]
// for the other half's, at its 4 positions p.  For each input j (j == n:
// y with post):
//  * grad_x / grad_y at positions p, p + 1: each coefficient pair times
//    each g pair (packed products) summed by halves (scalar adds: the
//    tree's first level, streams 2i + 2i+1), then the tree's upper levels
//    on position pairs (packed sums); own subtree + other subtree is the
//    tree's last add.
//  * the half partials of every (k, j): the 4 products of a g pair with x
//    duplicated, (p0 + p1) + (p2 + p3) by scalar then packed adds; the
//    other half's two pairs go to the partner (shuffle), whose own add
//    completes chunk_partial's last level; acc[j][i] (own streams
//    ko + 2i, ko + 2i + 1) adds the chunk's partial (packed).
template <int N, int DT>
__device__ __forceinline__ void post_split_chunk(const uint2* sm, uint32_t e, const float* tab,
                                                 F2 (&acc)[N + 1][N / 4], uint2* gx, uint64_t rs, uint2* gy,
                                                 uint32_t live) {
    static_assert(N == 8, "the packed split chunk is written for n = 8");
    constexpr int NH = N / 2, KP = NH / 2;   // streams per half, stream pairs per half
    const uint32_t ko = NH * e, kt = NH - ko;   // first own stream, first of the other half
    F2 go[KP][4], gt[KP][4];
#pragma unroll
    for (int i = 0; i < KP; ++i) {
        float a[4], b[4], c[4], d[4];
        unpack_half<DT>(sm[(ko + 2 * i) * 2 * kLanes], a);
        unpack_half<DT>(sm[(ko + 2 * i + 1) * 2 * kLanes], b);
        unpack_half<DT>(sm[(kt + 2 * i) * 2 * kLanes], c);
        unpack_half<DT>(sm[(kt + 2 * i + 1) * 2 * kLanes], d);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            go[i][p] = f2(a[p], b[p]);
            gt[i][p] = f2(c[p], d[p]);
        }
    }
#pragma unroll
    for (int j = 0; j <= N; ++j) {
        const bool is_y = j == N;
        float xf[4];
        unpack_half<DT>(sm[(is_y ? 2 * N : N + j) * 2 * kLanes], xf);
        F2 co[KP], ct[KP];
        {
            const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(tab + j * N + ko);
            const ulonglong2 b = *reinterpret_cast<const ulonglong2*>(tab + j * N + kt);
            co[0].v = a.x, co[1].v = a.y, ct[0].v = b.x, ct[1].v = b.y;
        }
        // grad_x (grad_y) at positions (0, 1) and (2, 3)
        F2 v[2];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            F2 lo[KP], lt[KP];
#pragma unroll
            for (int i = 0; i < KP; ++i) {
                lo[i] = f2(padd_halves(pmul(co[i], go[i][2 * pp])), padd_halves(pmul(co[i], go[i][2 * pp + 1])));
                lt[i] = f2(padd_halves(pmul(ct[i], gt[i][2 * pp])), padd_halves(pmul(ct[i], gt[i][2 * pp + 1])));
            }
            v[pp] = padd(padd(lo[0], lo[1]), padd(lt[0], lt[1]));
        }
        st_stream_half(is_y ? gy : gx + uint64_t(j) * rs, Elem<DT>::pack(f2_lo(v[0]), f2_hi(v[0])),
                       Elem<DT>::pack(f2_lo(v[1]), f2_hi(v[1])));
        // half partials of (k, j) for every k
        F2 xd[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) xd[p] = f2(xf[p], xf[p]);
#pragma unroll
        for (int i = 0; i < KP; ++i) {
            const F2 ho = padd(sadd2(pmul(go[i][0], xd[0]), pmul(go[i][1], xd[1])),
                               sadd2(pmul(go[i][2], xd[2]), pmul(go[i][3], xd[3])));
            const F2 ht = padd(sadd2(pmul(gt[i][0], xd[0]), pmul(gt[i][1], xd[1])),
                               sadd2(pmul(gt[i][2], xd[2]), pmul(gt[i][3], xd[3])));
            acc[j][i] = padd(acc[j][i], padd(ho, shfl_xor_f2(live, ht, 1)));
        }
    }
}

// Token t's table: tab[j*n + k] = res[t,k,j], tab[n*n + k] = post[t,k]
// (from the mix: computed, and tab[n*n + n + k] = sigmoid').  It is fetched
// a token ahead: consumer threads m < n*n + n start 4-byte asynchronous
// copies of their value (the mix value into mix[k] when post comes from the
// mix) while the block works on the previous token ...
template <int N, class Coeffs>
__device__ __forceinline__ void split_prefetch_table(const Coeffs& c, const float* __restrict__ res, uint64_t t,
                                                     uint32_t m, float* tab, float* mix) {
    if (m < uint32_t(N * N)) {
        cp_async4(&tab[(m % N) * N + m / N], res + uint64_t(N) * N * t + m);
    } else if (m < uint32_t(N * N + N)) {
        const uint32_t k = m - uint32_t(N * N);
        if constexpr (Coeffs::kBlockTable) cp_async4(&mix[k], c.mix + uint64_t(N) * t + k);
        else cp_async4(&tab[m], c.pre + uint64_t(N) * t + k);
    }
    cp_async_commit();
}

// ... and complete it at the token's start: each thread waits for its copy,
// the sigmoids are evaluated (post from the mix), then the consumers' barrier.
template <int N, class Coeffs, class Sync>
__device__ __forceinline__ void split_finish_table(const Coeffs& c, uint32_t m, float* tab, const float* mix,
                                                   Sync sync) {
    cp_async_wait_all();
    if constexpr (Coeffs::kBlockTable) {
        if (m >= uint32_t(N * N) && m < uint32_t(N * N + N)) {
            const int k = int(m) - N * N;
            c.pre_and_slope(mix[k], k, tab[m], tab[m + N]);
        }
    }
    sync();
}

// The block is the 16 consumer warps alone (512 threads, up to 128 registers
// a thread): there is no producer warp.  The ring's first STAGES items are
// issued by thread 0 at the start; afterwards the warp that releases a stage
// last (a shared-memory counter of releasing warps) refills it with the item
// STAGES ahead, which is the earliest moment any producer could.  Items are
// the block's (token, segment) pairs in order.  A stage is three tiled
// copies, each a box of 2048 consecutive values (256 chunks) of a token's
// rows: g's n rows, x's n rows and y's row (tensor maps of
// [T][rows][H / W groups][W values], W the widest of 256, 128, ..., 8 that
// divides H; the boxes of a row's last segment read zeros past its end).
// The copy engine set the pace, not the arithmetic: it works through a box
// row by row, and with 16-byte rows (W = 8) a stage is about 4000 of them
// (T = 4096, H = 7168: W = 8 366 us, W = 64 or 256 336 us; with W = 8,
// removing 45% of the FP32 work gained 5 us, and an L2 prefetch of the next
// items through the same tensor maps doubled the time).  Three copies a
// stage, not one a row: with linear copies the count set the pace (two
// stages: 17 copies of 4 KB a stage 377 us, 34 of 2 KB 443 us; three stages:
// 17 copies 380 us).
// A schedule whose two warp halves swap lane halves every token (so that
// neither idles in a row's last, half-empty round) needed two tiled copies
// per input a stage and measured 362 us at H = 7168 but 10-13 us more at
// H = 2048 .. 6144.
template <int N>
__device__ __forceinline__ void split_issue(uint64_t* full, unsigned char* stage_mem, uint32_t item, uint32_t nseg,
                                            uint32_t stages, const CUtensorMap* g, const CUtensorMap* x,
                                            const CUtensorMap* y, uint32_t W) {
    const uint32_t st = item % stages;
    const int t = int(blockIdx.x + (item / nseg) * gridDim.x);
    const int c0 = int((item % nseg) * (8u * kLanes / W));   // the segment's first group of W values
    unsigned char* dst = stage_mem + size_t(st) * post_bulk_stage_bytes(N);
    mbar_arrive_expect_tx(&full[st], post_bulk_stage_bytes(N));
    tensor_copy_4d(dst, g, 0, c0, 0, t, &full[st]);
    tensor_copy_4d(dst + size_t(N) * kLanes * 16, x, 0, c0, 0, t, &full[st]);
    tensor_copy_4d(dst + size_t(2 * N) * kLanes * 16, y, 0, c0, 0, t, &full[st]);
}

template <int N, int DT, int STAGES, class Coeffs>
__global__ void __launch_bounds__(kSplitConsumers, 1)
post_bwd_split_kernel(const __grid_constant__ CUtensorMap g, const __grid_constant__ CUtensorMap x,
                      const __grid_constant__ CUtensorMap y, Coeffs coeffs, const float* __restrict__ res,
                      Words<4>* __restrict__ grad_x, Words<4>* __restrict__ grad_y,
                      float* __restrict__ grad_res, uint64_t T, uint32_t V, uint32_t W,
                      unsigned int* __restrict__ timeouts) {
    static_assert(N % 8 == 0, "the position halves take n/2 streams, read 4 coefficients at a time");
    constexpr int M = N * N + N;
    constexpr uint32_t kWarps = kSplitConsumers / 32;
    extern __shared__ __align__(128) unsigned char smem_raw[];   // STAGES * (2n + 1) * 4 KB + 128
    // tiled copies land on 128-byte boundaries: the ring starts at the first
    // one in the dynamic allocation (which has 128 bytes to spare)
    unsigned char* const stage_mem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    __shared__ __align__(8) uint64_t full[STAGES];
    __shared__ uint32_t released[STAGES];
    __shared__ float red[kWarps][M];
    __shared__ __align__(16) float tab[2][kPostTable<N>];   // tokens alternate
    __shared__ float mix[2][N];
    const uint32_t nseg = (V + kLanes - 1) / kLanes;
    const uint64_t tokens = T > blockIdx.x ? (T - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t items = uint32_t(tokens * nseg);
    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            released[s] = 0;
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_enter();
    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < items && i < uint32_t(STAGES); ++i)
            split_issue<N>(full, stage_mem, i, nseg, STAGES, &g, &x, &y, W);
    }

    // warp 2q + b, thread 2i + e holds position half e of lane 32q + 2i + b
    const uint32_t w = threadIdx.x >> 5, l = threadIdx.x & 31u;
    const uint32_t e = l & 1u;
    const uint32_t j = 32u * (w >> 1) + (l & ~1u) + (w & 1u);   // the ORDER-256 lane
    const auto sync = [] { named_sync(1, kSplitConsumers); };
    bool ok = true;
    uint32_t item = 0, tok = 0;
    if (blockIdx.x < T) split_prefetch_table<N>(coeffs, res, blockIdx.x, threadIdx.x, tab[0], mix[0]);
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x, ++tok) {
        // the previous token's readers of tab[cur ^ 1] are past its fold
        const uint32_t cur = tok & 1u;
        split_finish_table<N>(coeffs, threadIdx.x, tab[cur], mix[cur], sync);
        if (t + gridDim.x < T)
            split_prefetch_table<N>(coeffs, res, t + gridDim.x, threadIdx.x, tab[cur ^ 1u], mix[cur ^ 1u]);
        const float* ttab = tab[cur];
        F2 acc[N + 1][N / 4];
#pragma unroll
        for (int jj = 0; jj <= N; ++jj)
#pragma unroll
            for (int i = 0; i < N / 4; ++i) acc[jj][i] = f2(0.0f, 0.0f);
#pragma unroll 1
        for (uint32_t s = 0; s < nseg; ++s, ++item) {
            const uint32_t st = item % STAGES;
            if (ok) ok = mbar_wait(&full[st], (item / STAGES) & 1u);
            const uint32_t c = s * kLanes + j;
            // in a row's last segment a warp may hold chunks in only some of
            // its threads (always both threads of a lane): the partner
            // exchange runs over those
            const uint32_t live = __ballot_sync(0xffffffffu, c < V);
            if (c < V) {
                const uint2* sm = reinterpret_cast<const uint2*>(stage_mem + size_t(st) * post_bulk_stage_bytes(N)) +
                                  2 * j + e;
                uint2* gx = reinterpret_cast<uint2*>(grad_x + uint64_t(N) * t * V + c) + e;
                uint2* gy = reinterpret_cast<uint2*>(grad_y + t * V + c) + e;
                post_split_chunk<N, DT>(sm, e, ttab, acc, gx, 2ull * V, gy, live);
            }
            // the warp is done with the stage; the last warp to say so refills
            // it with the item STAGES ahead, once the stage's copies have all
            // landed (a wait that ran out stops the refills)
            __syncwarp();
            if (l == 0) {
                if (release_count(&released[st], kWarps - 1) == kWarps - 1 && item + STAGES < items) {
                    fence_proxy_async_shared();
                    if (ok && mbar_wait_fast(&full[st], (item / STAGES) & 1u))
                        split_issue<N>(full, stage_mem, item + STAGES, nseg, STAGES, &g, &x, &y, W);
                    else
                        ok = false;
                }
            }
        }
        // the pairs in split_sum_index's order: own stream ko + c of input j
        // at c * n + j, grad_post of own stream ko + c at n*n/2 + c
        float flat[kSplitSums<N>];
#pragma unroll
        for (int jj = 0; jj <= N; ++jj)
#pragma unroll
            for (int i = 0; i < N / 4; ++i) {
                const int c0 = 2 * i, c1 = 2 * i + 1;
                flat[jj < N ? c0 * N + jj : N * N / 2 + c0] = f2_lo(acc[jj][i]);
                flat[jj < N ? c1 * N + jj : N * N / 2 + c1] = f2_hi(acc[jj][i]);
            }
        pair_sums_put<kSplitSums<N>>(flat, l, [&](int i, float v) { red[w][split_sum_index<N>(e, i)] = v; });
        post_fold_groups<N>([](int q, int m) { return __fadd_rn(red[2 * q][m], red[2 * q + 1][m]); }, coeffs,
                            ttab + N * N + N, grad_res, t, sync, kGroups, threadIdx.x);
    }
    // every copy issued has landed before the block's shared memory goes (in a
    // normal run the consumers waited for each already)
    sync();
    if (threadIdx.x == 0) {
        for (uint32_t i = items > uint32_t(STAGES) ? items - STAGES : 0; i < items; ++i)
            if (!mbar_wait(&full[i % STAGES], (i / STAGES) & 1u)) ok = false;
    }
    if (!ok) *timeouts = 1u;
}

// 2-byte path: any H and 2-byte alignment; the same lanes and chunks, the
// chunk's values read and written one by one (+0 past H).
__device__ __forceinline__ Words<4> ld_chunk2(const uint16_t* row, uint64_t h0, uint64_t H) {
    Words<4> v = {{0u, 0u, 0u, 0u}};
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (h0 + i < H) v.w[i >> 1] |= uint32_t(__ldg(row + h0 + i)) << (16 * (i & 1));
    return v;
}

__device__ __forceinline__ void st_chunk2(uint16_t* row, uint64_t h0, uint64_t H, const Words<4>& v) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (h0 + i < H) st_stream2(row + h0 + i, uint16_t(v.w[i >> 1] >> (16 * (i & 1))));
}

template <int N, int DT, class Coeffs>
__global__ void __launch_bounds__(kLanes)
post_bwd_element_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ x,
                        const uint16_t* __restrict__ y, Coeffs coeffs, const float* __restrict__ res,
                        uint16_t* __restrict__ grad_x, uint16_t* __restrict__ grad_y,
                        float* __restrict__ grad_res, uint64_t T, uint64_t H) {
    constexpr int M = N * N + N;
    __shared__ float red[kGroups][M];
    __shared__ float coef[kPostTable<N>];
    pdl_enter();
    const uint32_t j = threadIdx.x;
    const uint64_t C = (H + 7) / 8;
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
        PostCoeffs<N> cf;
        post_load_token<N>(coeffs, res, t, j, coef, cf, BlockSync());
        float acc[1][M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[0][m] = 0.0f;
        const uint64_t row0 = uint64_t(N) * t * H;
        for (uint64_t c = j; c < C; c += kLanes) {
            Words<4> gv[N], xv[N];
#pragma unroll
            for (int k = 0; k < N; ++k) {
                gv[k] = ld_chunk2(g + row0 + uint64_t(k) * H, 8 * c, H);
                xv[k] = ld_chunk2(x + row0 + uint64_t(k) * H, 8 * c, H);
            }
            const Words<4> yv = ld_chunk2(y + t * H, 8 * c, H);
            post_chunk<N, DT, 4>(
                cf, gv, xv, yv, acc,
                [&](int k, const Words<4>& o) { st_chunk2(grad_x + row0 + uint64_t(k) * H, 8 * c, H, o); },
                [&](const Words<4>& o) { st_chunk2(grad_y + t * H, 8 * c, H, o); });
        }
        post_fold_and_store<N, 1>(acc, red, coeffs, coef + N * N + N, grad_res, t);
    }
}

}  // namespace mhc
