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
// Kernels (HBM-bound: the forward moves (4n + 2) H bytes a token, the
// backward (6n + 4) H):
//  * forward, vector path: a flat grid over the [T,H] plane in 16- or
//    32-byte vectors; a thread loads the n x vectors and the y vector of its
//    position and writes the n output vectors.
//  * backward, vector path (16-byte): one 256-thread block per token, thread
//    j = ORDER-256 lane j taking chunks j, j + 256, ...; it writes grad_x and
//    grad_y for its chunk and adds the chunk partials of the n*n + n sums,
//    which fold like grad_pre's.
//  * other shapes and alignments: the same arithmetic with 2-byte accesses.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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

// The coefficients of the token a backward block works on.  Up to n = 4 they
// sit in registers; at n = 8 (72 values, next to 72 lane sums) in shared
// memory, read where they are used.
template <int N, bool kShared = (N >= 8)>
struct PostCoeffs {
    float pk[N], rk[N][N];
    __device__ __forceinline__ void load(const float* post, const float* res, uint64_t t, float*) {
        ld_post_coeffs<N>(post, res, t, pk, rk);
    }
    __device__ __forceinline__ float r(int k, int j) const { return rk[k][j]; }
    __device__ __forceinline__ float p(int k) const { return pk[k]; }
};

template <int N>
struct PostCoeffs<N, true> {
    const float* s;   // rk row-major, then pk
    // Every thread of the block calls this; the previous token's readers have
    // passed the fold's closing barrier.
    __device__ __forceinline__ void load(const float* post, const float* res, uint64_t t, float* smem) {
        if (threadIdx.x < uint32_t(N * N)) smem[threadIdx.x] = __ldg(res + uint64_t(N) * N * t + threadIdx.x);
        else if (threadIdx.x < uint32_t(N * N + N))
            smem[threadIdx.x] = __ldg(post + uint64_t(N) * t + (threadIdx.x - N * N));
        __syncthreads();
        s = smem;
    }
    __device__ __forceinline__ float r(int k, int j) const { return s[k * N + j]; }
    __device__ __forceinline__ float p(int k) const { return s[N * N + k]; }
};

// One output value of stream k from the n input values xs and y.
template <int N>
__device__ __forceinline__ float post_value(const float (&pk)[N], const float (&rk)[N][N], int k,
                                            const float (&xs)[N], float ys) {
    float p[N];
#pragma unroll
    for (int j = 0; j < N; ++j) p[j] = __fmul_rn(rk[k][j], xs[j]);
    return __fadd_rn(tree_sum<N>(p), __fmul_rn(pk[k], ys));
}

// --------------------------------------------------------------------------
// forward
// --------------------------------------------------------------------------

constexpr int kPostBlock = 256;

// Vector path: vector i of the [T, V] plane (V = H / (2*NW) per row).
template <int N, int DT, int NW>
__global__ void __launch_bounds__(kPostBlock)
post_fwd_vec_kernel(const Words<NW>* __restrict__ x, const Words<NW>* __restrict__ y,
                    const float* __restrict__ post, const float* __restrict__ res,
                    Words<NW>* __restrict__ out, uint32_t n_vec, uint32_t V, FastDivU32 divV) {
    pdl_enter();
    const uint32_t i = blockIdx.x * kPostBlock + threadIdx.x;
    if (i >= n_vec) return;
    const uint32_t t = fastdiv_u32(i, divV);
    const uint64_t row0 = uint64_t(N) * t * V + (i - t * V);   // x / out vector of stream 0
    Words<NW> xv[N];
#pragma unroll
    for (int j = 0; j < N; ++j) xv[j] = ld_stream<NW>(x + row0 + uint64_t(j) * V);
    const Words<NW> yv = ld_stream<NW>(y + i);
    float pk[N], rk[N][N];
    ld_post_coeffs<N>(post, res, t, pk, rk);
#pragma unroll
    for (int k = 0; k < N; ++k) {
        Words<NW> o;
#pragma unroll
        for (int e = 0; e < NW; ++e) {
            float xl[N], xh[N];
#pragma unroll
            for (int j = 0; j < N; ++j) {
                xl[j] = Elem<DT>::lo(xv[j].w[e]);
                xh[j] = Elem<DT>::hi(xv[j].w[e]);
            }
            o.w[e] = Elem<DT>::pack(post_value<N>(pk, rk, k, xl, Elem<DT>::lo(yv.w[e])),
                                    post_value<N>(pk, rk, k, xh, Elem<DT>::hi(yv.w[e])));
        }
        st_stream<NW>(out + row0 + uint64_t(k) * V, o);
    }
}

// 2-byte path: a 2-D grid of (2048-value row segment, token) blocks,
// grid-stride over tokens; thread j takes values e*256 + j (e < 8).
template <int N, int DT>
__global__ void __launch_bounds__(kNarrowBlock)
post_fwd_element_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ y,
                        const float* __restrict__ post, const float* __restrict__ res,
                        uint16_t* __restrict__ out, uint64_t T, uint64_t H) {
    pdl_enter();
    const uint64_t base = uint64_t(blockIdx.x) * kNarrowSeg + threadIdx.x;
    for (uint64_t t = blockIdx.y; t < T; t += gridDim.y) {
        float pk[N], rk[N][N];
        ld_post_coeffs<N>(post, res, t, pk, rk);
#pragma unroll 2
        for (int e = 0; e < kNarrowPerThread; ++e) {
            const uint64_t h = base + uint64_t(e) * kNarrowBlock;
            if (h < H) {
                float xs[N];
#pragma unroll
                for (int j = 0; j < N; ++j) xs[j] = Elem<DT>::one(ld_stream2(x + (uint64_t(N) * t + j) * H + h));
                const float ys = Elem<DT>::one(ld_stream2(y + t * H + h));
#pragma unroll
                for (int k = 0; k < N; ++k)
                    st_stream2(out + (uint64_t(N) * t + k) * H + h, Elem<DT>::cvt(post_value<N>(pk, rk, k, xs, ys)));
            }
        }
    }
}

// --------------------------------------------------------------------------
// backward
// --------------------------------------------------------------------------

// The ORDER-256 fold of M = n*n + n lane sums of a 256-thread block (one lane
// per thread): xor shuffles over each group of 32, the 8 group values
// through shared memory; grad_res[t,k,j] = value k*n + j, grad_post[t,k] =
// value n*n + k.
template <int N>
__device__ __forceinline__ void post_fold_and_store(float (&acc)[N * N + N], float (*red)[N * N + N],
                                                    float* __restrict__ grad_post,
                                                    float* __restrict__ grad_res, uint64_t t) {
    constexpr int M = N * N + N;
#pragma unroll
    for (int m = 0; m < M; ++m) {
#pragma unroll
        for (int s = 16; s >= 1; s >>= 1) acc[m] = __fadd_rn(acc[m], __shfl_xor_sync(0xffffffffu, acc[m], s));
    }
    if ((threadIdx.x & 31u) == 0) {
#pragma unroll
        for (int m = 0; m < M; ++m) red[threadIdx.x / 32][m] = acc[m];
    }
    __syncthreads();
    if (threadIdx.x < uint32_t(M)) {
        const int m = threadIdx.x;
        float w[kGroups];
#pragma unroll
        for (int i = 0; i < kGroups; ++i) w[i] = red[i][m];
#pragma unroll
        for (int s = kGroups / 2; s >= 1; s >>= 1) {
#pragma unroll
            for (int i = 0; i < s; ++i) w[i] = __fadd_rn(w[i], w[i + s]);
        }
        if (m < N * N) grad_res[uint64_t(N) * N * t + m] = w[0];
        else grad_post[uint64_t(N) * t + (m - N * N)] = w[0];
    }
    __syncthreads();   // red[] is reused by the next token
}

// The chunk's grad_x vector of input stream j (j < n) or its grad_y vector
// (j == n) from the n g vectors: coefficient column j of res, or post.
template <int N, int DT, class C>
__device__ __forceinline__ Words<4> post_chunk_grad(const C& cf, const Words<4> (&gv)[N], int j) {
    Words<4> o;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
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

// One chunk of a token: writes its grad_x and grad_y vectors and adds its
// partials to the n*n + n lane sums.  Stream by stream, so that only one
// stream's gradient vector is live at a time.
template <int N, int DT, class C, class StX, class StY>
__device__ __forceinline__ void post_chunk(const C& cf, const Words<4> (&gv)[N], const Words<4> (&xv)[N],
                                           const Words<4>& yv, float (&acc)[N * N + N], StX st_x, StY st_y) {
#pragma unroll
    for (int j = 0; j < N; ++j) {
        st_x(j, post_chunk_grad<N, DT>(cf, gv, j));
#pragma unroll
        for (int k = 0; k < N; ++k) acc[k * N + j] = __fadd_rn(acc[k * N + j], chunk_partial<DT, 4>(gv[k], xv[j], 0));
    }
    st_y(post_chunk_grad<N, DT>(cf, gv, N));
#pragma unroll
    for (int k = 0; k < N; ++k) acc[N * N + k] = __fadd_rn(acc[N * N + k], chunk_partial<DT, 4>(gv[k], yv, 0));
}

// 16-byte path: H % 8 == 0, the 2-byte buffers 16-byte aligned; V = H / 8
// vectors (= chunks) per row.
template <int N, int DT>
__global__ void __launch_bounds__(kLanes)
post_bwd_vec_kernel(const Words<4>* __restrict__ g, const Words<4>* __restrict__ x,
                    const Words<4>* __restrict__ y, const float* __restrict__ post,
                    const float* __restrict__ res, Words<4>* __restrict__ grad_x,
                    Words<4>* __restrict__ grad_y, float* __restrict__ grad_post,
                    float* __restrict__ grad_res, uint64_t T, uint32_t V) {
    constexpr int M = N * N + N;
    __shared__ float red[kGroups][M];
    __shared__ float coef[M];
    pdl_enter();
    const uint32_t j = threadIdx.x;
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
        PostCoeffs<N> cf;
        cf.load(post, res, t, coef);
        float acc[M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = 0.0f;
        const uint64_t row0 = uint64_t(N) * t * V;
        for (uint32_t v = j; v < V; v += kLanes) {
            Words<4> gv[N], xv[N];
#pragma unroll
            for (int k = 0; k < N; ++k) {
                gv[k] = ld_stream<4>(g + row0 + uint64_t(k) * V + v);
                xv[k] = ld_stream<4>(x + row0 + uint64_t(k) * V + v);
            }
            const Words<4> yv = ld_stream<4>(y + t * V + v);
            post_chunk<N, DT>(
                cf, gv, xv, yv, acc,
                [&](int k, const Words<4>& o) { st_stream<4>(grad_x + row0 + uint64_t(k) * V + v, o); },
                [&](const Words<4>& o) { st_stream<4>(grad_y + t * V + v, o); });
        }
        post_fold_and_store<N>(acc, red, grad_post, grad_res, t);
    }
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

template <int N, int DT>
__global__ void __launch_bounds__(kLanes)
post_bwd_element_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ x,
                        const uint16_t* __restrict__ y, const float* __restrict__ post,
                        const float* __restrict__ res, uint16_t* __restrict__ grad_x,
                        uint16_t* __restrict__ grad_y, float* __restrict__ grad_post,
                        float* __restrict__ grad_res, uint64_t T, uint64_t H) {
    constexpr int M = N * N + N;
    __shared__ float red[kGroups][M];
    __shared__ float coef[M];
    pdl_enter();
    const uint32_t j = threadIdx.x;
    const uint64_t C = (H + 7) / 8;
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
        PostCoeffs<N> cf;
        cf.load(post, res, t, coef);
        float acc[M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = 0.0f;
        const uint64_t row0 = uint64_t(N) * t * H;
        for (uint64_t c = j; c < C; c += kLanes) {
            Words<4> gv[N], xv[N];
#pragma unroll
            for (int k = 0; k < N; ++k) {
                gv[k] = ld_chunk2(g + row0 + uint64_t(k) * H, 8 * c, H);
                xv[k] = ld_chunk2(x + row0 + uint64_t(k) * H, 8 * c, H);
            }
            const Words<4> yv = ld_chunk2(y + t * H, 8 * c, H);
            post_chunk<N, DT>(
                cf, gv, xv, yv, acc,
                [&](int k, const Words<4>& o) { st_chunk2(grad_x + row0 + uint64_t(k) * H, 8 * c, H, o); },
                [&](const Words<4>& o) { st_chunk2(grad_y + t * H, 8 * c, H, o); });
        }
        post_fold_and_store<N>(acc, red, grad_post, grad_res, t);
    }
}

}  // namespace mhc
