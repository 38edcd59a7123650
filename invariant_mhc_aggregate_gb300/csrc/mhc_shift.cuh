// The realigned ("shifted") 16-byte paths, for rows of H >= 64 that neither
// a vector path nor the 4-byte pair path can take: odd H, or buffers only
// 2-byte aligned.
//
// A row of 2-byte values that starts `phase` values past a 16-byte boundary
// (phase = (address / 2) mod 8) is covered by the 16-byte-aligned vectors
// m = 0, 1, ..., vector m holding values 8m - phase .. 8m - phase + 7.  Eight
// values at any offset d (0..7) past the start of vector m are the window
// (vector m, vector m + 1) shifted by d values: funnel shifts of 32-bit words,
// with d the same in every thread of a row (no divergence).
//
// Each warp works on 32 consecutive vectors of a row per step: every lane
// loads one with an aligned 16-byte load (streaming), takes its neighbour's
// with warp shuffles, and lanes 0..30 use the window; lane 31 only supplies
// the neighbour of lane 30 (and is lane 0 of the next warp's step, so its
// vector is read twice: 1/31 of the loads, usually from L2).  Outputs are
// written with aligned 16-byte stores when the whole vector lies in the row;
// the at most 7 + 7 values at the row's two ends are computed and stored
// one by one.  Loads stay inside the buffer (a vector not wholly inside it,
// only at the buffer's ends, is read value by value), and no store leaves the
// row.  The data is not staged through shared memory; the only block
// barriers publish a token's sigmoid coefficients (when pre is computed from
// the mix) and fold the backward's lane sums, once per token.
//
// The kernels run the same per-element arithmetic, the same per-lane
// ORDER-256 chunks and the same fold as every other path, so the bytes are
// identical.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mhc {

using Vec16 = Words<4>;

// Values d .. d+7 of the 16-value window lo:hi (value 2i is the low half of
// word i).
template <int D>
__device__ __forceinline__ Vec16 window8_at(const uint32_t (&w)[8]) {
    Vec16 o;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o.w[i] = (D & 1) ? __funnelshift_r(w[D / 2 + i], w[D / 2 + i + 1], 16) : w[D / 2 + i];
    return o;
}

__device__ __forceinline__ Vec16 window8(const Vec16& lo, const Vec16& hi, int d) {
    const uint32_t w[8] = {lo.w[0], lo.w[1], lo.w[2], lo.w[3], hi.w[0], hi.w[1], hi.w[2], hi.w[3]};
    switch (d) {
        case 0: return window8_at<0>(w);
        case 1: return window8_at<1>(w);
        case 2: return window8_at<2>(w);
        case 3: return window8_at<3>(w);
        case 4: return window8_at<4>(w);
        case 5: return window8_at<5>(w);
        case 6: return window8_at<6>(w);
        default: return window8_at<7>(w);
    }
}

__device__ __forceinline__ int row_phase(const void* row) {
    return int((reinterpret_cast<uintptr_t>(row) >> 1) & 7u);
}

__device__ __forceinline__ uint16_t half_of(const Vec16& v, int i) {
    return uint16_t(v.w[i >> 1] >> (16 * (i & 1)));
}

// The buffer a row lives in: [lo, hi) as addresses.
struct Span {
    uintptr_t lo, hi;
};

// The 16 bytes at p (16-byte aligned) that lie inside `buf`, value by value
// (only vectors at the buffer's two ends get here: kept out of line).
static __device__ __noinline__ Vec16 load_vec_clipped(const uint16_t* p, Span buf) {
    Vec16 v = {{0u, 0u, 0u, 0u}};
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uintptr_t e = a + uintptr_t(2 * i);
        if (e >= buf.lo && e + 2 <= buf.hi)
            v.w[i >> 1] |= uint32_t(ld_stream2(reinterpret_cast<const void*>(e))) << (16 * (i & 1));
    }
    return v;
}

__device__ __forceinline__ Vec16 zero16() { return Vec16{{0u, 0u, 0u, 0u}}; }

// A row as the realigned kernels read it: its aligned vector 0 (which starts
// `phase` values before the row), and whether all the vectors that hold a
// row value lie inside the buffer (true for every row but possibly the
// buffer's first and last), in which case its loads need no buffer check.
// Row positions are 32-bit (the path takes H < 2^30).
struct RowRef {
    const uint16_t* v0;
    int phase;
    bool interior;
};

__device__ __forceinline__ RowRef row_ref(const uint16_t* row, int H, Span buf) {
    const int phase = row_phase(row);
    const uintptr_t lo = reinterpret_cast<uintptr_t>(row) - uintptr_t(2 * phase);
    const uintptr_t hi = lo + uintptr_t(16) * uintptr_t((H + phase + 7) / 8);
    return RowRef{reinterpret_cast<const uint16_t*>(lo), phase, lo >= buf.lo && hi <= buf.hi};
}

// Vector m of a row (values 8m - phase .. 8m - phase + 7) if it holds any of
// the row's values 0 .. H-1, else zeros.
__device__ __forceinline__ Vec16 load_vec(const RowRef& r, int m, int H, Span buf) {
    const int first = 8 * m - r.phase;
    if (first >= H || first <= -8) return zero16();
    const uint16_t* p = r.v0 + 8 * m;
    return r.interior ? ld_stream<4>(p) : load_vec_clipped(p, buf);
}

// The window of (own, the next lane's own) at offset d.
__device__ __forceinline__ Vec16 window_next(const Vec16& own, int d) {
    Vec16 nxt;
#pragma unroll
    for (int w = 0; w < 4; ++w) nxt.w[w] = __shfl_down_sync(0xffffffffu, own.w[w], 1);
    return window8(own, nxt, d);
}

// --------------------------------------------------------------------------
// forward: one block per (row segment, token), grid-stride over tokens.  A
// row's output vectors (at most (H + 14) / 8) are cut into segments of
// warps x 31 x U: rows of at least 496 vectors take 8-warp blocks with U = 2
// (segments of 496), shorter rows one block of ceil(vectors / 31) warps with
// U = 1, so that few lanes idle.  Warp w of the block takes the U runs of 31
// consecutive vectors starting at 31*U*w; output vectors that lie partly
// outside the row are computed from the same windows and stored value by
// value.
// --------------------------------------------------------------------------

constexpr int kShiftWarpVectors = 31;   // output vectors per warp and step

__host__ __device__ inline uint64_t shift_row_vectors(uint64_t H) { return (H + 14) / 8; }

template <int N, int DT, int U, class Coeffs>
__global__ void __launch_bounds__(512)
agg_fwd_shift_kernel(const uint16_t* __restrict__ res, Coeffs coeffs, uint16_t* __restrict__ out,
                     uint64_t T, uint64_t H) {
    __shared__ float table[2][N];
    pdl_enter();
    const Span rbuf{reinterpret_cast<uintptr_t>(res), reinterpret_cast<uintptr_t>(res + T * N * H)};
    const int Hi = int(H);
    const uint32_t lane = threadIdx.x & 31u;
    const int wbase = int(blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5)) * kShiftWarpVectors * U;
    int parity = 0;
    for (uint64_t t = blockIdx.y; t < T; t += gridDim.y) {
        uint16_t* orow = out + t * H;
        const int po = row_phase(orow);
        float p[N];
        if constexpr (!Coeffs::kBlockTable) coeffs.template load<N>(t, p);
        int d[N];
        Vec16 own[U][N];
#pragma unroll
        for (int k = 0; k < N; ++k) {
            const RowRef rr = row_ref(res + (uint64_t(N) * t + k) * H, Hi, rbuf);
            const int sh = (rr.phase >= po) ? 0 : -1;   // residual vector m + sh holds out vector m's start
            d[k] = (rr.phase - po) & 7;                  // ... at this offset
#pragma unroll
            for (int u = 0; u < U; ++u)
                own[u][k] = load_vec(rr, wbase + u * kShiftWarpVectors + int(lane) + sh, Hi, rbuf);
        }
        token_pre<N>(coeffs, t, p, table, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            Vec16 x[N];
#pragma unroll
            for (int k = 0; k < N; ++k) x[k] = window_next(own[u][k], d[k]);
            const int m = wbase + u * kShiftWarpVectors + int(lane);
            const int e0 = 8 * m - po;   // row value in lane 0 of output vector m
            if (lane < uint32_t(kShiftWarpVectors) && e0 < Hi && e0 + 8 > 0) {
                Vec16 o;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t w[N];
#pragma unroll
                    for (int k = 0; k < N; ++k) w[k] = x[k].w[e];
                    o.w[e] = agg_pair<N, DT>(p, w);
                }
                if (e0 >= 0 && e0 + 8 <= Hi) {
                    st_stream<4>(orow + e0, o);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (e0 + i >= 0 && e0 + i < Hi) st_stream2(orow + e0 + i, half_of(o, i));
                }
            }
        }
    }
}

// --------------------------------------------------------------------------
// backward: one block per token (grid-stride), 9 warps.  ORDER-256 lane L is
// held by lane L mod 31 of warp L / 31 (lanes 248 .. 255 by warp 8), so that
// each warp's working lanes hold consecutive chunks: in step i, lane l of
// warp w takes chunk c = 31w + l + 256i, and its lane 31 loads chunk
// 31w + 31 + 256i for lane 30's window.  The per-lane sums (each lane adds
// its chunks in increasing order) go through shared memory at the end of the
// token, where warp g folds group g (lanes 32g .. 32g+31) with the usual xor
// shuffles and the 8 group values fold as everywhere else.
// --------------------------------------------------------------------------

constexpr int kShiftBwdWarps = 9;
constexpr int kShiftBwdThreads = 32 * kShiftBwdWarps;

template <int N>
__host__ __device__ constexpr int shift_bwd_batch() { return N >= 8 ? 1 : 2; }

template <int N, int DT, class Coeffs>
__global__ void __launch_bounds__(kShiftBwdThreads)
agg_bwd_shift_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ res,
                     Coeffs coeffs, uint16_t* __restrict__ gres, uint64_t T, uint64_t H) {
    constexpr int B = shift_bwd_batch<N>();
    __shared__ float lanes_acc[kLanes][N];
    __shared__ float red[kGroups][N];
    __shared__ float table[N];    // kBlockTable: the token's pre ...
    __shared__ float slope[N];    // ... and sigmoid' (for the epilogue)
    pdl_enter();
    const Span gbuf{reinterpret_cast<uintptr_t>(g), reinterpret_cast<uintptr_t>(g + T * H)};
    const Span rbuf{reinterpret_cast<uintptr_t>(res), reinterpret_cast<uintptr_t>(res + T * N * H)};
    const int Hi = int(H);
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const int L = int(warp) * kShiftWarpVectors + int(lane);   // ORDER-256 lane (if < 256, lane < 31)
    const bool works = lane < uint32_t(kShiftWarpVectors) && L < kLanes;
    const bool loads = L <= kLanes;   // the working lanes and the next-vector lane of each warp
    const int C = (Hi + 7) / 8;
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const uint16_t* grow = g + t * H;
        const RowRef gref = row_ref(grow, Hi, gbuf);
        const int gph = gref.phase;
        RowRef rref[N];
        uint16_t* orow[N];
        int oph[N], osh[N], od[N];
#pragma unroll
        for (int k = 0; k < N; ++k) {
            rref[k] = row_ref(res + (uint64_t(N) * t + k) * H, Hi, rbuf);
            orow[k] = gres + (uint64_t(N) * t + k) * H;
            oph[k] = row_phase(orow[k]);
            osh[k] = (gph >= oph[k]) ? 0 : 1;    // this window gives grad_residual vector c + osh
            od[k] = (gph - oph[k]) & 7;          // at this offset
        }
        float pk[N];
        float m_own = 0.0f;
        if constexpr (Coeffs::kBlockTable) {
            if (threadIdx.x < N) m_own = coeffs.mix_at(uint64_t(N) * t + threadIdx.x);
        } else {
            coeffs.template load<N>(t, pk);
        }
        bool pk_ready = false;
        float acc[N];
#pragma unroll
        for (int k = 0; k < N; ++k) acc[k] = 0.0f;
        // every thread runs the same number of steps (shuffles); chunks past C are empty
        for (int i0 = 0; i0 * kLanes < C || !pk_ready; i0 += B) {
            Vec16 gv[B], rv[B][N];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int c = L + kLanes * (i0 + b);
                gv[b] = loads ? load_vec(gref, c, Hi, gbuf) : zero16();
#pragma unroll
                for (int k = 0; k < N; ++k) rv[b][k] = loads ? load_vec(rref[k], c, Hi, rbuf) : zero16();
            }
            if (!pk_ready) {
                if constexpr (Coeffs::kBlockTable) {
                    if (threadIdx.x < N)
                        coeffs.pre_and_slope(m_own, int(threadIdx.x), table[threadIdx.x], slope[threadIdx.x]);
                    __syncthreads();
#pragma unroll
                    for (int k = 0; k < N; ++k) pk[k] = table[k];
                } else {
                    coeffs.template to_pre<N>(pk);
                }
                pk_ready = true;
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int c = L + kLanes * (i0 + b);
                const bool live = works && c < C;
                // g realigned to the chunk (values 8c .. 8c+7), +0 past H
                Vec16 gn;
#pragma unroll
                for (int w = 0; w < 4; ++w) gn.w[w] = __shfl_down_sync(0xffffffffu, gv[b].w[w], 1);
                Vec16 gc = window8(gv[b], gn, gph);
                Vec16 rc[N];
#pragma unroll
                for (int k = 0; k < N; ++k) rc[k] = window_next(rv[b][k], rref[k].phase);
                if (8 * c + 8 > Hi) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (8 * c + e >= Hi) {
                            const uint32_t keep = (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
                            gc.w[e >> 1] &= keep;
#pragma unroll
                            for (int k = 0; k < N; ++k) rc[k].w[e >> 1] &= keep;
                        }
                    }
                }
                if (live) {
#pragma unroll
                    for (int k = 0; k < N; ++k) acc[k] = __fadd_rn(acc[k], chunk_partial<DT, 4>(gc, rc[k], 0));
                }
                // grad_residual vectors from g's window at each output row's offset
#pragma unroll
                for (int k = 0; k < N; ++k) {
                    const Vec16 gw = window8(gv[b], gn, od[k]);
                    const int e0 = 8 * (c + osh[k]) - oph[k];
                    if (works && e0 >= 0 && e0 + 8 <= Hi)
                        st_stream<4>(orow[k] + e0, scale_vec<DT, 4>(pk[k], gw));
                }
            }
        }
        // the fold: lane sums to shared memory (then as in every other path);
        // and the values of each grad_residual row that lie in no whole vector
        // ([0, head) and [tail, H), at most 7 + 7), one by one
        if (works) {
#pragma unroll
            for (int k = 0; k < N; ++k) lanes_acc[L][k] = acc[k];
        }
        __syncthreads();
        if (threadIdx.x < 16 * N) {   // threads 16k .. 16k+15 take row k
            const int k = int(threadIdx.x) / 16, s16 = int(threadIdx.x) % 16;
            float pkk = pk[0];   // pk[k] by selects (no dynamic register indexing)
#pragma unroll
            for (int kk = 1; kk < N; ++kk)
                if (kk == k) pkk = pk[kk];
            uint16_t* row = gres + (uint64_t(N) * t + k) * H;
            const int ph = row_phase(row);
            const int64_t head = (8 - ph) & 7;
            int64_t tail = ((int64_t(H) + ph) / 8) * 8 - ph;
            if (tail < head) tail = head;
            const int64_t h = (s16 < 8) ? int64_t(s16) : tail + s16 - 8;
            const bool mine = (s16 < 8) ? (h < head && h < int64_t(H)) : (h < int64_t(H));
            if (mine)
                st_stream2(row + h, Elem<DT>::cvt(__fmul_rn(pkk, Elem<DT>::one(ld_stream2(grow + h)))));
        }
        if (warp < uint32_t(kGroups)) {
            float a[1][N];
#pragma unroll
            for (int k = 0; k < N; ++k) a[0][k] = lanes_acc[threadIdx.x][k];
#pragma unroll
            for (int k = 0; k < N; ++k) {
#pragma unroll
                for (int sft = 16; sft >= 1; sft >>= 1)
                    a[0][k] = __fadd_rn(a[0][k], __shfl_xor_sync(0xffffffffu, a[0][k], sft));
            }
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < N; ++k) red[warp][k] = a[0][k];
            }
        }
        __syncthreads();
        if (threadIdx.x < N) {
            const int k = threadIdx.x;
            float w[kGroups];
#pragma unroll
            for (int i = 0; i < kGroups; ++i) w[i] = red[i][k];
#pragma unroll
            for (int sft = kGroups / 2; sft >= 1; sft >>= 1) {
#pragma unroll
                for (int i = 0; i < sft; ++i) w[i] = __fadd_rn(w[i], w[i + sft]);
            }
            if constexpr (Coeffs::kBlockTable) {
                coeffs.template store_grad_slope<N>(t, k, w[0], slope[k]);
            } else {
                coeffs.template store_grad<N>(t, k, w[0]);
            }
        }
        __syncthreads();   // lanes_acc, red and table are reused by the next token
    }
}

}  // namespace mhc
