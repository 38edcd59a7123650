// The realigned ("shifted") 16-byte paths, for rows of 64 <= H < 2^30 that
// no vector path can take (H not a multiple of 8, odd H included, or buffers
// not 16-byte aligned).  The forward leaves even H with 4-byte-aligned
// buffers to the 4-byte pair kernel, which is faster there.
//
// A row of 2-byte values that starts `phase` values past a 16-byte boundary
// (phase = (address / 2) mod 8) is covered by the 16-byte-aligned vectors
// m = 0, 1, ..., vector m holding values 8m - phase .. 8m - phase + 7.  Eight
// values at any offset d (0..7) past the start of vector m are the window
// (vector m, vector m + 1) shifted by d values: funnel shifts of 32-bit words,
// with d the same in every thread of a row (no divergence).
//
// The forward works on 32 consecutive vectors of a row per warp and step:
// every lane loads one (streaming), takes its neighbour's with warp
// shuffles, and lanes 0..30 use the window; lane 31 only supplies lane 30's
// neighbour (and is lane 0 of the next run, so 1/31 of the vectors are read
// twice, mostly from L2).  The backward keeps ORDER-256's one-lane-per-thread
// layout: each lane loads both aligned vectors of its chunk's windows with
// L1-allocating loads, the second being the next lane's first, so a warp's
// second load instruction finds its lines in L1 (or in flight there).
// Measured at H = 7167: shuffles are faster for the forward (46 against
// 55 us), paired loads for the backward (87 against 97 us; the shuffle
// version also needed a 9-warp block and a shared-memory fold).  For the
// pages' operation (n = 4, BF16, pre given) the forward fixes its window
// offsets at compile time (42.8 us), and the backward, when grad_residual
// sits at the residual's 16-byte offset and rows hold at least 256 chunks,
// is the bulk-copy kernel of mhc_shift_bulk.cuh (84.7 us).
// Outputs are written with aligned 16-byte stores when the whole vector lies
// in the row; the at most 7 + 7 values at the row's two ends are computed and
// stored one by one.  Loads stay inside the buffer (a vector not wholly
// inside it, only at the buffer's ends, is read value by value), and no store
// leaves the row.  These kernels do not stage data through shared memory;
// the only block barriers publish a token's sigmoid coefficients (when pre
// is computed from the mix) and fold the backward's lane sums, once per
// token.
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

// 16 bytes through the read-only path, allocating in L1 (the next lane loads
// the same vector as the second half of its window).
__device__ __forceinline__ Vec16 ld_l1_line(const void* p) {
    Vec16 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
    return v;
}

// Vector m of a row (values 8m - phase .. 8m - phase + 7) if it holds any of
// the row's values 0 .. H-1, else zeros: streaming (L1 = false: the forward,
// which passes vectors between lanes with shuffles) or L1-allocating (L1 =
// true: the backward, whose lanes load both vectors of their windows).
template <bool L1>
__device__ __forceinline__ Vec16 load_vec(const RowRef& r, int m, int H, Span buf) {
    const int first = 8 * m - r.phase;
    if (first >= H || first <= -8) return zero16();
    const uint16_t* p = r.v0 + 8 * m;
    if (!r.interior) return load_vec_clipped(p, buf);
    return L1 ? ld_l1_line(p) : ld_stream<4>(p);
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

// The window of (own, the next lane's own) at a compile-time offset D.
template <int D>
__device__ __forceinline__ Vec16 window_next_at(const Vec16& own) {
    Vec16 nxt;
#pragma unroll
    for (int w = 0; w < 4; ++w) nxt.w[w] = __shfl_down_sync(0xffffffffu, own.w[w], 1);
    const uint32_t w8[8] = {own.w[0], own.w[1], own.w[2], own.w[3], nxt.w[0], nxt.w[1], nxt.w[2], nxt.w[3]};
    return window8_at<D>(w8);
}

// The offset of row k's windows, two ways: read at run time (RuntimeWindows:
// each window a switch over the 8 offsets), or fixed at compile time from
// the token's first offset D0 and the rows' phase step H8 = H mod 8 (row k of
// a token starts k*H values after row 0, so its offset is D0 + k*H8 mod 8).
struct RuntimeWindows {
    const int* d;
    __device__ __forceinline__ Vec16 operator()(const Vec16& own, int k) const { return window_next(own, d[k]); }
};

template <int H8, int D0>
struct FixedWindows {
    // k is a constant once the callers' loops are unrolled, and the switch folds
    __device__ __forceinline__ Vec16 operator()(const Vec16& own, int k) const {
        switch (k) {
            case 0: return window_next_at<D0 & 7>(own);
            case 1: return window_next_at<(D0 + H8) & 7>(own);
            case 2: return window_next_at<(D0 + 2 * H8) & 7>(own);
            case 3: return window_next_at<(D0 + 3 * H8) & 7>(own);
            case 4: return window_next_at<(D0 + 4 * H8) & 7>(own);
            case 5: return window_next_at<(D0 + 5 * H8) & 7>(own);
            case 6: return window_next_at<(D0 + 6 * H8) & 7>(own);
            default: return window_next_at<(D0 + 7 * H8) & 7>(own);
        }
    }
};

// One token's output vectors of a warp step: each lane's window of every row,
// the n-term tree, and the store (values of a vector partly outside the row
// one by one).
template <int N, int DT, int U, class Windows>
__device__ __forceinline__ void shift_fwd_outputs(const Vec16 (&own)[U][N], const float (&p)[N], Windows win,
                                                  uint16_t* orow, int po, int wbase, uint32_t lane, int Hi) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        Vec16 x[N];
#pragma unroll
        for (int k = 0; k < N; ++k) x[k] = win(own[u][k], k);
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

// H8 >= 0: the rows' phase step H mod 8 is fixed for the launch, and each
// token's window offsets are dispatched once (on its first row's offset) to
// compile-time windows; H8 < 0: run-time windows.  Compile-time windows
// measured 46.2 -> 43.4 us at T = 4096, H = 7167 (n = 4, BF16); they are
// instantiated for that operation only, to bound the code size.
template <int N, int DT, int U, int H8, class Coeffs>
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
                own[u][k] = load_vec<false>(rr, wbase + u * kShiftWarpVectors + int(lane) + sh, Hi, rbuf);
        }
        token_pre<N>(coeffs, t, p, table, parity);
        if constexpr (H8 < 0) {
            shift_fwd_outputs<N, DT, U>(own, p, RuntimeWindows{d}, orow, po, wbase, lane, Hi);
        } else {
            switch (d[0]) {
                case 0: shift_fwd_outputs<N, DT, U>(own, p, FixedWindows<H8, 0>{}, orow, po, wbase, lane, Hi); break;
                case 1: shift_fwd_outputs<N, DT, U>(own, p, FixedWindows<H8, 1>{}, orow, po, wbase, lane, Hi); break;
                case 2: shift_fwd_outputs<N, DT, U>(own, p, FixedWindows<H8, 2>{}, orow, po, wbase, lane, Hi); break;
                case 3: shift_fwd_outputs<N, DT, U>(own, p, FixedWindows<H8, 3>{}, orow, po, wbase, lane, Hi); break;
                case 4: shift_fwd_outputs<N, DT, U>(own, p, FixedWindows<H8, 4>{}, orow, po, wbase, lane, Hi); break;
                case 5: shift_fwd_outputs<N, DT, U>(own, p, FixedWindows<H8, 5>{}, orow, po, wbase, lane, Hi); break;
                case 6: shift_fwd_outputs<N, DT, U>(own, p, FixedWindows<H8, 6>{}, orow, po, wbase, lane, Hi); break;
                default: shift_fwd_outputs<N, DT, U>(own, p, FixedWindows<H8, 7>{}, orow, po, wbase, lane, Hi); break;
            }
        }
    }
}

// --------------------------------------------------------------------------
// backward: one block per token (grid-stride); thread j is ORDER-256 lane j
// and takes chunks j, j + 256, ... in increasing order, as in every other
// path.  Blocks have 256 threads, or (NARROW), for rows of fewer than 256
// chunks, only the warps that hold chunks (at least 16n threads, for the
// row-end values): the lanes of the missing warps would hold +0, and the fold
// counts them so.  The full-width instance keeps the fold's group count a
// constant (at n = 4 that is 64 registers rather than 70: four blocks per SM
// rather than three).  For chunk c it loads the two aligned vectors of g
// and of each residual row that cover values 8c .. 8c+7 and realigns them;
// g's pair also gives the grad_residual vector c + osh_k of each output row
// k (at that row's offset).  The fold is the common one.
// --------------------------------------------------------------------------

template <int N>
__host__ __device__ constexpr int shift_bwd_batch() { return N >= 4 ? 1 : 2; }

template <int N, int DT, class Coeffs, bool NARROW>
__global__ void __launch_bounds__(kLanes)
agg_bwd_shift_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ res,
                     Coeffs coeffs, uint16_t* __restrict__ gres, uint64_t T, uint64_t H) {
    constexpr int B = shift_bwd_batch<N>();
    __shared__ float red[kGroups][N];
    __shared__ float table[N];    // kBlockTable: the token's pre ...
    __shared__ float slope[N];    // ... and sigmoid' (for the epilogue)
    pdl_enter();
    const Span gbuf{reinterpret_cast<uintptr_t>(g), reinterpret_cast<uintptr_t>(g + T * H)};
    const Span rbuf{reinterpret_cast<uintptr_t>(res), reinterpret_cast<uintptr_t>(res + T * N * H)};
    const int Hi = int(H);
    const int j = int(threadIdx.x);
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
            osh[k] = (gph >= oph[k]) ? 0 : 1;    // g's window gives grad_residual vector c + osh
            od[k] = (gph - oph[k]) & 7;          // at this offset
        }
        float pk[N];
        float m_own = 0.0f;
        if constexpr (Coeffs::kBlockTable) {
            if (j < N) m_own = coeffs.mix_at(uint64_t(N) * t + j);
        } else {
            coeffs.template load<N>(t, pk);
        }
        bool pk_ready = false;
        float acc[1][N];
#pragma unroll
        for (int k = 0; k < N; ++k) acc[0][k] = 0.0f;
        // with a block table the first pass runs in every thread (its loads are
        // guarded) so that all of them meet the barrier that publishes it
        for (int i0 = 0; i0 * kLanes + j < C || !pk_ready; i0 += B) {
            Vec16 glo[B], ghi[B], rlo[B][N], rhi[B][N];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int c = j + kLanes * (i0 + b);
                glo[b] = load_vec<true>(gref, c, Hi, gbuf);
                ghi[b] = load_vec<true>(gref, c + 1, Hi, gbuf);
#pragma unroll
                for (int k = 0; k < N; ++k) {
                    rlo[b][k] = load_vec<true>(rref[k], c, Hi, rbuf);
                    rhi[b][k] = load_vec<true>(rref[k], c + 1, Hi, rbuf);
                }
            }
            if (!pk_ready) {
                if constexpr (Coeffs::kBlockTable) {
                    if (j < N) coeffs.pre_and_slope(m_own, j, table[j], slope[j]);
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
                const int c = j + kLanes * (i0 + b);
                if (c >= C) continue;
                // g and the residual rows realigned to the chunk (values 8c .. 8c+7), +0 past H
                Vec16 gc = window8(glo[b], ghi[b], gph);
                Vec16 rc[N];
#pragma unroll
                for (int k = 0; k < N; ++k) rc[k] = window8(rlo[b][k], rhi[b][k], rref[k].phase);
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
#pragma unroll
                for (int k = 0; k < N; ++k) acc[0][k] = __fadd_rn(acc[0][k], chunk_partial<DT, 4>(gc, rc[k], 0));
                // grad_residual vectors from g's window at each output row's offset
#pragma unroll
                for (int k = 0; k < N; ++k) {
                    const int e0 = 8 * (c + osh[k]) - oph[k];
                    if (e0 >= 0 && e0 + 8 <= Hi)
                        st_stream<4>(orow[k] + e0, scale_vec<DT, 4>(pk[k], window8(glo[b], ghi[b], od[k])));
                }
            }
        }
        // the grad_residual values of each row that lie in no whole vector
        // ([0, head) and [tail, H), at most 7 + 7), one by one: threads
        // 16k .. 16k+15 take row k
        if (threadIdx.x < 16 * N) {
            const int k = j / 16, s16 = j % 16;
            float pkk = pk[0];   // pk[k] by selects (no dynamic register indexing)
#pragma unroll
            for (int kk = 1; kk < N; ++kk)
                if (kk == k) pkk = pk[kk];
            uint16_t* row = gres + (uint64_t(N) * t + k) * H;
            const int ph = row_phase(row);
            const int head = (8 - ph) & 7;
            int tail = ((Hi + ph) / 8) * 8 - ph;
            if (tail < head) tail = head;
            const int h = (s16 < 8) ? s16 : tail + s16 - 8;
            if ((s16 < 8) ? (h < head && h < Hi) : (h < Hi))
                st_stream2(row + h, Elem<DT>::cvt(__fmul_rn(pkk, Elem<DT>::one(ld_stream2(grow + h)))));
        }
        if constexpr (NARROW)
            fold_lanes_and_store<N, 1>(acc, red, coeffs, t, slope, int(blockDim.x / 32));
        else
            fold_lanes_and_store<N, 1>(acc, red, coeffs, t, slope);
    }
}

}  // namespace mhc
