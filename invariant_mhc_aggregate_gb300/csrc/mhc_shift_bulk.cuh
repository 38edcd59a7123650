// The realigned backward with bulk copies, for the pages' operation (n = 4,
// BF16 storage, pre given) on rows of at least 256 chunks whose
// grad_residual buffer sits at the residual's 16-byte offset (as two buffers
// allocated alike do).
//
// The register kernel of mhc_shift.cuh keeps each chunk's ten 16-byte loads
// in registers (two per row: a chunk straddles two aligned vectors), so a
// 64-register thread has one chunk in flight and the kernel waits on DRAM
// latency.  Here a producer thread streams the block's tokens through a
// ring of shared-memory stages with cp.async.bulk: stage (t, s) holds the
// aligned vectors 256s .. 256s + 257 of g's row and 256s .. 256s + 256 of
// each residual row (a row's aligned vector 0 starts on a 16-byte boundary,
// so every copy does; vectors past the row's last one are not copied).  The
// 256 consumer threads are ORDER-256's lanes: thread j reads chunk
// c = 256s + j's vectors from the stage with aligned 16-byte shared loads,
// its warp releases the stage, and the thread computes as the register
// kernel does, with
//  * g's window at run time, over three vectors: chunk c and chunk c + 1 in
//    the chunk grid, widened once;
//  * the residual windows and the grad_residual cuts at compile time: row k
//    of a token starts k*H values after row 0, so with H8 = H mod 8 fixed per
//    launch every row's offset follows from row 0's, and each token is
//    dispatched once on it (grad_residual rows share the residual rows'
//    offsets).  grad_residual vector c + 1 (c when the row's offset is 0) of a
//    row at offset om is values 8 - om .. 15 - om of the 16: a choice of
//    registers.
// Stores go straight to global memory; the at most 7 + 7 values at a
// grad_residual row's two ends that lie in no whole vector are stored one by
// one, from g's values in the first and last stages of the token.  The
// lanes, chunks, products, trees and fold are those of every other path, so
// the bytes are identical.
//
// Copies stay inside the rows' aligned spans.  For the first token those
// begin before the buffers when a buffer starts part-way into a 16-byte
// line, for the last they end past them when one ends part-way: such a
// token's copies leave out the (at most one) vector at each buffer end that
// is not wholly inside it, and its consumers read that vector value by
// value from global memory.
// Waits are bounded as in the other bulk-copy kernels (mhc_bulk.cuh): a wait
// that runs out sets the call's timeout flag, and no copy is issued after it.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mhc_bulk.cuh"

namespace mhc {

// Vectors a stage holds: g's row 258, each residual row 257; each row's
// place is padded to 264 vectors (4224 bytes, a multiple of 128), so that a
// warp's aligned 16-byte reads start on 128-byte lines.
constexpr int kShiftBulkG = kLanes + 8;
constexpr int kShiftBulkR = kLanes + 8;
constexpr int kShiftBulkGUsed = kLanes + 2;
constexpr int kShiftBulkRUsed = kLanes + 1;

template <int N>
__host__ __device__ constexpr uint32_t shift_bulk_stage_bytes() {
    return 16u * uint32_t(kShiftBulkG + N * kShiftBulkR);
}

// Values d .. d+15 of the 24-value window held in words w[0..11].
template <int D>
__device__ __forceinline__ void window16_at(const uint32_t (&w)[12], uint32_t (&o)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        o[i] = (D & 1) ? __funnelshift_r(w[D / 2 + i], w[D / 2 + i + 1], 16) : w[D / 2 + i];
}

__device__ __forceinline__ void window16(const uint32_t (&w)[12], int d, uint32_t (&o)[8]) {
    switch (d) {
        case 0: window16_at<0>(w, o); break;
        case 1: window16_at<1>(w, o); break;
        case 2: window16_at<2>(w, o); break;
        case 3: window16_at<3>(w, o); break;
        case 4: window16_at<4>(w, o); break;
        case 5: window16_at<5>(w, o); break;
        case 6: window16_at<6>(w, o); break;
        default: window16_at<7>(w, o); break;
    }
}

// Whether a token's rows' aligned spans (all the 16-byte vectors holding a
// value of its g row or of its residual rows) reach outside the buffers:
// only the first token when a buffer starts part-way into a 16-byte line,
// and the last when one ends part-way.
template <int N>
__device__ __forceinline__ bool shift_bulk_edge(const uint16_t* grow, const uint16_t* rrow, int H, Span gbuf,
                                                Span rbuf) {
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(grow) & ~uintptr_t(15);
    const uintptr_t g1 = (reinterpret_cast<uintptr_t>(grow + H) + 15) & ~uintptr_t(15);
    const uintptr_t r0 = reinterpret_cast<uintptr_t>(rrow) & ~uintptr_t(15);
    const uintptr_t r1 = (reinterpret_cast<uintptr_t>(rrow + uint64_t(N) * H) + 15) & ~uintptr_t(15);
    return g0 < gbuf.lo || g1 > gbuf.hi || r0 < rbuf.lo || r1 > rbuf.hi;
}

// An aligned vector p of an edge token: the staged copy `v` when it lies in
// the buffer (those are the vectors copied), else read value by value (out
// of line).
__device__ __forceinline__ Vec16 vec_edge(const Vec16& v, const uint16_t* p, Span buf) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return (a >= buf.lo && a + 16 <= buf.hi) ? v : load_vec_clipped(p, buf);
}

// Of `vectors` aligned 16-byte vectors from src, the range [first, last) to
// copy: all of them, or (clip: an edge token) those wholly inside `buf`.
struct CopyRange {
    int first, last;
    __device__ __forceinline__ CopyRange(const uint16_t* src, int vectors, bool clip, Span buf)
        : first(0), last(vectors) {
        if (clip) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(src);
            const uintptr_t lo = (buf.lo + 15) & ~uintptr_t(15), hi = buf.hi & ~uintptr_t(15);
            if (a < lo) first = int((lo - a) / 16);
            if (a + uintptr_t(16) * uintptr_t(vectors) > hi) last = a < hi ? int((hi - a) / 16) : 0;
            if (last < first) last = first;
        }
    }
    __device__ __forceinline__ uint32_t bytes() const { return 16u * uint32_t(last - first); }
};

// The barrier over the 256 consumer threads (named barrier 1).
struct ConsumerSync {
    __device__ __forceinline__ void operator()() const { named_sync(1, kLanes); }
};

// One token's segments, residual row 0 at offset R0 (with k unrolled, every
// residual window and grad_residual cut below is a constant).  ov0: aligned
// vector 0 of grad_residual row 0; rows k start k*H values later.
template <int N, int DT, int H8, int R0, int STAGES, bool EDGE>
__device__ __forceinline__ void shift_bulk_token(const unsigned char* stage_mem, uint64_t* full, uint64_t* empty,
                                                 uint32_t& item, bool& ok, int nseg, const uint16_t* grow,
                                                 const uint16_t* rrow, uint16_t* ov0, Span gbuf, Span rbuf,
                                                 const float (&pk)[N], float (&acc)[N], int Hi, int C, int j) {
    const int gph = row_phase(grow);
#pragma unroll 1
    for (int s = 0; s < nseg; ++s, ++item) {
        const uint32_t st = item % STAGES;
        if (ok) ok = mbar_wait_fast(&full[st], (item / STAGES) & 1u);
        const int c = s * kLanes + j;
        const bool mine = c < C;
        const Vec16* sg = reinterpret_cast<const Vec16*>(stage_mem + size_t(st) * shift_bulk_stage_bytes<N>());
        const Vec16* sr = sg + kShiftBulkG + j;
        float gf[16];
        if (mine) {
            uint32_t gw[12];
#pragma unroll
            for (int v = 0; v < 3; ++v) {
                const Vec16 x = EDGE ? vec_edge(sg[j + v], grow - gph + 8 * (c + v), gbuf) : sg[j + v];
#pragma unroll
                for (int w = 0; w < 4; ++w) gw[4 * v + w] = x.w[w];
            }
            uint32_t gwin[8];
            window16(gw, gph, gwin);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                gf[2 * i] = Elem<DT>::lo(gwin[i]);
                gf[2 * i + 1] = Elem<DT>::hi(gwin[i]);
            }
            const bool tail = 8 * c + 8 > Hi;   // the row's last chunk: products past H are +0
#pragma unroll
            for (int k = 0; k < N; ++k) {
                const int rph = (R0 + k * H8) & 7;
                const uint16_t* rv = rrow + (uint64_t(k) * uint64_t(Hi) - rph) + 8 * c;   // aligned vector c of row k
                const Vec16 rlo = sr[k * kShiftBulkR], rhi = sr[k * kShiftBulkR + 1];
                const Vec16 rc = EDGE ? window8(vec_edge(rlo, rv, rbuf), vec_edge(rhi, rv + 8, rbuf), rph)
                                      : window8(rlo, rhi, rph);
                float q[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    q[2 * i] = __fmul_rn(gf[2 * i], Elem<DT>::lo(rc.w[i]));
                    q[2 * i + 1] = __fmul_rn(gf[2 * i + 1], Elem<DT>::hi(rc.w[i]));
                }
                if (tail) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (8 * c + e >= Hi) q[e] = 0.0f;
                }
                acc[k] = __fadd_rn(acc[k], __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                                                     __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7]))));
            }
        }
        // the grad_residual values of each row that lie in no whole vector
        // ([0, head) and [tail, H), at most 7 each), value by value from g's
        // values in the stage that holds them (segment s's own vectors are
        // 256s .. 256s + 255; the last segment also has its two extra):
        // threads 8k .. 8k + 7 take row k
        if (j < 8 * N) {
            const int k = j / 8, e = j % 8;
            const int om = (R0 + k * H8) & 7;
            float pkk = pk[0];   // pk[k] by selects (no dynamic register indexing)
#pragma unroll
            for (int kk = 1; kk < N; ++kk)
                if (kk == k) pkk = pk[kk];
            const int head = (8 - om) & 7, tail = ((Hi + om) / 8) * 8 - om;
            const uint16_t* sg16 = reinterpret_cast<const uint16_t*>(sg);
            uint16_t* row = ov0 + (uint64_t(k) * uint64_t(Hi) + R0);
            if (s == 0 && e < head)
                st_stream2(row + e, Elem<DT>::cvt(__fmul_rn(pkk, Elem<DT>::one(EDGE ? ld_stream2(grow + e)
                                                                                      : sg16[e + gph]))));
            const int h = tail + e, p = h + gph - 8 * s * kLanes;   // its place in the stage
            if (h < Hi && h >= head && p >= 0 && (p < 8 * kLanes || s == nseg - 1))
                st_stream2(row + h, Elem<DT>::cvt(__fmul_rn(pkk, Elem<DT>::one(EDGE ? ld_stream2(grow + h)
                                                                                      : sg16[p]))));
        }
        // every shared-memory read of this stage is done
        __syncwarp();
        if ((j & 31) == 0) mbar_arrive(&empty[st]);
        if (!mine) continue;
#pragma unroll
        for (int k = 0; k < N; ++k) {
            const int om = (R0 + k * H8) & 7;
            const int sel = om ? 8 - om : 0;   // first of the vector's values in gf
            const int m = c + (om ? 1 : 0);    // its vector in the row
            uint4 o;
            o.x = Elem<DT>::pack(__fmul_rn(pk[k], gf[sel + 0]), __fmul_rn(pk[k], gf[sel + 1]));
            o.y = Elem<DT>::pack(__fmul_rn(pk[k], gf[sel + 2]), __fmul_rn(pk[k], gf[sel + 3]));
            o.z = Elem<DT>::pack(__fmul_rn(pk[k], gf[sel + 4]), __fmul_rn(pk[k], gf[sel + 5]));
            o.w = Elem<DT>::pack(__fmul_rn(pk[k], gf[sel + 6]), __fmul_rn(pk[k], gf[sel + 7]));
            // row k's aligned vector m, an element offset below 2^32 (H < 2^30)
            const uint32_t off = uint32_t(k) * uint32_t(Hi) + uint32_t(R0 - om) + 8u * uint32_t(m);
            if (8 * m - om + 8 <= Hi) __stcs(reinterpret_cast<uint4*>(ov0 + off), o);
        }
    }
}

template <int N, int DT, int H8, int STAGES, int MIN_BLOCKS, class Coeffs>
__global__ void __launch_bounds__(kLanes + 32, MIN_BLOCKS)
agg_bwd_shift_bulk_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ res, Coeffs coeffs,
                          uint16_t* __restrict__ gres, uint64_t T, uint64_t H, unsigned int* __restrict__ timeouts) {
    static_assert(!Coeffs::kBlockTable, "the token's pre is read, not computed");
    extern __shared__ __align__(128) unsigned char stage_mem[];   // STAGES stages
    __shared__ __align__(8) uint64_t full[STAGES];
    __shared__ __align__(8) uint64_t empty[STAGES];
    __shared__ float red[kGroups][N];
    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kLanes / 32);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_enter();
    const int Hi = int(H);
    const int C = (Hi + 7) / 8;
    const int nseg = (C + kLanes - 1) / kLanes;
    const Span gbuf{reinterpret_cast<uintptr_t>(g), reinterpret_cast<uintptr_t>(g + T * H)};
    const Span rbuf{reinterpret_cast<uintptr_t>(res), reinterpret_cast<uintptr_t>(res + T * N * H)};

    if (threadIdx.x >= kLanes) {
        // producer warp: one thread issues the copies
        if (threadIdx.x != kLanes) return;
        bool ok = true;
        uint32_t item = 0, issued = 0;
        for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
            const uint16_t* grow = g + t * H;
            const int gph = row_phase(grow);
            const int gvend = (gph + Hi + 7) / 8;   // aligned vectors holding a value of the row
            const uint16_t* rrow = res + uint64_t(N) * t * H;
            const int r0 = row_phase(rrow);
            const bool edge = shift_bulk_edge<N>(grow, rrow, Hi, gbuf, rbuf);
            for (int s = 0; s < nseg; ++s, ++item) {
                const uint32_t st = item % STAGES, round = item / STAGES;
                if (round > 0 && ok) ok = stage_reusable(full, empty, st, round);
                if (!ok) continue;   // after a wait ran out, no copy is issued
                issued = item + 1;
                const int v0 = s * kLanes;
                unsigned char* dst = stage_mem + size_t(st) * shift_bulk_stage_bytes<N>();
                int gn = gvend - v0 < kShiftBulkGUsed ? gvend - v0 : kShiftBulkGUsed;
                int rn[N];
#pragma unroll
                for (int k = 0; k < N; ++k) {
                    const int rvend = (((r0 + k * H8) & 7) + Hi + 7) / 8;
                    rn[k] = rvend - v0 < kShiftBulkRUsed ? rvend - v0 : kShiftBulkRUsed;
                }
                const uint16_t* src[N + 1];
                src[0] = grow - gph + 8 * v0;
#pragma unroll
                for (int k = 0; k < N; ++k) src[k + 1] = rrow + uint64_t(k) * H - ((r0 + k * H8) & 7) + 8 * v0;
                uint32_t total = 0;
#pragma unroll
                for (int r = 0; r <= N; ++r)
                    total += CopyRange(src[r], r == 0 ? gn : rn[r - 1], edge, r == 0 ? gbuf : rbuf).bytes();
                mbar_arrive_expect_tx(&full[st], total);   // (with no bytes the arrival completes the phase)
#pragma unroll
                for (int r = 0; r <= N; ++r) {
                    const CopyRange cr(src[r], r == 0 ? gn : rn[r - 1], edge, r == 0 ? gbuf : rbuf);
                    unsigned char* d = dst + 16 * (r == 0 ? 0 : kShiftBulkG + (r - 1) * kShiftBulkR);
                    if (cr.bytes() != 0)
                        bulk_copy_g2s(d + 16 * cr.first, src[r] + 8 * cr.first, cr.bytes(), &full[st]);
                }
            }
        }
        // every copy issued has landed before the block's shared memory goes
        for (uint32_t i = issued > uint32_t(STAGES) ? issued - STAGES : 0; i < issued; ++i)
            if (!mbar_wait(&full[i % STAGES], (i / STAGES) & 1u)) ok = false;
        if (!ok) *timeouts = 1u;
        return;
    }

    // consumers: thread j is ORDER-256 lane j
    const int j = int(threadIdx.x);
    bool ok = true;
    uint32_t item = 0;
    for (uint64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const uint16_t* grow = g + t * H;
        const uint16_t* rrow = res + uint64_t(N) * t * H;
        const int r0 = row_phase(rrow);
        uint16_t* ov0 = gres + uint64_t(N) * t * H - r0;
        const bool edge = shift_bulk_edge<N>(grow, rrow, Hi, gbuf, rbuf);
        float pk[N];
        coeffs.template load<N>(t, pk);
        coeffs.template to_pre<N>(pk);
        float acc[1][N];
#pragma unroll
        for (int k = 0; k < N; ++k) acc[0][k] = 0.0f;
        switch (r0) {
            case 0:
                if (edge) shift_bulk_token<N, DT, H8, 0, STAGES, true>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                else shift_bulk_token<N, DT, H8, 0, STAGES, false>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                break;
            case 1:
                if (edge) shift_bulk_token<N, DT, H8, 1, STAGES, true>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                else shift_bulk_token<N, DT, H8, 1, STAGES, false>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                break;
            case 2:
                if (edge) shift_bulk_token<N, DT, H8, 2, STAGES, true>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                else shift_bulk_token<N, DT, H8, 2, STAGES, false>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                break;
            case 3:
                if (edge) shift_bulk_token<N, DT, H8, 3, STAGES, true>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                else shift_bulk_token<N, DT, H8, 3, STAGES, false>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                break;
            case 4:
                if (edge) shift_bulk_token<N, DT, H8, 4, STAGES, true>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                else shift_bulk_token<N, DT, H8, 4, STAGES, false>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                break;
            case 5:
                if (edge) shift_bulk_token<N, DT, H8, 5, STAGES, true>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                else shift_bulk_token<N, DT, H8, 5, STAGES, false>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                break;
            case 6:
                if (edge) shift_bulk_token<N, DT, H8, 6, STAGES, true>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                else shift_bulk_token<N, DT, H8, 6, STAGES, false>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                break;
            default:
                if (edge) shift_bulk_token<N, DT, H8, 7, STAGES, true>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                else shift_bulk_token<N, DT, H8, 7, STAGES, false>(stage_mem, full, empty, item, ok, nseg, grow, rrow, ov0, gbuf, rbuf, pk, acc[0], Hi, C, j);
                break;
        }
        fold_lanes_and_store<N, 1>(acc, red, coeffs, t, nullptr, kGroups, ConsumerSync{});
    }
    if (!ok) *timeouts = 1u;
}

}  // namespace mhc
