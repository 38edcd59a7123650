/*
 * mhc_h_aggregate.h -- C ABI of the batch-invariant mHC pre "H Aggregate"
 * library for GB300 (sm_103a).
 *
 * The operation ("Add batch-invariant h_aggregate kernel", RL-Kernel pull
 * request 366, Summary):
 *
 *   residual  [T,4,H]  BF16      pre  [T,4]  FP32      out  [T,H]  BF16
 *   out[t,h] = bf16( (pre[t,0]*r[t,0,h] + pre[t,1]*r[t,1,h])
 *                  + (pre[t,2]*r[t,2,h] + pre[t,3]*r[t,3,h]) )
 *
 * with every product and sum one FP32 round-to-nearest-even operation (no
 * fused multiply-add), the fixed (0 + 1) + (2 + 3) tree, and BF16
 * round-to-nearest-even only at the output (same page, Batch invariance).
 *
 * Its backward (asked for by the reviewer on that page; the page gives no
 * formula, so this is the exact derivative of the one above):
 *
 *   grad_residual[t,k,h] = bf16( fp32(pre[t,k] * g[t,h]) )
 *   grad_pre[t,k]        = sum over h of g[t,h] * r[t,k,h]      (FP32)
 *
 * General form (this library's widening, not on the pages; the calls named
 * mhc_aggregate_*): n streams, n in {1, 2, 4, 8}, residual [T,n,H], pre [T,n],
 * out[t,h] = cvt(tree_n(pre[t,k] * r[t,k,h])), tree_n the balanced pairwise
 * tree of FP32 sums (n = 2: p0+p1; n = 4: the (0+1)+(2+3) above; n = 8:
 * ((p0+p1)+(p2+p3)) + ((p4+p5)+(p6+p7))), with storage BF16 or IEEE binary16
 * (cvt rounds to nearest even, overflow to infinity, subnormals kept); the
 * backward has the same form per stream k.
 *
 * grad_pre is summed in ORDER-256, which depends on H only:
 *   1. q_h = g[t,h] * r[t,k,h] in FP32 (exact: both factors are BF16);
 *   2. chunk c = elements 8c .. 8c+7 (+0.0 past H), partial
 *      ((q0+q1)+(q2+q3)) + ((q4+q5)+(q6+q7));
 *   3. lane j (0..255) starts at +0.0 and adds the partials of chunks
 *      j, j+256, j+512, ... in increasing order;
 *   4. each group of 32 lanes folds with strides 16, 8, 4, 2, 1
 *      (lane i < stride: a_i = a_i + a_(i+stride));
 *   5. the 8 group results fold with strides 4, 2, 1; the first is grad_pre.
 *
 * Determinism contract.  Every output byte depends only on the input bytes of
 * its own token and on H.  Calls on any split of the batch along T, with any
 * pointer alignment, on any stream, give byte-identical results, and repeated
 * calls give identical bytes.  NaN payloads are outside the contract.
 *
 * Layout.  Dense row-major: residual[t][k][h] at element (t*4 + k)*H + h;
 * pre[t][k] at t*4 + k; out and g at t*H + h; grad_residual like residual;
 * grad_pre like pre.  BF16 buffers are 2-byte aligned, FP32 buffers 4-byte
 * aligned.  Any such alignment is accepted: 32-byte-aligned BF16 buffers
 * with H % 16 == 0 take the 32-byte vector path, 16-byte-aligned ones with
 * H % 8 == 0 the 16-byte path; other rows of 64 <= H < 2^30 take the
 * realigned 16-byte path (the forward takes the 4-byte path instead when H is
 * even and the buffers 4-byte aligned), shorter rows the 4- or 2-byte path;
 * all give identical results.
 *
 * Pointers and ownership.  Every data pointer is a DEVICE pointer (or managed
 * memory) allocated and owned by the caller.  The library allocates nothing,
 * keeps no state between calls except a per-thread copy of the last CUDA
 * error code, the per-device record of bounded waits that ran out
 * (mhc_h_aggregate_wait_timeouts) and caches of the device addresses,
 * kernel attributes and driver entry point (the tensor-map encoder) it needs,
 * and its compute calls never synchronise: each
 * enqueues kernels on `stream` (NULL = the legacy default stream) and
 * returns.  Calls are safe from several
 * host threads at once.  Kernels are launched with programmatic stream
 * serialization: they may become resident while the previous kernel in the
 * stream finishes, but touch no memory until it has completed, so stream order
 * is kept for every producer and consumer of the buffers.
 *
 * Errors.  T == 0 returns MHC_OK without launching.  T < 0, H <= 0, a NULL
 * pointer, a misaligned pointer, a size whose byte count overflows int64, or
 * an output that overlaps an input or another output returns
 * MHC_ERR_INVALID_ARG without launching; H / 8 >= 2^31 on a vector path
 * returns MHC_ERR_UNSUPPORTED.  A failed launch returns
 * MHC_ERR_CUDA; the CUDA error code is then available from
 * mhc_h_aggregate_last_cuda_error() on the same thread.  Faults during
 * execution surface, as usual in CUDA, at the caller's next synchronisation.
 */
#ifndef MHC_H_AGGREGATE_H
#define MHC_H_AGGREGATE_H

#include <stdint.h>

/* The library is built with hidden symbol visibility; only the declarations
 * below are exported. */
#if defined(__GNUC__) || defined(__clang__)
#define MHC_API __attribute__((visibility("default")))
#else
#define MHC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t (declared here so that the header does not
 * need the CUDA headers). */
struct CUstream_st;
typedef struct CUstream_st* mhc_stream_t;

typedef enum mhc_status {
    MHC_OK = 0,
    MHC_ERR_INVALID_ARG = 1,
    MHC_ERR_UNSUPPORTED = 2,
    MHC_ERR_CUDA = 3
} mhc_status_t;

/* Kernel path a call takes (returned by the *_path queries). */
typedef enum mhc_path {
    MHC_PATH_NONE = -1,   /* the call would be rejected or launches nothing */
    MHC_PATH_VEC16 = 0,   /* 16-byte loads/stores: H % 8 == 0, buffers 16-byte aligned */
    MHC_PATH_PAIR = 1,    /* 4-byte loads/stores: H even, buffers 4-byte aligned (the
                             backward takes it only for H < 64) */
    MHC_PATH_ELEMENT = 2, /* 2-byte loads/stores: any H and alignment */
    MHC_PATH_VEC32 = 3,   /* 32-byte loads/stores: H % 16 == 0, buffers 32-byte aligned */
    MHC_PATH_SHIFT16 = 4  /* 16-byte loads/stores at each row's own alignment, realigned in
                             registers, for 64 <= H < 2^30 when no vector path applies
                             (the forward leaves even H with 4-byte-aligned buffers to
                             the PAIR path; the backward for n = 4, BF16, pre given,
                             H >= 2041 and grad_residual at the residual's 16-byte
                             offset stages its rows in shared memory with bulk copies) */
} mhc_path_t;

/* Version of this ABI; changes when a declaration here changes. */
MHC_API int32_t mhc_h_aggregate_abi_version(void);

/* Forward ("Add batch-invariant h_aggregate kernel", Summary and Batch
 * invariance).
 *   residual  in   BF16 [T,4,H]
 *   pre       in   FP32 [T,4]
 *   out       out  BF16 [T,H]; every element is written exactly once.
 */
MHC_API mhc_status_t mhc_h_aggregate_fwd(const void* residual, const float* pre, void* out,
                                 int64_t T, int64_t H, mhc_stream_t stream);

/* Backward (same page, reviewer request; formula above): one fused pass.
 *   grad_out       in   BF16 [T,H]    g, the gradient of out
 *   residual       in   BF16 [T,4,H]
 *   pre            in   FP32 [T,4]
 *   grad_residual  out  BF16 [T,4,H]
 *   grad_pre       out  FP32 [T,4]   ORDER-256 sums
 */
MHC_API mhc_status_t mhc_h_aggregate_bwd(const void* grad_out, const void* residual, const float* pre,
                                 void* grad_residual, float* grad_pre,
                                 int64_t T, int64_t H, mhc_stream_t stream);

/* The kernel path mhc_h_aggregate_fwd / _bwd would take for these arguments
 * (no launch, no CUDA call).  MHC_PATH_NONE when the call would be rejected or
 * when T == 0. */
MHC_API mhc_path_t mhc_h_aggregate_fwd_path(const void* residual, const float* pre, const void* out,
                                    int64_t T, int64_t H);
MHC_API mhc_path_t mhc_h_aggregate_bwd_path(const void* grad_out, const void* residual,
                                    const float* pre, const void* grad_residual,
                                    const float* grad_pre, int64_t T, int64_t H);

/* Storage type of residual, out, g and grad_residual (pre and grad_pre are
 * always FP32). */
typedef enum mhc_dtype {
    MHC_DTYPE_BF16 = 0,
    MHC_DTYPE_F16 = 1   /* IEEE binary16 */
} mhc_dtype_t;

/* General forward: n streams (n in {1, 2, 4, 8}; others return
 * MHC_ERR_UNSUPPORTED), BF16 or FP16 storage.  The pages' op is n = 4 with
 * BF16, which is exactly mhc_h_aggregate_fwd.  The paper has only n = 4 / BF16;
 * the tree for other n and the FP16 rounding are this library's reading.
 *   residual  in   [T,n,H] dtype
 *   pre       in   FP32 [T,n]
 *   out       out  [T,H] dtype
 */
MHC_API mhc_status_t mhc_aggregate_fwd(const void* residual, const float* pre, void* out, int64_t T,
                               int32_t n, int64_t H, mhc_dtype_t dtype, mhc_stream_t stream);

/* General backward, same n and dtype rules; n = 4 with BF16 is exactly
 * mhc_h_aggregate_bwd.
 *   grad_out       in   [T,H] dtype
 *   residual       in   [T,n,H] dtype
 *   pre            in   FP32 [T,n]
 *   grad_residual  out  [T,n,H] dtype: cvt(fp32(pre[t,k] * g[t,h]))
 *   grad_pre       out  FP32 [T,n]: ORDER-256 sums of g * r[t,k]
 */
MHC_API mhc_status_t mhc_aggregate_bwd(const void* grad_out, const void* residual, const float* pre,
                               void* grad_residual, float* grad_pre, int64_t T, int32_t n,
                               int64_t H, mhc_dtype_t dtype, mhc_stream_t stream);

/* Kernel path of the general calls (no launch, no CUDA call); the storage type
 * does not change the path. */
MHC_API mhc_path_t mhc_aggregate_fwd_path(const void* residual, const float* pre, const void* out,
                                  int64_t T, int32_t n, int64_t H);
MHC_API mhc_path_t mhc_aggregate_bwd_path(const void* grad_out, const void* residual, const float* pre,
                                  const void* grad_residual, const float* grad_pre, int64_t T,
                                  int32_t n, int64_t H);

/* ---- The pre coefficients computed from the mix --------------------------
 *
 * Source: "perf: fuse mHC coefficient backward epilogue" (Liger-Kernel pull
 * request 1402), Summary: the mHC coefficient backward ends in the
 * derivatives of the pre / post sigmoids, grad_mix, and the gradients of the
 * bias b and of scalar alphas; Risks and Limitations: those two reductions run
 * in a fixed, deterministic order.  The page prints no formula.  This
 * library's reading, for the pre coefficients only:
 *
 *   z[t,k]   = alpha * mix[t,k] + b[k]       (FP32: RN multiply, then RN add)
 *   pre[t,k] = sigmoid(z[t,k])
 *   out      = the general forward above with that pre
 *
 *   grad_z[t,k]   = grad_pre[t,k] * sigmoid'(z[t,k])   (grad_pre: ORDER-256)
 *   grad_mix[t,k] = alpha * grad_z[t,k]
 *   grad_b[k]     = sum over t of grad_z[t,k]
 *   grad_alpha    = sum over t of tree_n(grad_z[t,k] * mix[t,k])
 *
 * The last two are summed over tokens in ORDER-256 with t in place of h
 * (chunks of 8 tokens, +0 past T), so they depend on T and on every token,
 * but on nothing else.
 *
 * The sigmoid is this library's fixed binary32 sequence, so that results are
 * a function of the input bits alone: e = exp32(-|z|) with exp32 the
 * argument reduction of Cody and Waite (x = k ln2 + r, k = the integer
 * nearest RN(x * RN(log2 e)), ties to even, r = (x - k*L1) - k*L2 with
 * L1 = 0x1.62e4p-1, L2 = 0x1.7f7d1cp-20), the degree-7 Taylor polynomial of
 * e^r in Horner form with coefficients RN(1/i!), and the scaling
 * (q * 2^(k/2)) * 2^(k - k/2) (k/2 rounded toward zero); x < -104 gives +0.
 * Then d = 1 + e; for z >= 0 sigmoid = 1/d and 1 - sigmoid = e/d, for z < 0
 * the two swap; sigmoid' = sigmoid * (1 - sigmoid).  Every step is one RN
 * binary32 operation.  sigmoid is within 2.5 ulp and sigmoid' within 4.5 ulp
 * of the exact values.
 *
 * alpha is a DEVICE pointer to one FP32 value and b a DEVICE pointer to n
 * FP32 values; neither may overlap an output.  Other rules as above.
 */

/* pre[t,k] = sigmoid(alpha * mix[t,k] + b[k]) on its own (the same bits as
 * the fused calls compute internally).
 *   mix  in   FP32 [T,n]
 *   pre  out  FP32 [T,n]
 */
MHC_API mhc_status_t mhc_pre_sigmoid(const float* mix, const float* alpha, const float* b,
                                     float* pre, int64_t T, int32_t n, mhc_stream_t stream);

/* Fused forward: out = mhc_aggregate_fwd(residual, sigmoid(alpha * mix + b)),
 * byte for byte, in one kernel (no pre buffer).
 *   residual  in   [T,n,H] dtype
 *   mix       in   FP32 [T,n]
 *   out       out  [T,H] dtype
 * Takes the kernel path mhc_aggregate_fwd_path(residual, mix, out, T, n, H).
 */
MHC_API mhc_status_t mhc_aggregate_sigmoid_fwd(const void* residual, const float* mix,
                                               const float* alpha, const float* b, void* out,
                                               int64_t T, int32_t n, int64_t H, mhc_dtype_t dtype,
                                               mhc_stream_t stream);

/* Fused backward, one kernel.
 *   grad_out       in   [T,H] dtype
 *   residual       in   [T,n,H] dtype
 *   mix            in   FP32 [T,n]
 *   grad_residual  out  [T,n,H] dtype: as mhc_aggregate_bwd with pre = sigmoid(z)
 *   grad_z         out  FP32 [T,n]: grad_pre * sigmoid'(z)
 *   grad_mix       out  FP32 [T,n]: alpha * grad_z
 * Takes the kernel path mhc_aggregate_bwd_path(grad_out, residual, mix,
 * grad_residual, grad_z, T, n, H).
 */
MHC_API mhc_status_t mhc_aggregate_sigmoid_bwd(const void* grad_out, const void* residual,
                                               const float* mix, const float* alpha,
                                               const float* b, void* grad_residual, float* grad_z,
                                               float* grad_mix, int64_t T, int32_t n, int64_t H,
                                               mhc_dtype_t dtype, mhc_stream_t stream);

/* The gradients of b and alpha from the fused backward's grad_z.
 *   grad_z      in   FP32 [T,n]
 *   mix         in   FP32 [T,n]
 *   grad_b      out  FP32 [n]
 *   grad_alpha  out  FP32 [1]
 * T == 0 writes +0 to every output (one launch); grad_z and mix may then be
 * NULL.  One kernel, one block.
 */
MHC_API mhc_status_t mhc_sigmoid_param_grad(const float* grad_z, const float* mix, float* grad_b,
                                            float* grad_alpha, int64_t T, int32_t n,
                                            mhc_stream_t stream);

/* ---- mHC post: the layer output expanded back onto the n streams ----------
 *
 * "Add batch-invariant h_aggregate kernel", Summary, names this stage ("MHC
 * Post") without defining it; "perf: fuse mHC coefficient backward epilogue",
 * Summary, names its post coefficients and the n*n residual-mixing
 * coefficients.  This library's reading (the hyper-connection update), with
 * the rules of the aggregate above:
 *
 *   out[t,k,h] = cvt( tree_n( res[t,k,j] * x[t,j,h] ) + post[t,k] * y[t,h] )
 *
 * every product and sum one RN binary32 operation, the n mixing terms in the
 * balanced pairwise tree, the post term added last.  Its backward:
 *
 *   grad_x[t,j,h]   = cvt( tree_n over k of res[t,k,j] * g[t,k,h] )
 *   grad_y[t,h]     = cvt( tree_n over k of post[t,k] * g[t,k,h] )
 *   grad_res[t,k,j] = sum over h of g[t,k,h] * x[t,j,h]    (ORDER-256)
 *   grad_post[t,k]  = sum over h of g[t,k,h] * y[t,h]      (ORDER-256)
 *
 *   x, out, g, grad_x   [T,n,H] dtype      y, grad_y   [T,H] dtype
 *   post, grad_post     FP32 [T,n]         res, grad_res  FP32 [T,n,n]
 *                                           (row k = output stream k)
 * n in {1, 2, 4, 8}; the other rules (errors, ownership, determinism,
 * alignment) as for the aggregate.  Paths: both calls take 16-byte vectors
 * (MHC_PATH_VEC16) when H % 8 == 0 and every 2-byte buffer is 16-byte
 * aligned, else the 2-byte path (MHC_PATH_ELEMENT).
 */
MHC_API mhc_status_t mhc_post_fwd(const void* x, const void* y, const float* post, const float* res,
                                  void* out, int64_t T, int32_t n, int64_t H, mhc_dtype_t dtype,
                                  mhc_stream_t stream);

MHC_API mhc_status_t mhc_post_bwd(const void* grad_out, const void* x, const void* y,
                                  const float* post, const float* res, void* grad_x, void* grad_y,
                                  float* grad_post, float* grad_res, int64_t T, int32_t n,
                                  int64_t H, mhc_dtype_t dtype, mhc_stream_t stream);

/* The mHC post with its post coefficients computed from their own mix, as
 * the pre coefficients are for the aggregate ("perf: fuse mHC coefficient
 * backward epilogue", Summary, names the post sigmoid's derivative beside
 * the pre one):
 *
 *   post[t,k] = sigmoid(z[t,k]),  z[t,k] = RN(RN(alpha * mix[t,k]) + b[k])
 *   (the library's binary32 sigmoid, as for mhc_pre_sigmoid)
 *
 * mhc_post_sigmoid_fwd gives mhc_post_fwd's out at that post.
 * mhc_post_sigmoid_bwd gives mhc_post_bwd's grad_x, grad_y and grad_res, and
 * in place of grad_post grad_z[t,k] = RN(grad_post[t,k] * sigmoid'(z[t,k]))
 * and grad_mix[t,k] = RN(alpha * grad_z[t,k]) (FP32 [T,n]); grad_b and
 * grad_alpha then come from mhc_sigmoid_param_grad(grad_z, mix).  mix is
 * FP32 [T,n], alpha one FP32 value, b FP32 [n]; the other arguments and all
 * rules as for mhc_post_fwd / mhc_post_bwd (mix and grad_z take the places
 * of post and grad_post in the alignment and overlap rules; grad_mix,
 * alpha and b must overlap no output). */
MHC_API mhc_status_t mhc_post_sigmoid_fwd(const void* x, const void* y, const float* mix,
                                          const float* alpha, const float* b, const float* res,
                                          void* out, int64_t T, int32_t n, int64_t H,
                                          mhc_dtype_t dtype, mhc_stream_t stream);

MHC_API mhc_status_t mhc_post_sigmoid_bwd(const void* grad_out, const void* x, const void* y,
                                          const float* mix, const float* alpha, const float* b,
                                          const float* res, void* grad_x, void* grad_y,
                                          float* grad_z, float* grad_mix, float* grad_res,
                                          int64_t T, int32_t n, int64_t H, mhc_dtype_t dtype,
                                          mhc_stream_t stream);

/* Kernel path of mhc_post_fwd / mhc_post_bwd (no launch, no CUDA call); the
 * sigmoid variants take the same path for the same buffers. */
MHC_API mhc_path_t mhc_post_fwd_path(const void* x, const void* y, const float* post,
                                     const float* res, const void* out, int64_t T, int32_t n,
                                     int64_t H);
MHC_API mhc_path_t mhc_post_bwd_path(const void* grad_out, const void* x, const void* y,
                                     const float* post, const float* res, const void* grad_x,
                                     const void* grad_y, const float* grad_post,
                                     const float* grad_res, int64_t T, int32_t n, int64_t H);

/* Static text for a status code. */
MHC_API const char* mhc_status_string(mhc_status_t status);

/* The cudaError_t value behind the last MHC_ERR_CUDA returned on the calling
 * thread; a call that launches successfully resets it to 0. */
MHC_API int32_t mhc_h_aggregate_last_cuda_error(void);

/* Kernels that stream their inputs through shared memory with bulk copies
 * (the mHC post backward on its 16-byte path, and the aggregate backward on
 * its realigned path for n = 4, BF16, pre given, rows of at least 2041
 * values and grad_residual at the residual's 16-byte offset) bound every
 * wait for a copy or for a free stage (1 s of the GPU's global timer), so no
 * wait can hang the GPU.  After a wait runs out the block issues no further
 * copy, waits (again bounded) for the copies it has in flight, and runs to
 * its end.  This returns 1 if a wait ran out on the current device since the
 * previous call, else 0, and clears the record; -1 if a CUDA call fails.  It
 * synchronizes the device.  A return of 1 means that the outputs of every
 * such call on the device since the previous call are invalid. */
MHC_API int64_t mhc_h_aggregate_wait_timeouts(void);

#ifdef __cplusplus
}
#endif

#endif /* MHC_H_AGGREGATE_H */
