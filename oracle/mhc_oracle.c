/*
 * CPU oracle for the batch-invariant mHC pre "H Aggregate" collapse and its
 * backward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain definition that the
 * CUDA library is checked against.  Only the test suite, the package smoke
 * check and the CPU-baseline leg of the benchmark may load it.  It shares no
 * code, header, helper or constant with the CUDA path.
 *
 * Build: plain C11, `-O2 -ffp-contract=off`, no fast math.  Every float
 * operation below is one IEEE-754 binary32 operation rounded to nearest even,
 * evaluated in float (FLT_EVAL_METHOD == 0) and never contracted into an FMA.
 * On aarch64 GCC contracts by default, so the flag is required, not cosmetic.
 *
 * Sources (web pages, cited by title and section):
 *   "Add batch-invariant h_aggregate kernel" (RL-Kernel pull request 366)
 *     - Summary: shapes residual [T,4,H] BF16, pre [T,4] FP32, output [T,H]
 *       BF16, and the formula
 *         out = bf16((pre0*r0 + pre1*r1) + (pre2*r2 + pre3*r3)).
 *     - Batch invariance: FP32 round-to-nearest multiplies and adds, the fixed
 *       (0 + 1) + (2 + 3) tree, BF16 conversion only at the input and output
 *       boundaries, the two values of a BF16 pair computed independently.
 *     - Reviewer comment: asks for the backward of h_aggregate (gradient
 *       accuracy and gradient invariance).  The page gives no backward
 *       formula; the one used here is the exact derivative of the Summary
 *       formula, with these roundings:
 *         grad_residual[t,k,h] = bf16( fp32(pre[t,k] * g[t,h]) )
 *         grad_pre[t,k]        = sum over h of g[t,h] * r[t,k,h]  (FP32)
 *       and the FP32 sum taken in ORDER-256 (defined at oracle_grad_pre_token
 *       below), an order that depends on H only.
 *
 * Readings where the page is silent:
 *   - "BF16 conversion" is round-to-nearest, ties to even (RNE) on the upper
 *     16 bits of the binary32 pattern; overflow rounds to infinity.
 *   - Denormals are kept (no flush to zero) on both inputs and results.
 *   - A NaN result is made quiet with its sign kept; NaN payloads are not part
 *     of the contract.
 *
 * Layout: all arrays are dense row-major.  residual[t][k][h] is element
 * (t*4 + k)*H + h; pre[t][k] is element t*4 + k; out and g are [T][H];
 * grad_residual is [T][4][H]; grad_pre is [T][4].  BF16 values are carried as
 * their 16-bit patterns (uint16_t).
 */
#include <float.h>
#include <stdint.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in float (FLT_EVAL_METHOD == 0)"
#endif
#if defined(__FAST_MATH__)
#error "the oracle must not be built with fast math"
#endif

/* ----------------------------------------------------------------------- */
/* BF16 <-> FP32                                                            */
/* ----------------------------------------------------------------------- */

/* A BF16 pattern is the upper half of the binary32 pattern with the same
 * sign, exponent and leading 7 fraction bits, so widening is exact. */
float oracle_float_from_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 value to the nearest BF16 value, ties to even.
 *
 * Written from the definition: keep the upper 16 bits (sign, exponent, 7
 * fraction bits) and look at the 16 discarded bits.  Above half an ulp rounds
 * the magnitude up; exactly half rounds up only when the kept pattern is odd.
 * Because the encoding is sign-magnitude, rounding the magnitude bits is
 * rounding to nearest for either sign, and a carry out of the fraction steps
 * the exponent (the largest finite values round up to infinity). */
uint16_t oracle_bf16_from_float(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t exponent = (u >> 23) & 0xFFu;
    uint32_t fraction = u & 0x7FFFFFu;
    if (exponent == 0xFFu && fraction != 0u) {
        /* NaN: keep sign and the top payload bits, force the quiet bit. */
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u) != 0u)) {
        kept += 1u;
    }
    return (uint16_t)kept;
}

void oracle_bf16_from_float_array(const float* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_bf16_from_float(x[i]);
}

void oracle_float_from_bf16_array(const uint16_t* x, float* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_float_from_bf16(x[i]);
}

/* ----------------------------------------------------------------------- */
/* Forward                                                                  */
/* ----------------------------------------------------------------------- */

/* One output element, exactly as the Summary formula and the Batch invariance
 * rules state: four binary32 products, the (0 + 1) + (2 + 3) tree of binary32
 * sums, one BF16 rounding at the end.  Each operation is its own statement. */
static uint16_t forward_element(const float pre[4], const uint16_t r[4]) {
    float p0 = pre[0] * oracle_float_from_bf16(r[0]);
    float p1 = pre[1] * oracle_float_from_bf16(r[1]);
    float p2 = pre[2] * oracle_float_from_bf16(r[2]);
    float p3 = pre[3] * oracle_float_from_bf16(r[3]);
    float s01 = p0 + p1;
    float s23 = p2 + p3;
    float s = s01 + s23;
    return oracle_bf16_from_float(s);
}

void oracle_h_aggregate_fwd(const uint16_t* residual, const float* pre, uint16_t* out,
                            int64_t T, int64_t H) {
    for (int64_t t = 0; t < T; ++t) {
        const float* pre_t = pre + t * 4;
        for (int64_t h = 0; h < H; ++h) {
            uint16_t r[4];
            for (int64_t k = 0; k < 4; ++k) r[k] = residual[(t * 4 + k) * H + h];
            out[t * H + h] = forward_element(pre_t, r);
        }
    }
}

/* ----------------------------------------------------------------------- */
/* Backward: grad_residual                                                   */
/* ----------------------------------------------------------------------- */

/* d out / d r[t,k,h] = pre[t,k]; the upstream gradient is multiplied in
 * binary32 (one rounding) and the product rounded once more to BF16. */
void oracle_h_aggregate_bwd_grad_residual(const uint16_t* g, const float* pre,
                                          uint16_t* grad_residual, int64_t T, int64_t H) {
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t k = 0; k < 4; ++k) {
            float p = pre[t * 4 + k];
            for (int64_t h = 0; h < H; ++h) {
                float prod = p * oracle_float_from_bf16(g[t * H + h]);
                grad_residual[(t * 4 + k) * H + h] = oracle_bf16_from_float(prod);
            }
        }
    }
}

/* ----------------------------------------------------------------------- */
/* Backward: grad_pre in ORDER-256                                           */
/* ----------------------------------------------------------------------- */

/* ORDER-256, the summation order of grad_pre[t,k] = sum_h g[t,h]*r[t,k,h].
 * It depends on H only: never on T, on how the batch is split, or on any
 * launch shape.
 *
 *   (a) q_h = g[t,h] * r[t,k,h] in binary32.  Both factors are BF16 (8
 *       significant bits), so the product is exact.
 *   (b) Chunks of 8: chunk c covers h = 8c .. 8c+7, for c = 0 .. C-1 with
 *       C = ceil(H/8).  Positions h >= H contribute +0.0f.  The chunk's
 *       partial sum is s_c = ((q0 + q1) + (q2 + q3)) + ((q4 + q5) + (q6 + q7))
 *       with q_e the product at h = 8c + e.
 *   (c) 256 lanes: lane j starts at +0.0f and adds s_c for c = j, j + 256,
 *       j + 512, ... < C, in increasing c:  acc_j = acc_j + s_c.
 *   (d) Eight groups of 32 lanes (group w holds lanes 32w .. 32w+31).  In
 *       each group, for stride 16, 8, 4, 2, 1 in turn, lane i < stride takes
 *       a_i = a_i + a_(i+stride).  The group's value is a_0.
 *   (e) The eight group values W_0 .. W_7: for stride 4, 2, 1 in turn, W_w =
 *       W_w + W_(w+stride) for w < stride.  grad_pre[t,k] = W_0.
 */
enum { ORDER_LANES = 256, ORDER_GROUP = 32, ORDER_GROUPS = ORDER_LANES / ORDER_GROUP,
       ORDER_CHUNK = 8 };

/* Step (b): the binary32 tree over one chunk of 8 products. */
static float chunk_partial(const float q[ORDER_CHUNK]) {
    float a01 = q[0] + q[1];
    float a23 = q[2] + q[3];
    float a45 = q[4] + q[5];
    float a67 = q[6] + q[7];
    float a0123 = a01 + a23;
    float a4567 = a45 + a67;
    return a0123 + a4567;
}

/* Step (d): fold one group of 32 lane values onto its first lane. */
static float group_tree(float a[ORDER_GROUP]) {
    for (int stride = ORDER_GROUP / 2; stride >= 1; stride /= 2) {
        for (int i = 0; i < stride; ++i) a[i] = a[i] + a[i + stride];
    }
    return a[0];
}

/* Step (e): fold the eight group values onto the first. */
static float groups_tree(float w[ORDER_GROUPS]) {
    for (int stride = ORDER_GROUPS / 2; stride >= 1; stride /= 2) {
        for (int i = 0; i < stride; ++i) w[i] = w[i] + w[i + stride];
    }
    return w[0];
}

static float widen(uint16_t v, int dtype);

/* grad_pre[t,k] for one token and one k: g_row is g[t,:], r_row is r[t,k,:],
 * stored as BF16 (dtype 0) or binary16 (dtype 1).  The product of two BF16 or
 * two binary16 values is exact in binary32. */
static float grad_pre_row(const uint16_t* g_row, const uint16_t* r_row, int64_t H, int dtype) {
    float lane[ORDER_LANES];
    for (int j = 0; j < ORDER_LANES; ++j) lane[j] = 0.0f;

    int64_t C = (H + ORDER_CHUNK - 1) / ORDER_CHUNK;
    for (int64_t c = 0; c < C; ++c) {
        float q[ORDER_CHUNK];
        for (int e = 0; e < ORDER_CHUNK; ++e) {
            int64_t h = c * ORDER_CHUNK + e;
            q[e] = (h < H) ? widen(g_row[h], dtype) * widen(r_row[h], dtype) : 0.0f;
        }
        int j = (int)(c % ORDER_LANES);
        lane[j] = lane[j] + chunk_partial(q);
    }

    float w[ORDER_GROUPS];
    for (int grp = 0; grp < ORDER_GROUPS; ++grp) w[grp] = group_tree(lane + grp * ORDER_GROUP);
    return groups_tree(w);
}

static float oracle_grad_pre_token(const uint16_t* g_row, const uint16_t* r_row, int64_t H) {
    return grad_pre_row(g_row, r_row, H, 0);
}

void oracle_h_aggregate_bwd_grad_pre(const uint16_t* g, const uint16_t* residual,
                                     float* grad_pre, int64_t T, int64_t H) {
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t k = 0; k < 4; ++k) {
            grad_pre[t * 4 + k] =
                oracle_grad_pre_token(g + t * H, residual + (t * 4 + k) * H, H);
        }
    }
}

void oracle_h_aggregate_bwd(const uint16_t* g, const uint16_t* residual, const float* pre,
                            uint16_t* grad_residual, float* grad_pre, int64_t T, int64_t H) {
    oracle_h_aggregate_bwd_grad_residual(g, pre, grad_residual, T, H);
    oracle_h_aggregate_bwd_grad_pre(g, residual, grad_pre, T, H);
}

/* ----------------------------------------------------------------------- */
/* General stream count n and FP16 storage                                   */
/* ----------------------------------------------------------------------- */

/* The pages fix n = 4 streams and BF16 storage.  The general form used here
 * (a reading, not on the pages) keeps every rule of the Batch invariance
 * section: for n in {1, 2, 4, 8}
 *     out[t,h] = cvt( tree_n( pre[t,k] * r[t,k,h] ) )
 * where tree_n is the balanced pairwise tree of binary32 sums (n = 2:
 * p0 + p1; n = 4: (p0 + p1) + (p2 + p3); n = 8: ((p0+p1)+(p2+p3)) +
 * ((p4+p5)+(p6+p7))), cvt is round-to-nearest-even into the storage format,
 * and the backward is the derivative with the same roundings and ORDER-256.
 * Storage is BF16 (dtype 0) or IEEE binary16 (dtype 1). */

/* IEEE binary16 -> binary32, exact: normal, subnormal, zero, inf and NaN
 * patterns are rebuilt field by field. */
float oracle_float_from_f16(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t exponent = (h >> 10) & 0x1Fu;
    uint32_t fraction = h & 0x3FFu;
    uint32_t u;
    if (exponent == 0x1Fu) {
        u = sign | 0x7F800000u | (fraction << 13);              /* inf or NaN */
    } else if (exponent != 0u) {
        u = sign | ((exponent + 112u) << 23) | (fraction << 13); /* normal: bias 15 -> 127 */
    } else if (fraction == 0u) {
        u = sign;                                                 /* signed zero */
    } else {
        /* subnormal: fraction * 2^-24, normalised into binary32 */
        uint32_t e = 113u;  /* exponent field of 2^-14 */
        while ((fraction & 0x400u) == 0u) {
            fraction <<= 1;
            e -= 1u;
        }
        u = sign | (e << 23) | ((fraction & 0x3FFu) << 13);
    }
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> IEEE binary16, round to nearest, ties to even.  Written from
 * the definition.  A normal binary32 x is m * 2^(e-23) with a 24-bit
 * significand m.  Its binary16 quantum is 2^(e-10) in the normal range
 * (e >= -14) and 2^-24 below it, so the low `shift` bits of m fall under the
 * quantum: they decide the rounding (above half: up; exactly half: up only to
 * an even count).  A carry can step into the next binade, and results of
 * 65520 (= 2^16 - 2^4) or more become infinity.  Binary32 subnormals are far
 * below 2^-25 and become signed zeros. */
uint16_t oracle_f16_from_float(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t exponent = (u >> 23) & 0xFFu;
    uint32_t fraction = u & 0x7FFFFFu;
    if (exponent == 0xFFu) {
        if (fraction != 0u) return (uint16_t)(sign | 0x7E00u | (fraction >> 13)); /* quiet NaN */
        return (uint16_t)(sign | 0x7C00u);                                        /* inf */
    }
    if (exponent == 0u) return sign;
    int e = (int)exponent - 127;
    if (e >= 16) return (uint16_t)(sign | 0x7C00u);
    if (e <= -26) return sign;                   /* |x| < 2^-25: below half the smallest subnormal */
    uint32_t m = fraction | 0x800000u;
    int subnormal = e < -14;
    int shift = subnormal ? (-1 - e) : 13;       /* 14..24 for subnormal results */
    uint32_t kept = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (kept & 1u) != 0u)) kept += 1u;
    if (subnormal) return (uint16_t)(sign | kept);  /* a carry to 0x400 is the smallest normal */
    int biased = e + 15;
    if (kept == 0x800u) {                        /* rounded up into the next binade */
        kept = 0x400u;
        biased += 1;
    }
    if (biased >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | ((uint32_t)biased << 10) | (kept & 0x3FFu));
}

void oracle_f16_from_float_array(const float* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f16_from_float(x[i]);
}

void oracle_float_from_f16_array(const uint16_t* x, float* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_float_from_f16(x[i]);
}

static float widen(uint16_t v, int dtype) {
    return dtype == 0 ? oracle_float_from_bf16(v) : oracle_float_from_f16(v);
}

static uint16_t narrow(float x, int dtype) {
    return dtype == 0 ? oracle_bf16_from_float(x) : oracle_f16_from_float(x);
}

/* tree_n: level by level, element i of the next level is the sum of elements
 * 2i and 2i+1 of this one, until one value is left. */
static float pairwise_tree(float p[8], int n) {
    for (int width = n; width > 1; width /= 2) {
        for (int i = 0; i < width / 2; ++i) p[i] = p[2 * i] + p[2 * i + 1];
    }
    return p[0];
}

static int valid_streams(int64_t n) { return n == 1 || n == 2 || n == 4 || n == 8; }

/* Returns 0, or -1 for an unsupported n or dtype (nothing written). */
int oracle_aggregate_fwd(const uint16_t* residual, const float* pre, uint16_t* out,
                         int64_t T, int64_t n, int64_t H, int dtype) {
    if (!valid_streams(n) || (dtype != 0 && dtype != 1)) return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            float p[8];
            for (int64_t k = 0; k < n; ++k)
                p[k] = pre[t * n + k] * widen(residual[(t * n + k) * H + h], dtype);
            out[t * H + h] = narrow(pairwise_tree(p, (int)n), dtype);
        }
    }
    return 0;
}

int oracle_aggregate_bwd(const uint16_t* g, const uint16_t* residual, const float* pre,
                         uint16_t* grad_residual, float* grad_pre,
                         int64_t T, int64_t n, int64_t H, int dtype) {
    if (!valid_streams(n) || (dtype != 0 && dtype != 1)) return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t k = 0; k < n; ++k) {
            float p = pre[t * n + k];
            for (int64_t h = 0; h < H; ++h) {
                float prod = p * widen(g[t * H + h], dtype);
                grad_residual[(t * n + k) * H + h] = narrow(prod, dtype);
            }
            grad_pre[t * n + k] = grad_pre_row(g + t * H, residual + (t * n + k) * H, H, dtype);
        }
    }
    return 0;
}
