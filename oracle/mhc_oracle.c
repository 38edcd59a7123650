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
 *     - Batch invariance: every multiply and add is one binary32
 *       round-to-nearest operation in the fixed (0 + 1) + (2 + 3) tree; the
 *       BF16 inputs are widened exactly, and each output is rounded to BF16
 *       once; each value of a BF16 pair is computed on its own.
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
#include <stdlib.h>
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

/* ----------------------------------------------------------------------- */
/* The pre coefficients from the mix, fused into the aggregate               */
/* ----------------------------------------------------------------------- */

/* Source: "perf: fuse mHC coefficient backward epilogue" (Liger-Kernel pull
 * request 1402), Summary: the coefficient backward ends in the derivatives of
 * the pre / post sigmoids, grad_mix, and FP32 gradients of the bias b (24
 * columns for HC = 4) and of three scalar alphas; Risks and Limitations: the
 * grad_b / alpha reductions run in a fixed, deterministic order instead of
 * eager PyTorch's.  The page prints no formula.  The reading used here, for
 * the pre part only (the post and residual-mixing parts feed other stages):
 *
 *     z[t,k]   = alpha * mix[t,k] + b[k]        RN multiply, then RN add
 *     pre[t,k] = sigmoid(z[t,k]) = 1 / (1 + e^(-z[t,k]))
 *     out      = the aggregate of residual with that pre (as above)
 *
 * and its derivative, with grad_pre[t,k] the ORDER-256 value of the plain
 * backward:
 *
 *     grad_z[t,k]   = grad_pre[t,k] * sigmoid'(z[t,k])
 *     grad_mix[t,k] = alpha * grad_z[t,k]
 *     grad_b[k]     = sum over t of grad_z[t,k]
 *     grad_alpha    = sum over t of tree_n( grad_z[t,k] * mix[t,k] )
 *
 * (24 columns = n pre + n post + n*n residual-mixing columns at n = 4, one
 * alpha per group, which is what the page's counts say).  The two sums over
 * t use ORDER-256 with tokens in place of h (see oracle_sigmoid_param_grad).
 *
 * The page fixes no evaluation of the sigmoid.  To keep every result a fixed
 * function of its inputs on any device, it is defined here as the sequence of
 * binary32 RN operations below (exp32, then sigmoid32), which both this
 * oracle and the CUDA library carry out step for step.
 */

/* Round to the nearest integer, ties to even (|y| < 2^30). */
static float round_half_even(float y) {
    int32_t n = (int32_t)y;                 /* toward zero; exact for |y| < 2^31 */
    float frac = y - (float)n;              /* exact: the dropped fraction */
    if (frac > 0.5f || (frac == 0.5f && (n & 1))) n += 1;
    else if (frac < -0.5f || (frac == -0.5f && (n & 1))) n -= 1;
    return (float)n;
}

/* 2^e as a binary32 value, for -126 <= e <= 127 (built from its fields). */
static float pow2_f32(int32_t e) {
    uint32_t u = (uint32_t)(e + 127) << 23;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* e^x in binary32, defined as this fixed sequence of RN operations:
 *   1. Argument reduction of Cody and Waite (W. J. Cody and W. Waite,
 *      "Software Manual for the Elementary Functions", 1980): x = k ln2 + r
 *      with k = round_half_even(x * log2e) and r = (x - k*L1) - k*L2, where
 *      L1 + L2 is ln 2 split so that L1 has 15 significant bits (k*L1 is then
 *      exact for |k| < 2^9).
 *   2. e^r by its Taylor polynomial of degree 7, sum of r^i / i!, evaluated by
 *      Horner's rule from the highest term: q = c7; q = c_i + r*q for
 *      i = 6 .. 0, with c_i = RN(1 / i!).
 *   3. e^x = (q * 2^(k1)) * 2^(k - k1) with k1 = k / 2 rounded toward zero:
 *      the first product is exact, the second rounds once (also into the
 *      subnormal range).
 * NaN gives NaN, x > 89 gives +inf and x < -104 gives +0 (the correctly
 * rounded values there).  Error: within 1.2 ulp of e^x on [-104, 0]. */
static const float EXP_LOG2E = 0x1.715476p+0f;     /* RN(log2 e) */
static const float EXP_L1 = 0x1.62e4p-1f;          /* ln 2, high part (15 bits) */
static const float EXP_L2 = 0x1.7f7d1cp-20f;       /* RN(ln 2 - L1) */

float oracle_exp32(float x) {
    if (x != x) return x;
    if (x > 89.0f) {
        uint32_t inf = 0x7F800000u;
        float f;
        memcpy(&f, &inf, sizeof f);
        return f;
    }
    if (x < -104.0f) return 0.0f;
    float k = round_half_even(x * EXP_LOG2E);
    float hi = k * EXP_L1;
    float lo = k * EXP_L2;
    float r = (x - hi) - lo;
    const float c[8] = {1.0f, 1.0f, 1.0f / 2.0f, 1.0f / 6.0f, 1.0f / 24.0f, 1.0f / 120.0f,
                        1.0f / 720.0f, 1.0f / 5040.0f};
    float q = c[7];
    for (int i = 6; i >= 0; --i) q = c[i] + r * q;
    int32_t ki = (int32_t)k;
    int32_t k1 = ki / 2;
    float partial = q * pow2_f32(k1);
    return partial * pow2_f32(ki - k1);
}

/* sigmoid(z) and 1 - sigmoid(z), both from e = e^(-|z|) in (0, 1]:
 *   d = 1 + e;  for z >= 0: sigmoid = 1/d, 1 - sigmoid = e/d;
 *               for z <  0: sigmoid = e/d, 1 - sigmoid = 1/d.
 * No term overflows, the small one of the two is never formed by
 * cancellation, and sigmoid(-z) is bit for bit 1 - sigmoid(z) as computed
 * here.  sigmoid'(z) = sigmoid * (1 - sigmoid), one RN product. */
static void sigmoid32(float z, float* s, float* one_minus_s) {
    float a = (z < 0.0f) ? -z : z;
    float e = oracle_exp32(-a);
    float d = 1.0f + e;
    float big = 1.0f / d;
    float small = e / d;
    if (z >= 0.0f) {
        *s = big;
        *one_minus_s = small;
    } else {
        *s = small;
        *one_minus_s = big;
    }
}

float oracle_sigmoid32(float z) {
    float s, t;
    sigmoid32(z, &s, &t);
    return s;
}

float oracle_sigmoid32_grad(float z) {
    float s, t;
    sigmoid32(z, &s, &t);
    return s * t;
}

static float pre_activation(float alpha, float mix, float b) {
    float scaled = alpha * mix;
    return scaled + b;
}

/* pre[t,k] = sigmoid(alpha * mix[t,k] + b[k]); mix and pre are [T,n], b is
 * [n], alpha one value.  Returns 0, or -1 for an unsupported n. */
int oracle_pre_sigmoid(const float* mix, const float* alpha, const float* b, float* pre,
                       int64_t T, int64_t n) {
    if (!valid_streams(n)) return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < n; ++k)
            pre[t * n + k] = oracle_sigmoid32(pre_activation(alpha[0], mix[t * n + k], b[k]));
    return 0;
}

/* The coefficient-gradient epilogue: for coefficients c = sigmoid(z),
 * z = RN(RN(alpha * mix) + b[k]), and the gradient grad_c of a loss with
 * respect to c, grad_z = RN(grad_c * sigmoid'(z)) and
 * grad_mix = RN(alpha * grad_z), all [T,n]. */
static void sigmoid_epilogue(const float* grad_c, const float* mix, const float* alpha,
                             const float* b, float* grad_z, float* grad_mix, int64_t T, int64_t n) {
    for (int64_t i = 0; i < T * n; ++i) {
        float z = pre_activation(alpha[0], mix[i], b[i % n]);
        grad_z[i] = grad_c[i] * oracle_sigmoid32_grad(z);
        grad_mix[i] = alpha[0] * grad_z[i];
    }
}

/* out = aggregate(residual, sigmoid(alpha * mix + b)). */
int oracle_aggregate_sigmoid_fwd(const uint16_t* residual, const float* mix, const float* alpha,
                                 const float* b, uint16_t* out, int64_t T, int64_t n, int64_t H,
                                 int dtype) {
    if (!valid_streams(n) || (dtype != 0 && dtype != 1)) return -1;
    float* pre = (float*)malloc(sizeof(float) * (size_t)(T * n + 1));
    if (!pre) return -2;
    oracle_pre_sigmoid(mix, alpha, b, pre, T, n);
    int rc = oracle_aggregate_fwd(residual, pre, out, T, n, H, dtype);
    free(pre);
    return rc;
}

/* grad_residual as in oracle_aggregate_bwd with pre = sigmoid(z), and
 * grad_z[t,k] = grad_pre[t,k] * sigmoid'(z[t,k]), grad_mix = alpha * grad_z. */
int oracle_aggregate_sigmoid_bwd(const uint16_t* g, const uint16_t* residual, const float* mix,
                                 const float* alpha, const float* b, uint16_t* grad_residual,
                                 float* grad_z, float* grad_mix, int64_t T, int64_t n, int64_t H,
                                 int dtype) {
    if (!valid_streams(n) || (dtype != 0 && dtype != 1)) return -1;
    float* pre = (float*)malloc(sizeof(float) * (size_t)(T * n + 1));
    float* grad_pre = (float*)malloc(sizeof(float) * (size_t)(T * n + 1));
    if (!pre || !grad_pre) {
        free(pre);
        free(grad_pre);
        return -2;
    }
    oracle_pre_sigmoid(mix, alpha, b, pre, T, n);
    int rc = oracle_aggregate_bwd(g, residual, pre, grad_residual, grad_pre, T, n, H, dtype);
    if (rc == 0) sigmoid_epilogue(grad_pre, mix, alpha, b, grad_z, grad_mix, T, n);
    free(pre);
    free(grad_pre);
    return rc;
}

/* Sum of x_0 .. x_(T-1) (x_t = x[t * stride]) in ORDER-256 with tokens in
 * place of h: chunks of 8 consecutive tokens (+0 past T) summed by the chunk
 * tree, lane j adding the partials of chunks j, j + 256, ... in increasing
 * order from +0, then the group and cross-group trees. */
static float order256_over_tokens(const float* x, int64_t stride, int64_t T) {
    float acc[ORDER_LANES];
    for (int j = 0; j < ORDER_LANES; ++j) acc[j] = 0.0f;
    int64_t chunks = (T + ORDER_CHUNK - 1) / ORDER_CHUNK;
    for (int64_t chunk = 0; chunk < chunks; ++chunk) {
        float v[ORDER_CHUNK];
        for (int e = 0; e < ORDER_CHUNK; ++e) {
            int64_t t = chunk * ORDER_CHUNK + e;
            v[e] = (t < T) ? x[t * stride] : 0.0f;
        }
        int lane = (int)(chunk % ORDER_LANES);
        acc[lane] = acc[lane] + chunk_partial(v);
    }
    float w[ORDER_GROUPS];
    for (int grp = 0; grp < ORDER_GROUPS; ++grp) w[grp] = group_tree(acc + grp * ORDER_GROUP);
    return groups_tree(w);
}

/* grad_b[k] = sum_t grad_z[t,k] and grad_alpha[0] = sum_t tree_n(grad_z[t,k] *
 * mix[t,k]), both over tokens in ORDER-256.  Returns 0, -1 for an unsupported
 * n, -2 when out of memory. */
int oracle_sigmoid_param_grad(const float* grad_z, const float* mix, float* grad_b,
                              float* grad_alpha, int64_t T, int64_t n) {
    if (!valid_streams(n)) return -1;
    for (int64_t k = 0; k < n; ++k) grad_b[k] = order256_over_tokens(grad_z + k, n, T);
    float* per_token = (float*)malloc(sizeof(float) * (size_t)(T + 1));
    if (!per_token) return -2;
    for (int64_t t = 0; t < T; ++t) {
        float p[8];
        for (int64_t k = 0; k < n; ++k) p[k] = grad_z[t * n + k] * mix[t * n + k];
        per_token[t] = pairwise_tree(p, (int)n);
    }
    grad_alpha[0] = order256_over_tokens(per_token, 1, T);
    free(per_token);
    return 0;
}

void oracle_exp32_array(const float* x, float* y, int64_t count) {
    for (int64_t i = 0; i < count; ++i) y[i] = oracle_exp32(x[i]);
}

/* s[i] = sigmoid(z[i]), ds[i] = sigmoid'(z[i]). */
void oracle_sigmoid32_array(const float* z, float* s, float* ds, int64_t count) {
    for (int64_t i = 0; i < count; ++i) {
        s[i] = oracle_sigmoid32(z[i]);
        ds[i] = oracle_sigmoid32_grad(z[i]);
    }
}

/* ----------------------------------------------------------------------- */
/* mHC post: the layer output expanded back onto the n residual streams      */
/* ----------------------------------------------------------------------- */

/* Source: "Add batch-invariant h_aggregate kernel", Summary, names the stage
 * ("MHC Post") without defining it; "perf: fuse mHC coefficient backward
 * epilogue", Summary, names its post coefficients (post sigmoid) and the
 * residual-mixing coefficients (the n*n columns) and the "pre/post-residual
 * kernels".  Reading used here (the hyper-connection update; not on the
 * pages), with the pages' rules for the pre aggregate:
 *
 *   out[t,k,h] = cvt( tree_n( res[t,k,j] * x[t,j,h] ) + post[t,k] * y[t,h] )
 *
 * x [T,n,H] the n residual streams, y [T,H] the layer output, post [T,n] and
 * res [T,n,n] FP32 (row k: output stream k; column j: input stream j), out
 * [T,n,H]; every product and sum one RN binary32 operation, the n mixing
 * terms in the balanced pairwise tree, then the post term added last; cvt
 * rounds to the storage type.  The backward is the derivative with the same
 * roundings:
 *
 *   grad_x[t,j,h]   = cvt( tree_n over k of res[t,k,j] * g[t,k,h] )
 *   grad_y[t,h]     = cvt( tree_n over k of post[t,k] * g[t,k,h] )
 *   grad_res[t,k,j] = sum over h of g[t,k,h] * x[t,j,h]    (ORDER-256)
 *   grad_post[t,k]  = sum over h of g[t,k,h] * y[t,h]      (ORDER-256)
 */

static uint16_t post_element(const uint16_t* x, const uint16_t* y, const float* post,
                             const float* res, int64_t t, int64_t k, int64_t h, int64_t n,
                             int64_t H, int dtype) {
    float p[8];
    for (int64_t j = 0; j < n; ++j)
        p[j] = res[(t * n + k) * n + j] * widen(x[(t * n + j) * H + h], dtype);
    float mixed = pairwise_tree(p, (int)n);
    float lifted = post[t * n + k] * widen(y[t * H + h], dtype);
    return narrow(mixed + lifted, dtype);
}

/* Returns 0, or -1 for an unsupported n or dtype (nothing written). */
int oracle_post_fwd(const uint16_t* x, const uint16_t* y, const float* post, const float* res,
                    uint16_t* out, int64_t T, int64_t n, int64_t H, int dtype) {
    if (!valid_streams(n) || (dtype != 0 && dtype != 1)) return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < n; ++k)
            for (int64_t h = 0; h < H; ++h)
                out[(t * n + k) * H + h] = post_element(x, y, post, res, t, k, h, n, H, dtype);
    return 0;
}

int oracle_post_bwd(const uint16_t* g, const uint16_t* x, const uint16_t* y, const float* post,
                    const float* res, uint16_t* grad_x, uint16_t* grad_y, float* grad_post,
                    float* grad_res, int64_t T, int64_t n, int64_t H, int dtype) {
    if (!valid_streams(n) || (dtype != 0 && dtype != 1)) return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t j = 0; j < n; ++j) {
                float q[8];
                for (int64_t k = 0; k < n; ++k)
                    q[k] = res[(t * n + k) * n + j] * widen(g[(t * n + k) * H + h], dtype);
                grad_x[(t * n + j) * H + h] = narrow(pairwise_tree(q, (int)n), dtype);
            }
            float q[8];
            for (int64_t k = 0; k < n; ++k) q[k] = post[t * n + k] * widen(g[(t * n + k) * H + h], dtype);
            grad_y[t * H + h] = narrow(pairwise_tree(q, (int)n), dtype);
        }
        for (int64_t k = 0; k < n; ++k) {
            const uint16_t* g_row = g + (t * n + k) * H;
            grad_post[t * n + k] = grad_pre_row(g_row, y + t * H, H, dtype);
            for (int64_t j = 0; j < n; ++j)
                grad_res[(t * n + k) * n + j] = grad_pre_row(g_row, x + (t * n + j) * H, H, dtype);
        }
    }
    return 0;
}

/* ----------------------------------------------------------------------- */
/* mHC post with its coefficients computed from their own mix               */
/* ----------------------------------------------------------------------- */

/* "perf: fuse mHC coefficient backward epilogue", Summary, names the post
 * sigmoid's derivative next to the pre sigmoid's, with grad_mix and the
 * grad_b / alpha gradients.  Reading used here, as for pre (no other scale
 * is on the pages):
 *
 *   post[t,k] = sigmoid(z[t,k]),  z[t,k] = RN(RN(alpha * mix[t,k]) + b[k])
 *   out       = oracle_post_fwd(x, y, post, res)
 *   grad_z    = RN(grad_post * sigmoid'(z)),  grad_mix = RN(alpha * grad_z)
 *
 * with grad_post from oracle_post_bwd; grad_b and grad_alpha are then
 * oracle_sigmoid_param_grad(grad_z, mix). */
int oracle_post_sigmoid_fwd(const uint16_t* x, const uint16_t* y, const float* mix,
                            const float* alpha, const float* b, const float* res, uint16_t* out,
                            int64_t T, int64_t n, int64_t H, int dtype) {
    if (!valid_streams(n) || (dtype != 0 && dtype != 1)) return -1;
    float* post = (float*)malloc(sizeof(float) * (size_t)(T * n + 1));
    if (!post) return -2;
    oracle_pre_sigmoid(mix, alpha, b, post, T, n);
    int rc = oracle_post_fwd(x, y, post, res, out, T, n, H, dtype);
    free(post);
    return rc;
}

int oracle_post_sigmoid_bwd(const uint16_t* g, const uint16_t* x, const uint16_t* y, const float* mix,
                            const float* alpha, const float* b, const float* res, uint16_t* grad_x,
                            uint16_t* grad_y, float* grad_z, float* grad_mix, float* grad_res,
                            int64_t T, int64_t n, int64_t H, int dtype) {
    if (!valid_streams(n) || (dtype != 0 && dtype != 1)) return -1;
    float* post = (float*)malloc(sizeof(float) * (size_t)(T * n + 1));
    float* grad_post = (float*)malloc(sizeof(float) * (size_t)(T * n + 1));
    if (!post || !grad_post) {
        free(post);
        free(grad_post);
        return -2;
    }
    oracle_pre_sigmoid(mix, alpha, b, post, T, n);
    int rc = oracle_post_bwd(g, x, y, post, res, grad_x, grad_y, grad_post, grad_res, T, n, H, dtype);
    if (rc == 0) sigmoid_epilogue(grad_post, mix, alpha, b, grad_z, grad_mix, T, n);
    free(post);
    free(grad_post);
    return rc;
}
