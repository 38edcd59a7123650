"""Planted mistakes in copies of the CPU oracle must each fail at least one pin.

Every mutant below is a plausible slip (a wrong tree, a dropped term, a wrong
index, a fused multiply-add, a different rounding) applied to a copy of
``oracle/mhc_oracle.c`` in a temporary directory.  The copy is compiled with the
oracle's own flags and run through the pin checks of ``_pins``; the test passes
when some check rejects it.  This shows the pins constrain the oracle, not just
agree with it.  Nothing here touches the oracle that the other tests use.
"""

import os

import pytest

import oracle
import _pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mhc_oracle.c")

GROUP_TREE = """    for (int stride = ORDER_GROUP / 2; stride >= 1; stride /= 2) {
        for (int i = 0; i < stride; ++i) a[i] = a[i] + a[i + stride];
    }
    return a[0];"""

GROUPS_TREE = """    for (int stride = ORDER_GROUPS / 2; stride >= 1; stride /= 2) {
        for (int i = 0; i < stride; ++i) w[i] = w[i] + w[i + stride];
    }
    return w[0];"""

CHUNK_TREE = """    float a01 = q[0] + q[1];
    float a23 = q[2] + q[3];
    float a45 = q[4] + q[5];
    float a67 = q[6] + q[7];
    float a0123 = a01 + a23;
    float a4567 = a45 + a67;
    return a0123 + a4567;"""

FWD_TREE = """    float s01 = p0 + p1;
    float s23 = p2 + p3;
    float s = s01 + s23;"""

MUTANTS = {
    # forward
    "fwd_left_to_right": (FWD_TREE, "    float s = ((p0 + p1) + p2) + p3;"),
    "fwd_pairs_02_13": (FWD_TREE, "    float s = (p0 + p2) + (p1 + p3);"),
    "fwd_fma": ("    float s01 = p0 + p1;",
                "    float s01 = __builtin_fmaf(pre[0], oracle_float_from_bf16(r[0]), p1);"),
    "fwd_layout_k_major": ("r[k] = residual[(t * 4 + k) * H + h];",
                           "r[k] = residual[(k * T + t) * H + h];"),
    "fwd_wrong_pre_component": ("float p0 = pre[0] *", "float p0 = pre[1] *"),
    "fwd_dropped_term": ("float s23 = p2 + p3;", "float s23 = p2;"),
    "fwd_flush_subnormal": ("    return oracle_bf16_from_float(s);\n}",
                            "    return oracle_bf16_from_float((s < 1.17549435e-38f && "
                            "s > -1.17549435e-38f) ? 0.0f : s);\n}"),
    # BF16 rounding
    "bf16_truncate": ("        kept += 1u;", "        kept += 0u;"),
    "bf16_ties_away": ("(dropped == 0x8000u && (kept & 1u) != 0u)", "(dropped == 0x8000u)"),
    "bf16_ties_down": ("(dropped == 0x8000u && (kept & 1u) != 0u)", "(0)"),
    # grad_residual
    "gr_pre_rounded_first": (
        "float prod = p * oracle_float_from_bf16(g[t * H + h]);",
        "float prod = oracle_float_from_bf16(oracle_bf16_from_float(p)) * "
        "oracle_float_from_bf16(g[t * H + h]);"),
    "gr_wrong_k": ("float p = pre[t * 4 + k];", "float p = pre[t * 4 + (3 - k)];"),
    # grad_pre
    "gp_lanes_128": ("ORDER_LANES = 256", "ORDER_LANES = 128"),
    "gp_chunk_sequential": (CHUNK_TREE, "    float s = q[0];\n"
                            "    for (int e = 1; e < ORDER_CHUNK; ++e) s = s + q[e];\n"
                            "    return s;"),
    "gp_chunk_stride4": (CHUNK_TREE, "    return ((q[0] + q[4]) + (q[1] + q[5])) + "
                         "((q[2] + q[6]) + (q[3] + q[7]));"),
    "gp_group_adjacent_first": (GROUP_TREE, """    for (int stride = 1; stride < ORDER_GROUP; stride *= 2) {
        for (int i = 0; i + stride < ORDER_GROUP; i += 2 * stride) a[i] = a[i] + a[i + stride];
    }
    return a[0];"""),
    "gp_group_sequential": (GROUP_TREE, """    float s = a[0];
    for (int i = 1; i < ORDER_GROUP; ++i) s = s + a[i];
    return s;"""),
    "gp_groups_sequential": (GROUPS_TREE, """    float s = w[0];
    for (int i = 1; i < ORDER_GROUPS; ++i) s = s + w[i];
    return s;"""),
    "gp_lane_descending": ("for (int64_t c = 0; c < C; ++c) {",
                           "for (int64_t c = C - 1; c >= 0; --c) {"),
    "gp_drop_ragged_tail": ("int64_t C = (H + ORDER_CHUNK - 1) / ORDER_CHUNK;",
                            "int64_t C = H / ORDER_CHUNK;"),
    "gp_wrong_row": ("residual + (t * 4 + k) * H, H);", "residual + (t * 4 + (k ^ 1)) * H, H);"),
    "gp_lane_starts_at_first_partial": (
        "lane[j] = lane[j] + chunk_partial(q);",
        "lane[j] = (c < ORDER_LANES) ? chunk_partial(q) : lane[j] + chunk_partial(q);"),
    "gp_fma_products": ("lane[j] = lane[j] + chunk_partial(q);",
                        "lane[j] = __builtin_fmaf(1.0f + 0x1p-23f, chunk_partial(q), lane[j]);"),
    # FP16 storage and the general stream count
    "f16_truncate": ("    if (rem > half || (rem == half && (kept & 1u) != 0u)) kept += 1u;\n",
                     "    (void)half;\n"),
    "f16_ties_away": ("(rem == half && (kept & 1u) != 0u)", "(rem == half)"),
    "f16_flush_subnormal_results": ("if (subnormal) return (uint16_t)(sign | kept);",
                                    "if (subnormal) return sign;"),
    "f16_saturate_instead_of_inf": ("    if (biased >= 31) return (uint16_t)(sign | 0x7C00u);",
                                    "    if (biased >= 31) return (uint16_t)(sign | 0x7BFFu);"),
    "f16_widen_subnormal_off_by_one": ("            e -= 1u;\n        }", "            e -= 2u;\n        }"),
    "hc_tree_sequential": ("        for (int i = 0; i < width / 2; ++i) p[i] = p[2 * i] + p[2 * i + 1];\n    }\n    return p[0];",
                           "    }\n    for (int i = 1; i < n; ++i) p[0] = p[0] + p[i];\n    return p[0];"),
    "hc_tree_stride_pairs": ("p[i] = p[2 * i] + p[2 * i + 1];", "p[i] = p[i] + p[i + width / 2];"),
    "hc_wrong_pre_stride": ("p[k] = pre[t * n + k] * widen(", "p[k] = pre[t * 4 + (k & 3)] * widen("),
    # the fused pre coefficients (sigmoid of alpha * mix + b)
    "exp_one_part_ln2": ("float r = (x - hi) - lo;", "float r = x - hi;"),
    "exp_k_truncated": ("float k = round_half_even(x * EXP_LOG2E);",
                        "float k = (float)(int32_t)(x * EXP_LOG2E);"),
    "exp_ties_away": ("(frac == 0.5f && (n & 1))", "(frac == 0.5f)"),
    "exp_negative_ties_away": ("(frac == -0.5f && (n & 1))", "(frac == -0.5f)"),
    "exp_dropped_taylor_term": ("float q = c[7];", "float q = 0.0f;"),
    "exp_wrong_coefficient": ("1.0f / 6.0f", "1.0f / 5.0f"),
    "exp_unsplit_scale": ("int32_t k1 = ki / 2;", "int32_t k1 = ki;"),
    "exp_overflow_guard_early": ("    if (x > 89.0f) {", "    if (x > 88.0f) {"),
    "exp_underflow_guard_early": ("if (x < -104.0f) return 0.0f;", "if (x < -87.0f) return 0.0f;"),
    "sigmoid_branch_swapped": ("    if (z >= 0.0f) {\n        *s = big;", "    if (z < 0.0f) {\n        *s = big;"),
    "sigmoid_grad_by_cancellation": ("    return s * t;", "    return s * (1.0f - s);"),
    "sigmoid_one_formula": ("    float a = (z < 0.0f) ? -z : z;", "    float a = z;"),
    "preact_fma": ("    return scaled + b;", "    return __builtin_fmaf(alpha, mix, b) + 0.0f * scaled;"),
    "preact_bias_first_column": ("pre_activation(alpha[0], mix[t * n + k], b[k])",
                                 "pre_activation(alpha[0], mix[t * n + k], b[0])"),
    "bwd_grad_z_uses_sigmoid": ("grad_c[i] * oracle_sigmoid32_grad(z)", "grad_c[i] * oracle_sigmoid32(z)"),
    "bwd_grad_mix_unscaled": ("grad_mix[i] = alpha[0] * grad_z[i];", "grad_mix[i] = grad_z[i];"),
    "bwd_bias_index": ("pre_activation(alpha[0], mix[i], b[i % n])", "pre_activation(alpha[0], mix[i], b[i / n % n])"),
    "param_alpha_without_mix": ("p[k] = grad_z[t * n + k] * mix[t * n + k];", "p[k] = grad_z[t * n + k];"),
    "param_tokens_descending": ("for (int64_t chunk = 0; chunk < chunks; ++chunk) {",
                                "for (int64_t chunk = chunks - 1; chunk >= 0; --chunk) {"),
    "param_drop_ragged_tail": ("int64_t chunks = (T + ORDER_CHUNK - 1) / ORDER_CHUNK;",
                               "int64_t chunks = T / ORDER_CHUNK;"),
    "param_lanes_128": ("int lane = (int)(chunk % ORDER_LANES);", "int lane = (int)(chunk % 128);"),
    # mHC post
    "post_term_inside_tree": ("    float mixed = pairwise_tree(p, (int)n);\n    float lifted = post[t * n + k] * widen(y[t * H + h], dtype);",
                              "    float lifted = post[t * n + k] * widen(y[t * H + h], dtype);\n"
                              "    p[n - 1] = p[n - 1] + lifted; lifted = 0.0f;\n"
                              "    float mixed = pairwise_tree(p, (int)n);"),
    "post_wrong_post_index": ("float lifted = post[t * n + k] *", "float lifted = post[t * n + (k ^ (n > 1))] *"),
    "post_res_transposed": ("p[j] = res[(t * n + k) * n + j] * widen(x[(t * n + j) * H + h], dtype);",
                            "p[j] = res[(t * n + j) * n + k] * widen(x[(t * n + j) * H + h], dtype);"),
    "post_bwd_grad_x_untransposed": ("q[k] = res[(t * n + k) * n + j] * widen(g[(t * n + k) * H + h], dtype);",
                                     "q[k] = res[(t * n + j) * n + k] * widen(g[(t * n + k) * H + h], dtype);"),
    "post_bwd_grad_y_without_post": ("for (int64_t k = 0; k < n; ++k) q[k] = post[t * n + k] * widen(",
                                     "for (int64_t k = 0; k < n; ++k) q[k] = 1.0f * widen("),
    "post_bwd_grad_post_against_x": ("grad_post[t * n + k] = grad_pre_row(g_row, y + t * H, H, dtype);",
                                     "grad_post[t * n + k] = grad_pre_row(g_row, x + (t * n + k) * H, H, dtype);"),
    # mHC post with post = sigmoid(alpha * mix + b)
    "post_sigmoid_fwd_mix_as_post": ("int rc = oracle_post_fwd(x, y, post, res, out, T, n, H, dtype);",
                                     "int rc = oracle_post_fwd(x, y, mix, res, out, T, n, H, dtype);"),
    "post_sigmoid_bwd_mix_as_post": ("int rc = oracle_post_bwd(g, x, y, post, res, grad_x, grad_y, grad_post,",
                                     "int rc = oracle_post_bwd(g, x, y, mix, res, grad_x, grad_y, grad_post,"),
    "post_sigmoid_bwd_outputs_swapped": ("sigmoid_epilogue(grad_post, mix, alpha, b, grad_z, grad_mix, T, n);",
                                         "sigmoid_epilogue(grad_post, mix, alpha, b, grad_mix, grad_z, T, n);"),
    "post_bwd_grad_res_wrong_row": ("grad_res[(t * n + k) * n + j] = grad_pre_row(g_row, x + (t * n + j) * H, H, dtype);",
                                    "grad_res[(t * n + k) * n + j] = grad_pre_row(g_row, x + (t * n + k) * H, H, dtype);"),
    "hc_grad_pre_wrong_row": ("grad_pre_row(g + t * H, residual + (t * n + k) * H, H, dtype)",
                              "grad_pre_row(g + t * H, residual + (t * n + (k ^ 1)) * H, H, dtype)"),
}


def _caught(o) -> list:
    failures = []
    for check in _pins.ALL_CHECKS:
        try:
            check(o)
        except AssertionError as e:
            failures.append(f"{check.__name__}: {str(e)[:80]}")
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mutated), str(tmp_path / "libmutant.so"),
                                 extra_flags=["-Wno-unused-function", "-Wno-unused-variable",
                                              "-Wno-unused-parameter"])
    failures = _caught(oracle.Oracle(lib))
    assert failures, f"mutant {name} passed every pin"
