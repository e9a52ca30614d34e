"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

Every case edits one spot of ``oracle/moe_oracle.c``, compiles the edited copy
under ``oracle/_build/``, routes the oracle through it, and expects the named
pin test to fail.  A pin set that lets any of these through is too weak.
"""
import os

import pytest

import oracle
import test_oracle_gated as gated
import test_oracle_pins as pins

MUTATIONS = [
    ("nibble_order_swapped",
     "unsigned code = (c % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);",
     "unsigned code = (c % 2 == 0) ? (byte >> 4) : (byte & 0x0Fu);",
     [pins.test_nvfp4_matmul_hand_fixture]),
    ("wrong_scale_block",
     "if (or_e4m3(scales[r * (K / 16) + c / 16], &s) != OR_OK) return OR_ERR_NAN;",
     "if (or_e4m3(scales[r * (K / 16) + ((c / 16) ^ 1)], &s) != OR_OK) return OR_ERR_NAN;",
     [pins.test_nvfp4_matmul_hand_fixture]),
    ("global_dropped_in_matmul",
     "double h = g * acc;",
     "double h = acc;",
     [pins.test_nvfp4_matmul_hand_fixture]),
    ("global_doubled_in_matmul",
     "double h = g * acc;",
     "double h = 2.0 * g * acc;",
     [pins.test_nvfp4_matmul_hand_fixture]),
    ("relu_instead_of_relu_squared",
     "out_bf16[m * N + j] = or_bf16_from_double(r * r);",
     "out_bf16[m * N + j] = or_bf16_from_double(r);",
     [pins.test_nvfp4_matmul_hand_fixture]),
    ("bf16_truncates",
     "if (frac > 0.5) r = fl + 1.0;",
     "if (0) r = fl + 1.0;",
     [pins.test_bf16_rounding_matches_exact_rationals]),
    ("bf16_ties_away_from_zero",
     "else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;",
     "else r = fl + 1.0;",
     [pins.test_bf16_rounding_matches_exact_rationals, pins.test_weighted_row_sum_hand_fixtures]),
    ("routing_not_stable",
     "  for (int64_t p = 0; p < R; ++p) {\n    int32_t e = ids[p];\n    if (e >= 0 && e < E) {\n      int32_t r = fill[e]++;",
     "  for (int64_t p = R - 1; p >= 0; --p) {\n    int32_t e = ids[p];\n    if (e >= 0 && e < E) {\n      int32_t r = fill[e]++;",
     [pins.test_routing_hand_fixtures]),
    ("down_weights_transposed",
     "if (weight_at(dc, ds, I, c, i, &w) != OR_OK)",
     "if (weight_at(dc, ds, I, i, c % I, &w) != OR_OK)",
     [lambda: pins.test_gather_equals_dense_masked(("tiny",))]),
    ("e4m3_subnormals_flushed",
     "double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);",
     "double mag = (e == 0) ? 0.0 : ldexp(1.0 + (double)m / 8.0, (int)e - 7);",
     [pins.test_e4m3_matches_torch_for_every_byte]),
    ("e4m3_sign_ignored",
     "  *out = s ? -mag : mag;",
     "  *out = mag;",
     [pins.test_e4m3_matches_torch_for_every_byte]),
    ("e2m1_subnormal_wrong",
     "double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);",
     "double mag = (e == 0) ? 1.0 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);",
     [pins.test_e2m1_matches_ocp_table]),
    ("dst_not_added",
     "      double acc = or_bf16_to_double(dst[t * H + c]);",
     "      double acc = 0.0;",
     [pins.test_single_pair_reduces_to_two_matvecs]),
    ("routing_weight_ignored",
     "acc += (double)topk_w[p] * y[(p - t0 * k) * H + c];",
     "acc += y[(p - t0 * k) * H + c];",
     [lambda: pins.test_gather_equals_dense_masked(("tiny",))]),
    ("up_global_missing",
     "      h *= (double)up_global[e];",
     "      h *= 1.0;",
     [lambda: pins.test_gather_equals_dense_masked(("tiny",))]),
    ("relu_dropped_in_layer",
     "        double r = h > 0.0 ? h : 0.0;\n        av = r * r;",
     "        double r = h;\n        av = r * r;",
     [pins.test_all_negative_preactivations_leave_dst_unchanged]),
    ("router_ties_to_higher_index",
     "        if (best < 0 || z > best_z) {",
     "        if (best < 0 || z >= best_z) {",
     [pins.test_router_hand_fixture_with_ties_and_bias]),
    ("router_bias_ignored",
     "        const float z = bias ? row[e] + bias[e] : row[e];",
     "        const float z = row[e];",
     [pins.test_router_hand_fixture_with_ties_and_bias]),
    ("router_weights_not_normalised",
     "    for (int j = 0; j < k; ++j) w[t * k + j] = (float)(exp(zp[j] - zp[0]) / sum);",
     "    for (int j = 0; j < k; ++j) w[t * k + j] = (float)(exp(zp[j] - zp[0]));",
     [pins.test_router_closed_forms]),
    ("gate_and_up_swapped",
     "av = gv / (1.0 + exp(-gv)) * h;",
     "av = h / (1.0 + exp(-h)) * gv;",
     [gated.test_large_positive_gate_passes_the_up_projection, gated.test_silu_odd_part_is_the_product]),
    ("logistic_sign_flipped",
     "av = gv / (1.0 + exp(-gv)) * h;",
     "av = gv / (1.0 + exp(gv)) * h;",
     [gated.test_logistic_points_from_fixture, gated.test_large_positive_gate_passes_the_up_projection]),
    ("gelu_instead_of_silu",
     "av = gv / (1.0 + exp(-gv)) * h;",
     "av = gv * 0.5 * (1.0 + erf(gv / sqrt(2.0))) * h;",
     [gated.test_logistic_points_from_fixture]),
    ("gate_global_dropped",
     "gv *= (double)gate_global[e];",
     "gv *= 1.0;",
     [gated.test_large_positive_gate_passes_the_up_projection]),
    ("gate_reads_up_weights",
     "if (weight_at(gc, gs, H, i, c, &w) != OR_OK)",
     "if (weight_at(uc, us, H, i, c, &w) != OR_OK)",
     [gated.test_large_positive_gate_passes_the_up_projection,
      lambda: gated.test_gated_gather_equals_dense_masked((5, 64, 32, 4, 3, 51))]),
]


@pytest.mark.parametrize("name,old,new,catchers", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, catchers):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = oracle.build_variant(src.replace(old, new), name)
    try:
        with oracle.use_library(path):
            for catch in catchers:
                with pytest.raises((AssertionError, ValueError)):
                    catch()
    finally:
        os.remove(path)  # the loaded copy stays mapped; only the file goes
    # the unmutated oracle still passes the same pins
    for catch in catchers:
        catch()
