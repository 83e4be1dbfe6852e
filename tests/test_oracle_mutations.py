"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
never in the product), builds it, points the oracle binding at the mutant and
runs the pins of tests/test_oracle.py: at least one pin must fail.  Every
mutation keeps all memory accesses in bounds.
"""
import ctypes
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.h")

MUTANTS = [
    ("router drops the bias", "if (bias) acc += (double)bias[e];", "(void)bias;"),
    ("router reads W_r transposed", "oracle_bf16_to_double(w_router[(size_t)e * H + h]);",
     "oracle_bf16_to_double(w_router[(size_t)h * E + e]);"),
    ("ties go to the higher index", "    return ia < ib;", "    return ia > ib;"),
    ("softmax denominator without the max shift", "for (int e = 0; e < E; ++e) denom += exp(l[e] - mx);",
     "for (int e = 0; e < E; ++e) denom += exp(l[e]);"),
    ("weights renormalised over the top-k",
     "weight[(size_t)t * k + j] = exp(l[idx[(size_t)t * k + j]] - mx) / denom;",
     "weight[(size_t)t * k + j] = exp(l[idx[(size_t)t * k + j]] - mx) / (denom * 0.0 + 1.0) / "
     "(exp(l[idx[(size_t)t * k]] - mx) + (k > 1 ? exp(l[idx[(size_t)t * k + 1]] - mx) : 0.0));"),
    ("group score is the group's smallest logit", "if (l[e] > best) best = l[e];\n            gscore[g] = best;",
     "if (l[e] < best) best = l[e];\n            gscore[g] = best;"),
    ("group ties go to the higher group", "if (bg < 0 || ranks_before(gscore[g], g, gscore[bg], bg)) bg = g;",
     "if (bg < 0 || ranks_before(gscore[g], -g, gscore[bg], -bg)) bg = g;"),
    ("window keeps one batch too many", "const int first = n_batches > window ? n_batches - window : 0;",
     "const int first = n_batches > window + 1 ? n_batches - window - 1 : 0;"),
    ("expert load ignores its replica", "if (replica_of && replica_of[e] >= 0) acc += slot_window[replica_of[e]];",
     "(void)replica_of;"),
    ("trigger compares the mean", "*trigger = (double)mx * (double)B > threshold * (double)total;",
     "*trigger = (double)total > threshold * (double)total;"),
    ("e4m3 ties round away from zero", "const double m = rint(a * ldexp(1.0, 9));",
     "const double m = round(a * ldexp(1.0, 9));"),
    ("e4m3 normal mantissa truncated", "double m = rint((a * ldexp(1.0, -e) - 1.0) * 8.0);",
     "double m = floor((a * ldexp(1.0, -e) - 1.0) * 8.0);"),
    ("row scale uses the wrong maximum", "const float s = amax > 0.0f ? amax / 448.0f : 1.0f;",
     "const float s = amax > 0.0f ? amax / 240.0f : 1.0f;"),
    ("fp8 gate ignores the token scale", "g *= (double)sx * (double)sg[i];", "g *= (double)sg[i];"),
    ("fp8 down ignores the weight-row scale", "y[o] = acc * (double)sh * (double)sd[o];", "y[o] = acc * (double)sh;"),
    ("fp8 down reads its weights transposed", "dec[qd[(size_t)o * K + i]];",
     "dec[qd[(size_t)i * H + o]];"),
    ("payload scale per row instead of per block",
     "oracle_quantize_blocks_e4m3(1, cols, ORACLE_PAYLOAD_BLOCK, yb, q, sc);",
     "oracle_quantize_blocks_e4m3(1, cols, cols, yb, q, sc);\n        for (int b = 1; b < nb; ++b) sc[b] = sc[0];"),
    ("payload skipped in the E4M3 layer", "oracle_payload_e4m3((int)n, H, yd, yd, y_codes, y_scale);", "(void)n;"),
    ("payload dequantised with the wrong block's scale",
     "oracle_e4m3_decode(q[c]) * (double)sc[c / ORACLE_PAYLOAD_BLOCK];",
     "oracle_e4m3_decode(q[c]) * (double)sc[(c / ORACLE_PAYLOAD_BLOCK + 1) % nb];"),
    ("payload quantised from unrounded values",
     "for (int c = 0; c < cols; ++c) yb[c] = oracle_double_to_bf16(yr[c]);",
     "for (int c = 0; c < cols; ++c) { float f_ = (float)yr[c]; uint32_t b_; memcpy(&b_, &f_, 4); "
     "yb[c] = (uint16_t)(b_ >> 16); }"),
    ("bf16 rounding truncates", "const double r = rint(v / step) * step;", "const double r = trunc(v / step) * step;"),
    ("home slot ignores the replica slots", "return (e / epb) * spb + (e % epb);", "return e;"),
    ("replica used by even tokens", "replica_of[e] >= 0 && (t % 2) == 1", "replica_of[e] >= 0 && (t % 2) == 0"),
    ("dispatch fills slots in reverse order", "for (int a = 0; a < n; ++a) {\n        const int32_t slot = slot_of[a];",
     "for (int a = n - 1; a >= 0; --a) {\n        const int32_t slot = slot_of[a];"),
    ("SiLU of the wrong sign", "static double silu(double v) { return v / (1.0 + exp(-v)); }",
     "static double silu(double v) { return v / (1.0 + exp(v)); }"),
    ("gate and up swapped", "h[i] = silu(g) * u;", "h[i] = silu(u) * g;"),
    ("down projection reads columns reversed",
     "acc += h[i] * oracle_bf16_to_double(w_down[(size_t)o * I + i]);",
     "acc += h[i] * oracle_bf16_to_double(w_down[(size_t)o * I + (I - 1 - i)]);"),
    ("combine drops the shared expert", "out[(size_t)t * H + o] = acc + y_shared[(size_t)t * H + o];",
     "out[(size_t)t * H + o] = acc;"),
    ("combine uses the wrong top-k weight", "acc += weight[(size_t)t * k + j] * y_disp[(size_t)row * H + o];",
     "acc += weight[(size_t)t * k] * y_disp[(size_t)row * H + o];"),
    ("replica plan breaks count ties toward the higher id", "if (best < 0 || counts[e] > counts[best]) best = e;",
     "if (best < 0 || counts[e] >= counts[best]) best = e;"),
    ("replica plan does not halve hot experts",
     "load2[e / epb] += chosen[e] ? (int64_t)counts[e] : 2 * (int64_t)counts[e];",
     "load2[e / epb] += 2 * (int64_t)counts[e];"),
]

PINS = [
    pins.test_bf16_decoding_fixed_patterns,
    lambda: pins.test_router_logits_match_float64_matmul(True),
    pins.test_topk_matches_bruteforce_sort_and_softmax,
    pins.test_topk_tie_rule_hand_cases,
    pins.test_softmax_weights_are_not_renormalised,
    pins.test_grouped_topk_reduces_to_plain_topk,
    pins.test_grouped_topk_keeps_the_best_groups,
    pins.test_grouped_topk_hand_case,
    pins.test_worked_example_block_mapping,
    pins.test_home_slots_of_redundant_layout,
    pins.test_slot_map_replica_parity_and_invalid_ids,
    pins.test_histogram_and_dispatch_invariants,
    pins.test_swiglu_row_matches_torch_float64,
    lambda: pins.test_layer_matches_dense_bruteforce("tiny_k3_2shared"),
    pins.test_replica_plan_rule_on_hand_worked_counts,
    pins.test_replica_plan_hot_list_ties_go_to_lower_id,
    pins.test_replica_plan_falls_back_to_home_block,
    pins.test_replicated_layer_equals_plain_layer_exactly,
    pins.test_e4m3_encoder_special_values,
    pins.test_e4m3_round_trip_and_monotone,
    pins.test_e4m3_encoder_matches_torch_conversion,
    pins.test_row_quantizer_scale_and_error_bound,
    pins.test_bf16_rounding_of_doubles,
    pins.test_fp8_down_row_is_a_scaled_product_of_decoded_codes,
    pins.test_fp8_gate_up_row_reduces_to_bf16_on_exact_values,
    pins.test_fp8_expert_row_is_gate_up_then_bf16_row_quantised_down,
    pins.test_fp8_layer_matches_dense_bruteforce_on_dequantised_tensors,
    pins.test_block_quantizer_matches_torch_per_block,
    pins.test_payload_is_the_bf16_row_block_quantised,
    pins.test_eplb_window_hand_case,
    pins.test_eplb_window_matches_histograms_of_recent_batches,
]


def _build_mutant(tmp, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site not found: {old[:60]}"
    mutated = src.replace(old, new, 1)
    shutil.copy(HDR, tmp)
    c = os.path.join(tmp, "moe_oracle.c")
    so = os.path.join(tmp, "libmutant.so")
    with open(c, "w") as f:
        f.write(mutated)
    subprocess.run(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-o", so, c, "-lm"],
                   check=True)
    lib = ctypes.CDLL(so)
    lib.oracle_home_slot.restype = ctypes.c_int32
    lib.oracle_slot_map.restype = ctypes.c_int
    lib.oracle_moe_forward.restype = ctypes.c_int
    lib.oracle_plan_replicas.restype = ctypes.c_int
    return lib


def test_unmutated_oracle_passes_every_pin():
    for pin in PINS:
        pin()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    oracle.lib()
    saved = oracle._lib
    oracle._lib = _build_mutant(str(tmp_path), old, new)
    failed = []
    try:
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                failed.append(getattr(pin, "__name__", "lambda"))
    finally:
        oracle._lib = saved
    assert failed, f"no pin caught the planted mistake: {name}"
