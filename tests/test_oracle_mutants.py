"""The pins catch plausible mistakes in the oracle.

Each case plants one plausible mistake in a copy of the oracle's C source (on the CPU; the
library the tests and the CUDA path use is untouched), compiles it, points the oracle binding at
it, and runs a battery of the pin tests: at least one of them must fail. The mistakes are the
kinds a reader of the pages could make: a rounding tie broken the wrong way, the nibble order
swapped, a factor of the scale pick dropped, the global scale left out of the reciprocal or of
the decode, the wrong global-scale constant, no saturation of the block scale, the softmax
scale dropped, the wrong query-head to KV-head map, the LSE in the wrong logarithm, the FP8
workspace copy scaled the wrong way, the two tokens of a token pair swapped, the two-component
(2FP4) residual taken with the wrong sign."""
import numpy as np
import pytest

import oracle
import test_oracle_attention as ta
import test_oracle_codec as tc
import test_oracle_cold as tco
import test_oracle_format as tf

MUTANTS = [
    ("E2M1 ties away from zero",
     [("    double m = round_to_format(fabs(y), 2, 0);",
       "    double m = round_to_format(fabs(y) * (1.0 + 1e-9), 2, 0);")]),
    ("nibble order swapped when packing",
     [("    data[idx] = hi ? (uint8_t)((data[idx] & 0x0F) | (code << 4)) : (uint8_t)((data[idx] & 0xF0) | code);",
       "    data[idx] = !hi ? (uint8_t)((data[idx] & 0x0F) | (code << 4)) : (uint8_t)((data[idx] & 0xF0) | code);"),
      ("    return hi ? (data[idx] >> 4) : (data[idx] & 15);",
       "    return !hi ? (data[idx] >> 4) : (data[idx] & 15);")]),
    ("scale pick divides by 4 g instead of 6 g",
     [("    double d = fp32(6.0 * g);", "    double d = fp32(4.0 * g);")]),
    ("reciprocal of the scale without g",
     [("    double sg = fp32(s * g);", "    double sg = fp32(s);")]),
    ("decode to 16 bits without g",
     [("((uint16_t*)dst)[o] = bf16_bits(bf16_round(fp32(v * g)));",
       "((uint16_t*)dst)[o] = bf16_bits(bf16_round(fp32(v)));")]),
    ("global scale amax / 448",
     [("    double g = fp32(amax / 2688.0);", "    double g = fp32(amax / 448.0);")]),
    ("block scale not saturated at 448",
     [("    if (m > 448.0)\n        m = 448.0;\n", "")]),
    ("softmax scale dropped",
     [("double zt = sm_scale * dot;", "double zt = dot;"),
      ("double w = exp(sm_scale * dot - zmax);", "double w = exp(dot - zmax);")]),
    ("query head h reads KV head h mod H",
     [("            int h = qh / G;", "            int h = qh % H;")]),
    ("LSE in log2",
     [("lse[(size_t)b * Hq + qh] = zmax + log(l);", "lse[(size_t)b * Hq + qh] = zmax + log2(l);")]),
    ("FP8 workspace copy multiplied by ws_scale instead of its reciprocal",
     [("    double m = fp32(1.0 / fp32(ws_scale)); /* FP32 scalar and its FP32 reciprocal */",
       "    double m = fp32(ws_scale);")]),
    ("token pairs: the two tokens of a pair swapped",
     [("        *hi = t & 1;", "        *hi = (t + 1) & 1;")]),
    ("2FP4 residual with the wrong sign",
     [("            r[k] = fp32(x[k] - fp32(v1 * g));", "            r[k] = fp32(x[k] + fp32(v1 * g));")]),
]

BATTERY = [
    (tf.test_e2m1_grid_matches_golden, ()),
    (tf.test_e2m1_ties_golden, ()),
    (tf.test_e2m1_rounding_brute_force, ()),
    (tf.test_e4m3_saturation, ()),
    (tc.test_worked_block_golden, ()),
    (tc.test_grid_exactness_every_scale, (2.0 ** -7,)),
    (tc.test_tie_table_inside_blocks, ()),
    (tc.test_encode_steps_against_ieee_fp32_arithmetic, ()),
    (tc.test_closed_form_error_bound, ()),
    (tc.test_layout_positions_and_page_ids, ()),
    (tc.test_decode_against_ieee_fp32_arithmetic, ()),
    (tc.test_global_scale_rule, ()),
    (tc.test_global_scale_maps_tensor_max_to_top_of_both_grids, ()),
    (ta.test_zero_query_gives_mean_of_values_and_log_length, ()),
    (ta.test_gqa_head_mapping, ()),
    (ta.test_two_tokens_closed_form, ()),
    (ta.test_dominant_score_selects_its_value, ()),
    (tc.test_fp8_copy_scales_by_the_reciprocal_of_ws_scale, ()),
    (tc.test_token_pair_positions, ()),
    (tco.test_2fp4_second_component_encodes_the_first_ones_error, (0.0123,)),
]


def test_the_battery_passes_on_the_oracle():
    for fn, args in BATTERY:
        fn(*args)


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_a_planted_mistake(name, edits, tmp_path, monkeypatch):
    src = open(oracle._SRC).read()
    for old, new in edits:
        assert src.count(old) >= 1, f"mutation site not found: {old[:60]}"
        src = src.replace(old, new)
    c_file = tmp_path / "mutant.c"
    c_file.write_text(src)
    lib = oracle.bind(oracle.compile_to(str(c_file), str(tmp_path / "mutant.so")))
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    with np.errstate(all="ignore"):
        for fn, args in BATTERY:
            try:
                fn(*args)
            except Exception:  # an assertion, or the mutant producing unusable output
                caught.append(fn.__name__)
    assert caught, f"no pin caught: {name}"
