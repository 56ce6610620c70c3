"""The oracle pins have teeth: each planted mistake in a copy of the oracle's C
source (built on the CPU, in a temporary directory) makes some pin fail."""
import importlib.util
import os
import shutil

import pytest

import test_oracle_pins as pins

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_DIR = os.path.join(os.path.dirname(HERE), "oracle")

# (name, original text, planted mistake)
MUTATIONS = [
    ("drop_last_head", "for (int h = 0; h < ORA_IDX_HEADS; ++h) {\n                double dot",
     "for (int h = 0; h < ORA_IDX_HEADS - 1; ++h) {\n                double dot"),
    ("drop_last_dim", "for (int d = 0; d < ORA_IDX_DIM; ++d) dot +=",
     "for (int d = 0; d < ORA_IDX_DIM - 1; ++d) dot +="),
    ("scale_from_next_slot", "(s % ORA_PAGE) * 4);", "((s + 1) % ORA_PAGE) * 4);"),
    ("relu_dropped", "double relu = x > 0.0 ? x : 0.0;", "double relu = x;"),
    ("softmax_shift_leaks", "double p = exp(x[j] - m);", "double p = exp(x[j] - m + 0.5);"),
    ("value_dim_dropped", "for (int d = 0; d < ORA_V_DIM; ++d)\n                    o[d] +=",
     "for (int d = 1; d < ORA_V_DIM; ++d)\n                    o[d] +="),
    ("lse_wrong_base", "m + log(Z)", "m + log2(Z)"),
    ("ties_to_upper_index", "return (x->index > y->index) - (x->index < y->index);",
     "return (x->index < y->index) - (x->index > y->index);"),
    ("latent_wrong_slot",
     "+ (size_t)(t % ORA_PAGE)) * ORA_LAT_DIM;\n                double dot",
     "+ (size_t)((t + 1) % ORA_PAGE)) * ORA_LAT_DIM;\n                double dot"),
    ("e4m3_subnormal_exponent", "mag = ldexp((double)m / 8.0, -6);",
     "mag = ldexp((double)m / 8.0, -7);"),
    ("e4m3_bias", "mag = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("dcp_never_resends", "                mask |= 1u << s;", "                mask |= 0u;"),
    ("dcp_suspicion_inverted", "ora_item_cmp(&all[start[s] + c - 1], &cut) < 0",
     "ora_item_cmp(&all[start[s] + c - 1], &cut) > 0"),
    ("layernorm_unbiased_variance", "var /= ORA_IDX_DIM;", "var /= (ORA_IDX_DIM - 1);"),
    ("key_scale_next_slot", "memcpy(kp + ORA_PAGE * ORA_IDX_DIM + (size_t)slot * 4,",
     "memcpy(kp + ORA_PAGE * ORA_IDX_DIM + (size_t)((slot + 1) % ORA_PAGE) * 4,"),
    ("e4m3_ties_to_odd", "(d == bestd && (c & 1) == 0)", "(d == bestd && (c & 1) == 1)"),
    ("e2m1_exponent_bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)"),
    ("e2m1_ties_to_odd", "(d == bestd && c % 2 == 0)", "(d == bestd && c % 2 == 1)"),
    ("e8m0_bias", "return ldexp(1.0, (int)code - 127);", "return ldexp(1.0, (int)code - 126);"),
    ("mx_emax_off_by_one", "(int)floor(log2(amax)) - 2;", "(int)floor(log2(amax)) - 1;"),
    ("mx_packing_high_nibble_first", "if (j % 2 == 0)\n                codes[j / 2] = c;",
     "if (j % 2 == 1)\n                codes[j / 2] = c;"),
    ("mx_scale_wrong_block", "scales[d / ORA_MX_BLOCK]",
     "scales[(d / ORA_MX_BLOCK + 1) % ORA_MX_SCALES]"),
    ("mx_key_scales_next_slot", "(size_t)slot * ORA_MX_SCALES);",
     "(size_t)((slot + 1) % ORA_PAGE) * ORA_MX_SCALES);"),
    ("mx_relu_dropped", "(qk > 0.0 ? qk : 0.0)", "qk"),
    ("nvfp4_scale_per_32", "scales[d / ORA_NV_BLOCK] & 0x7F", "scales[d / (2 * ORA_NV_BLOCK)] & 0x7F"),
    ("nvfp4_rope_unscaled", "L[ORA_V_DIM + j] = oracle_e4m3_decode(rope[j]) * latent_scale;",
     "L[ORA_V_DIM + j] = oracle_e4m3_decode(rope[j]);"),
    ("nvfp4_value_from_wrong_dims", "o[d] += pj * L[(size_t)j * ORA_LAT_DIM + d];",
     "o[d] += pj * L[(size_t)j * ORA_LAT_DIM + d + 64];"),
    ("nvfp4_scale_from_block_max", "scales[b] = oracle_e4m3_encode(amax / 6.0);",
     "scales[b] = oracle_e4m3_encode(amax / 4.0);"),
]

PIN_TESTS = [
    pins.test_e4m3_all_codes_match_torch,
    pins.test_indexer_single_head_is_relu_dot,
    pins.test_indexer_last_dim_and_scale_slot,
    pins.test_indexer_relu_is_per_head_before_weighting,
    pins.test_indexer_einsum_crosscheck,
    lambda m: [pins.test_topk_brute_force_with_ties(m, L, k) for L, k in [(100, 8), (1000, 64)]],
    lambda m: pins.test_topk_dcp_equals_single_shard_topk(m, 8),
    pins.test_topk_dcp_resend_pattern,
    pins.test_e4m3_encode_round_trip_and_torch_cast,
    pins.test_write_kv_layernorm_scale_codes_and_placement,
    pins.test_write_kv_zero_key,
    pins.test_mla_dense_matches_sdpa,
    pins.test_mla_single_token_and_zero_query,
    pins.test_mla_split_merge_by_lse,
    pins.test_e2m1_golden_table,
    pins.test_e2m1_encode_round_trip_and_golden_rounding,
    pins.test_e8m0_all_codes,
    pins.test_mx_quantize_scale_exponent_and_packing,
    pins.test_mx_quantize_exact_on_grid_and_error_bound,
    pins.test_indexer_mx_equals_fp8_scorer_on_shared_grid,
    pins.test_indexer_mx_last_dim_and_scale_slot,
    pins.test_write_key_mx_codes_and_placement,
    pins.test_nvfp4_latent_layout_last_dims,
    pins.test_nvfp4_encode_exact_on_shared_grid_and_error_bound,
    pins.test_mla_nvfp4_equals_fp8_on_shared_grid,
]


def _mutated_oracle(tmp_path, name, old, new):
    src = open(os.path.join(ORACLE_DIR, "dsa_oracle.c")).read()
    assert src.count(old) == 1, name
    d = tmp_path / name
    d.mkdir()
    shutil.copy(os.path.join(ORACLE_DIR, "oracle.py"), d / "oracle.py")
    (d / "dsa_oracle.c").write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"oracle_mut_{name}", d / "oracle.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build(force=True)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    mod = _mutated_oracle(tmp_path, name, old, new)
    caught = []
    for t in PIN_TESTS:
        try:
            t(mod)
        except (AssertionError, ValueError):
            caught.append(getattr(t, "__name__", "topk"))
    assert caught, f"no pin catches the planted mistake {name}"
