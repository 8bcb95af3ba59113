"""The oracle's pins catch plausible mistakes (no GPU).

Each case plants one mistake in a copy of oracle/oracle.c, builds it into a
temporary library, points the oracle binding at it and runs the pins that
should notice; at least one of them must fail.  A mistake no pin notices
would mean the oracle is pinned to itself only.  The real oracle is restored
after every case.
"""
import importlib
import os
import shutil
import subprocess

import pytest

import oracle

ORACLE_DIR = os.path.dirname(os.path.abspath(oracle.__file__))

# (name, text in oracle.c, planted mistake, pins: (module, test, kwargs))
MUTANTS = [
    ("e2m1 ties round to odd",
     "(d == bd && (c & 1) == 0)", "(d == bd && (c & 1) == 1)",
     [("test_oracle_formats", "test_e2m1_encode_golden", {}),
      ("test_oracle_formats", "test_e2m1_encode_is_nearest_even_on_a_dense_grid", {})]),
    ("bf16 truncates",
     "double val = nearbyint(a / q) * q;", "double val = floor(a / q) * q;",
     [("test_oracle_formats", "test_bf16_rounding_matches_torch_on_fp32_values", {}),
      ("test_oracle_formats", "test_bf16_rounds_once_from_fp64", {})]),
    ("tensor scale amax / 448",
     "float sg = amax / 2688.0f;", "float sg = amax / 448.0f;",
     [("test_oracle_quant", "test_equal_block_at_tensor_max_gives_six_and_448", {}),
      ("test_oracle_quant", "test_codes_and_scales_are_nearest_by_brute_force", {})]),
    ("block scale ab / 4",
     "float q = ab / 6.0f;", "float q = ab / 4.0f;",
     [("test_oracle_quant", "test_equal_block_at_tensor_max_gives_six_and_448", {}),
      ("test_oracle_quant", "test_codes_and_scales_are_nearest_by_brute_force", {})]),
    ("nibbles swapped when packing",
     "out[i] = (uint8_t)(lo | (hi << 4));", "out[i] = (uint8_t)(hi | (lo << 4));",
     [("test_oracle_quant", "test_low_nibble_holds_the_even_element", {})]),
    ("nibbles swapped when unpacking",
     "uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);",
     "uint8_t code = (c & 1) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4);",
     [("test_oracle_quant", "test_dequantize_matches_format_tables", {}),
      ("test_oracle_quant", "test_dequantization_error_bound", {})]),
    ("branch norm without eps",
     "double inv = 1.0 / sqrt(ms + eps);", "double inv = 1.0 / sqrt(ms);",
     [("test_oracle_step", "test_constant_rows_closed_form", {}),
      ("test_oracle_step", "test_norm_is_scale_free_without_eps", {})]),
    ("post-norm weight dropped",
     "s[h] = (float)((double)s[h] + br[h] * inv * (double)w_post[h]);",
     "s[h] = (float)((double)s[h] + br[h] * inv);",
     [("test_oracle_step", "test_constant_rows_closed_form", {}),
      ("test_oracle_step", "test_norm_is_scale_free_without_eps", {})]),
    ("front norm without eps",
     "double inv_front = 1.0 / sqrt(ms + eps);", "double inv_front = 1.0 / sqrt(ms);",
     [("test_oracle_step", "test_front_constant_rows_closed_form", {})]),
    ("front stream rounded to bf16 twice",
     "s[h] = (float)oracle_bf16_decode(embedded[(int64_t)r * H + h]);",
     "s[h] = (float)oracle_bf16_decode(oracle_bf16_from_double(0.5 * oracle_bf16_decode(embedded[(int64_t)r * H + h])));",
     [("test_oracle_step", "test_front_stream_is_the_embedding_exactly", {})]),
    ("top-k ties to the higher id",
     "if (best < 0 || p[e] > p[best]) best = e;", "if (best < 0 || p[e] >= p[best]) best = e;",
     [("test_oracle_step", "test_ties_go_to_the_lower_expert_and_are_flagged", {}),
      ("test_oracle_step", "test_topk_brute_force_subsets", {"k": 2})]),
    ("gates not renormalised",
     "gates[r * k + s] = p[sel[s]] / sum;", "gates[r * k + s] = p[sel[s]];",
     [("test_oracle_step", "test_tiny_layer_statistics", {}),
      ("test_oracle_step", "test_topk_brute_force_subsets", {"k": 2})]),
    ("near-tie flag threshold 1e-3",
     "flags[r] = (uint8_t)(g < 1e-6);", "flags[r] = (uint8_t)(g < 1e-3);",
     [("test_oracle_step", "test_ties_go_to_the_lower_expert_and_are_flagged", {}),
      ("test_oracle_step", "test_near_tie_flag_is_the_gap_below_1e6", {})]),
    ("silu on up instead of gate",
     "h[(int64_t)pos * I + j] = (float)(silu(G) * U);", "h[(int64_t)pos * I + j] = (float)(G * silu(U));",
     [("test_oracle_step", "test_single_expert_with_gate_one_is_a_dense_gated_mlp", {}),
      ("test_oracle_step", "test_every_expert_selected_matches_gated_dense_sum", {})]),
    ("down uses the up projection's scale",
     "float sg_down = w->gscale[3 * e + 2];", "float sg_down = w->gscale[3 * e + 1];",
     [("test_oracle_step", "test_single_expert_with_gate_one_is_a_dense_gated_mlp", {}),
      ("test_oracle_step", "test_every_expert_selected_matches_gated_dense_sum", {})]),
    ("gather without gates",
     "acc += gates[r * k + s] * (double)o[((int64_t)r * k + s) * H + hh];",
     "acc += (double)o[((int64_t)r * k + s) * H + hh];",
     [("test_oracle_step", "test_every_expert_selected_matches_gated_dense_sum", {})]),
    ("dense: MLP input normalises the uncast stream",
     "t[h] = oracle_bf16_decode(oracle_bf16_from_double((double)s[h]));", "t[h] = (double)s[h];",
     [("test_oracle_dense", "test_mlp_input_normalises_the_stream_cast_to_bf16", {})]),
    ("dense: post-attention norm without eps",
     "double inv_attn = 1.0 / sqrt(ms / H + eps);", "double inv_attn = 1.0 / sqrt(ms / H);",
     [("test_oracle_dense", "test_post_attention_norm_of_constant_rows_closed_form", {})]),
    ("dense: silu on up instead of gate",
     "double v = g / (1.0 + exp(-g)) * u;", "double v = u / (1.0 + exp(-u)) * g;",
     [("test_oracle_dense", "test_single_entry_weights_name_each_product", {})]),
    ("dense: projection weight read transposed",
     "* oracle_bf16_decode(B[(int64_t)n * K + k]);", "* oracle_bf16_decode(B[(int64_t)k * N + n]);",
     [("test_oracle_dense", "test_projections_are_library_matmuls_over_exact_sums", {}),
      ("test_oracle_dense", "test_single_entry_weights_name_each_product", {})]),
    ("dense: output norm weight dropped",
     "s[h] = (float)((double)s[h] + br[h] * inv_out * (double)w_post_ffn[h]);",
     "s[h] = (float)((double)s[h] + br[h] * inv_out);",
     [("test_oracle_dense", "test_output_norm_of_a_constant_down_projection", {}),
      ("test_oracle_dense", "test_scale_free_without_eps", {})]),
    ("dense: output branch added without its norm",
     "double inv_out = 1.0 / sqrt(ms / H + eps);", "double inv_out = 1.0;",
     [("test_oracle_dense", "test_output_norm_of_a_constant_down_projection", {}),
      ("test_oracle_dense", "test_scale_free_without_eps", {})]),
    ("context KV: rotation with the sine's sign flipped",
     "y1 = x1 * cos(ang) - x2 * sin(ang);", "y1 = x1 * cos(ang) + x2 * sin(ang);",
     [("test_oracle_ctxkv", "test_one_hot_key_rotates_into_its_partner_dimension", {})]),
    ("context KV: rotation angle exponent -j/D",
     "pow(theta, -2.0 * j / D)", "pow(theta, -1.0 * j / D)",
     [("test_oracle_ctxkv", "test_one_hot_key_rotates_into_its_partner_dimension", {})]),
    ("context KV: key norm without eps",
     "double inv = 1.0 / sqrt(ms / D + qk_eps);", "double inv = 1.0 / sqrt(ms / D);",
     [("test_oracle_ctxkv", "test_key_norm_of_constant_heads_and_values_pass_through", {})]),
    ("context KV: keys rotated before their bf16 cast",
     "kn[i] = oracle_bf16_decode(oracle_bf16_from_double(oracle_bf16_decode(k[i]) * inv));",
     "kn[i] = oracle_bf16_decode(k[i]) * inv;",
     [("test_oracle_ctxkv", "test_one_hot_key_rotates_into_its_partner_dimension", {})]),
    ("context KV: every layer normalised with layer 0's weight",
     "double v = oracle_bf16_decode(f[h]) * inv_pre * (double)w_pre[(int64_t)l * H + h];",
     "double v = oracle_bf16_decode(f[h]) * inv_pre * (double)w_pre[h];",
     [("test_oracle_ctxkv", "test_constant_rows_closed_form", {})]),
    ("context KV: layer norms' mean square not divided by H",
     "double inv_pre = 1.0 / sqrt(ms_fc / H + eps);", "double inv_pre = 1.0 / sqrt(ms_fc + eps);",
     [("test_oracle_ctxkv", "test_constant_rows_closed_form", {})]),
    ("context KV: every layer's keys written to layer 0's cache",
     "memcpy(k_cache + ((int64_t)l * n_slots + slot) * KD,", "memcpy(k_cache + (slot) * KD,",
     [("test_oracle_ctxkv", "test_cache_scatter_by_brute_force", {})]),
    ("context KV: slot 0 skipped as if negative",
     "if (slot < 0 || slot >= n_slots) continue;", "if (slot <= 0 || slot >= n_slots) continue;",
     [("test_oracle_ctxkv", "test_cache_scatter_by_brute_force", {})]),
    ("context KV: values copied from the key heads",
     "memcpy(v_out + o, row + KD + hd * D, sizeof(uint16_t) * D);",
     "memcpy(v_out + o, row + hd * D, sizeof(uint16_t) * D);",
     [("test_oracle_ctxkv", "test_key_norm_of_constant_heads_and_values_pass_through", {})]),
    ("context KV: keys rotated by the row index instead of the position",
     "double ang = (double)positions[r] * pow(", "double ang = (double)r * pow(",
     [("test_oracle_ctxkv", "test_one_hot_key_rotates_into_its_partner_dimension", {})]),
    ("e4m3 subnormals decoded at half their value",
     "mag = ldexp((double)m / 8.0, -6);", "mag = ldexp((double)m / 8.0, -7);",
     [("test_oracle_formats", "test_e4m3_decode_matches_torch_and_golden", {})]),
    ("e4m3 saturates to NaN instead of 448",
     "if (a >= 448.0) return (uint8_t)(s | 0x7E);", "if (a >= 448.0) return (uint8_t)(s | 0x7F);",
     [("test_oracle_formats", "test_e4m3_encode_matches_torch_in_range_and_saturates", {})]),
    ("router bias subtracted",
     "if (bias) acc += (double)bias[e];", "if (bias) acc -= (double)bias[e];",
     [("test_oracle_step", "test_k_equals_E_is_the_full_softmax", {"bias": True})]),
    ("softmax at temperature 2",
     "p[e] = exp(logit[e] - m);", "p[e] = exp(0.5 * (logit[e] - m));",
     [("test_oracle_step", "test_k_equals_E_is_the_full_softmax", {"bias": False})]),
    ("pooler lists idle experts as active",
     "if (count[e] > 0) active[na++] = e;", "if (count[e] >= 0) active[na++] = e;",
     [("test_oracle_step", "test_pooler_invariants", {"rows": 2, "E": 9, "k": 2})]),
    ("pooler orders an expert's pairs by descending row",
     "for (int r = 0; r < rows; ++r)\n      for (int s = 0; s < k; ++s)\n        if (ids[r * k + s] == e)",
     "for (int r = rows - 1; r >= 0; --r)\n      for (int s = 0; s < k; ++s)\n        if (ids[r * k + s] == e)",
     [("test_oracle_step", "test_pooler_invariants", {"rows": 13, "E": 9, "k": 3})]),
    ("h quantized from the first expert's rows",
     "oracle_nvfp4_quantize(h + (int64_t)offset[e] * I, n, I,", "oracle_nvfp4_quantize(h, n, I,",
     [("test_oracle_step", "test_every_expert_selected_matches_gated_dense_sum", {}),
      ("test_oracle_step", "test_tiny_layer_statistics", {})]),
    ("down dequantizes every h with expert 0's scale",
     "h_sg[e], 1, I, hh + (int64_t)pos * I);", "h_sg[0], 1, I, hh + (int64_t)pos * I);",
     [("test_oracle_step", "test_every_expert_selected_matches_gated_dense_sum", {})]),
    ("gather reads the pairs slot-major",
     "acc += gates[r * k + s] * (double)o[((int64_t)r * k + s) * H + hh];",
     "acc += gates[r * k + s] * (double)o[((int64_t)s * rows + r) * H + hh];",
     [("test_oracle_step", "test_every_expert_selected_matches_gated_dense_sum", {}),
      ("test_oracle_step", "test_row_permutation_permutes_outputs", {})]),
    ("dense: SiLU * mul takes the up value from the gate half",
     "double u = oracle_bf16_decode(gu[(int64_t)r * 2 * I + I + j]);",
     "double u = oracle_bf16_decode(gu[(int64_t)r * 2 * I + j]);",
     [("test_oracle_dense", "test_single_entry_weights_name_each_product", {})]),
]


@pytest.fixture(scope="module")
def mutant_libs(tmp_path_factory):
    """Builds every mutant in parallel: name -> library path."""
    src = open(os.path.join(ORACLE_DIR, "oracle.c")).read()
    root = tmp_path_factory.mktemp("oracle_mutants")
    shutil.copy(os.path.join(ORACLE_DIR, "oracle.h"), root / "oracle.h")
    procs, libs = [], {}
    for i, (name, old, new, _) in enumerate(MUTANTS):
        assert src.count(old) == 1, f"mutation site of '{name}' not found once in oracle.c"
        c = root / f"m{i}.c"
        c.write_text(src.replace(old, new))
        so = root / f"libm{i}.so"
        procs.append(subprocess.Popen(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
             "-I", str(root), "-o", str(so), str(c), "-lm"], stderr=subprocess.PIPE))
        libs[name] = str(so)
    for p in procs:
        _, err = p.communicate()
        assert p.returncode == 0, err.decode()
    return libs


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_a_pin_catches_the_planted_mistake(name, mutant_libs):
    pins = next(m[3] for m in MUTANTS if m[0] == name)
    saved = (oracle.LIB, oracle._lib)
    oracle.LIB, oracle._lib = mutant_libs[name], None
    caught = []
    try:
        for module, test, kwargs in pins:
            fn = getattr(importlib.import_module(module), test)
            try:
                fn(**kwargs)
            except AssertionError:
                caught.append(test)
    finally:
        oracle.LIB, oracle._lib = saved
    assert caught, f"no pin notices '{name}'"
