"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/oracle.c`` (on the CPU,
in a temporary directory), builds it, and runs the oracle pin suites against
the broken copy: at least one pin has to fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "drop_first_partial": ("acc = acc + orc_bf16_decode(partials[r][in_off + j]);",
                           "acc = acc + (r ? orc_bf16_decode(partials[r][in_off + j]) : 0.0f);"),
    "residual_sign": ("x[j] = x[j] + orc_bf16_decode(residual[loc_off + j]);",
                      "x[j] = x[j] - orc_bf16_decode(residual[loc_off + j]);"),
    "add_in_sign": ("x[j] = x[j] + orc_bf16_decode(add_in[loc_off + j]);",
                    "x[j] = x[j] - orc_bf16_decode(add_in[loc_off + j]);"),
    "add_in_wrong_row": ("x[j] = x[j] + orc_bf16_decode(add_in[loc_off + j]);",
                         "x[j] = x[j] + orc_bf16_decode(add_in[in_off + j]);"),
    "token_split_extra_to_last": ("*count = base + (rank < extra ? 1 : 0);",
                                  "*count = base + (rank >= world - extra ? 1 : 0);"),
    "mean_over_h_minus_1": ("float variance = mean_of_squares(ss, (double)H);",
                            "float variance = mean_of_squares(ss, (double)(H - 1));"),
    "eps_dropped": ("float t = variance + eps;", "float t = variance;"),
    "norm_of_rounded_x": ("float y = (x[j] * scale) * orc_bf16_decode(gamma[j]);",
                          "float y = (orc_bf16_decode(orc_bf16_encode(x[j])) * scale) * orc_bf16_decode(gamma[j]);"),
    "gamma_reversed": ("float y = (x[j] * scale) * orc_bf16_decode(gamma[j]);",
                       "float y = (x[j] * scale) * orc_bf16_decode(gamma[H - 1 - j]);"),
    "block_scale_240": ("float s = amax / 448.0f;", "float s = amax / 240.0f;"),
    "fp4_nibbles_swapped": ("(uint8_t)(lo | (hi << 4))", "(uint8_t)(hi | (lo << 4))"),
    "e4m3_ties_away": ("r = nearbyint(a / q) * q;\n        if (r > 448.0)",
                       "r = round(a / q) * q;\n        if (r > 448.0)"),
    "e2m1_ties_away": ("r = nearbyint(a / q) * q;\n        if (r > 6.0)",
                       "r = round(a / q) * q;\n        if (r > 6.0)"),
    "bf16_truncates": ("double n = nearbyint(a / q);", "double n = floor(a / q);"),
    "sf_over_4": ("orc_e4m3_encode(g_scale * (amax / 6.0f))", "orc_e4m3_encode(g_scale * (amax / 4.0f))"),
    "qk_no_div_r": ("(double)(Vq / (float)R + eps)", "(double)(Vq + eps)"),
    "qk_weight_slice": ("orc_bf16_decode(wq[r * Q + j])", "orc_bf16_decode(wq[j])"),
    "qk_k_uses_q_mean": ("(double)(Vk / (float)R + eps)", "(double)(Vq / (float)R + eps)"),
    "single_matrix_no_div_r": ("(double)(V / (float)R + eps)", "(double)(V + eps)"),
    "single_matrix_weight_slice": ("orc_bf16_decode(weight[r * W + j])", "orc_bf16_decode(weight[j])"),
    "swizzle8_row_stride": ("return tile * 32 + (m % 8) * 4 + (k % 4);", "return tile * 32 + (m % 8) * 3 + (k % 4);"),
    "no_fp32_overflow": ("    if (ss >= ldexp(2.0 - ldexp(1.0, -24), 127))\n        return INFINITY;\n", ""),
    "ag_block_scale_240": ("float xs = amax / 448.0f;", "float xs = amax / 240.0f;"),
    "ag_y_uses_x_eps": ("segment_rmsnorm(row + q, kv, y_gamma, y_eps,", "segment_rmsnorm(row + q, kv, y_gamma, x_eps,"),
    "ag_y_uses_x_gamma": ("segment_rmsnorm(row + q, kv, y_gamma,", "segment_rmsnorm(row + q, kv, x_gamma,"),
    # (an earlier rank's slice never has fewer rows, so the planted read stays in bounds)
    "ag_wrong_rank": ("const uint16_t *row = inputs[rank] + (t - start) * hidden;",
                      "const uint16_t *row = inputs[rank > 0 ? rank - 1 : 0] + (t - start) * hidden;"),
    "fp8_tensor_divides": ("orc_e4m3_encode(n[j] * scale_factor)", "orc_e4m3_encode(n[j] / scale_factor)"),
    "fp4_element_scale_inverted": ("float es = (d == 0.0f) ? 0.0f : g_scale / d;",
                                   "float es = (d == 0.0f) ? 0.0f : d / g_scale;"),
    "partial_out_one_column_short": ("if (partial && partial_norm_out && j < partial_cols)",
                                     "if (partial && partial_norm_out && j + 1 < partial_cols)"),
    "fp8_block_zero_scale_divides": ("quant_out[ri * H + j] = (s == 0.0f) ? 0 : orc_e4m3_encode(n[j] / s);",
                                     "quant_out[ri * H + j] = orc_e4m3_encode(n[j] / s);"),
    "ag_copy_drops_rope": ("for (int64_t j = 0; j < hidden; ++j)\n                allgather_out[ri * hidden + j] = row[j];",
                           "for (int64_t j = 0; j < q + kv; ++j)\n                allgather_out[ri * hidden + j] = row[j];"),
    "partials_descending": ("for (int r = 0; r < R; ++r)\n                acc = acc + orc_bf16_decode(partials[r][in_off + j]);",
                            "for (int r = R - 1; r >= 0; --r)\n                acc = acc + orc_bf16_decode(partials[r][in_off + j]);"),
    "norm_scale_times_gamma_first": ("float y = (x[j] * scale) * orc_bf16_decode(gamma[j]);",
                                     "float y = x[j] * (scale * orc_bf16_decode(gamma[j]));"),
    "residual_before_add_in": (
        "        if (add_in)\n            for (int64_t j = 0; j < H; ++j)\n"
        "                x[j] = x[j] + orc_bf16_decode(add_in[loc_off + j]);\n\n"
        "        /* residual add, in fp32; residual_out is its bf16 rounding */\n"
        "        for (int64_t j = 0; j < H; ++j)\n"
        "            x[j] = x[j] + orc_bf16_decode(residual[loc_off + j]);\n",
        "        for (int64_t j = 0; j < H; ++j)\n"
        "            x[j] = x[j] + orc_bf16_decode(residual[loc_off + j]);\n"
        "        if (add_in)\n            for (int64_t j = 0; j < H; ++j)\n"
        "                x[j] = x[j] + orc_bf16_decode(add_in[loc_off + j]);\n"),
    "qk_shards_descending": ("for (int r = 0; r < R; ++r) {\n            const uint16_t *base = shards[r] + t * row_stride;\n"
                             "            double sq = 0.0, sk = 0.0;",
                             "for (int r = R - 1; r >= 0; --r) {\n            const uint16_t *base = shards[r] + t * row_stride;\n"
                             "            double sq = 0.0, sk = 0.0;"),
    "single_matrix_shards_descending": ("for (int r = 0; r < R; ++r) {\n            const uint16_t *base = shards[r] + t * row_stride;\n"
                                        "            double s = 0.0;",
                                        "for (int r = R - 1; r >= 0; --r) {\n            const uint16_t *base = shards[r] + t * row_stride;\n"
                                        "            double s = 0.0;"),
    "sf_scale_before_divide": ("orc_e4m3_encode(g_scale * (amax / 6.0f))", "orc_e4m3_encode((g_scale * amax) / 6.0f)"),
    "fp4_scale_folded_late": ("uint8_t lo = (d == 0.0f) ? 0 : orc_e2m1_encode(n[j] * es);",
                              "uint8_t lo = (d == 0.0f) ? 0 : orc_e2m1_encode((n[j] * g_scale) / d);"),
    "fp8_block_reciprocal_multiply": ("(s == 0.0f) ? 0 : orc_e4m3_encode(n[j] / s);",
                                      "(s == 0.0f) ? 0 : orc_e4m3_encode(n[j] * (1.0f / s));"),
    "fp8_block_scale_reciprocal": ("float s = amax / 448.0f;", "float s = amax * (1.0f / 448.0f);"),
    "swizzle_rows_cols": ("return tile * 512 + j * 16 + i * 4 + (k % 4);",
                          "return tile * 512 + i * 16 + j * 4 + (k % 4);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    import oracle

    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mut = tmp_path / "oracle_mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    oracle.build(force=True, src=str(mut), out=str(lib))
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_formats.py", "tests/test_oracle_fused.py",
                        "tests/test_oracle_qk.py", "tests/test_oracle_rs.py", "tests/test_oracle_ag.py",
                        "tests/test_oracle_golden.py"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 1, f"no pin caught mutant {name}:\n{r.stdout[-2000:]}"
