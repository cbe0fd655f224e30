"""Plant plausible mistakes in copies of the oracle source and check that some pin fails.

Each mutant is one textual change to ``oracle/mla_oracle.c`` (a dropped term, a flipped
sign, a transposed or wrong operand, an off-by-one).  The copy is compiled into a temporary
directory on the CPU and the pins of ``oracle_pins.py`` run against it; at least one must
raise.  The real oracle source is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402
import oracle_pins as pins  # noqa: E402

MUTANTS = {
    "naive_rope_term_dropped": (
        "for (int r = 0; r < DR; ++r) dot += qr[r] * kvr[r];\n            s[t] = dot * softmax_scale;",
        "s[t] = dot * softmax_scale;"),
    "naive_w_uk_transposed": ("a += Wk[d * DC + c] * ckv[c];", "a += Wk[c * DHC + d] * ckv[c];"),
    "naive_value_through_w_uk": ("a += Wv[d * DC + c] * ckv[c];", "a += Wk[d * DC + c] * ckv[c];"),
    "naive_softmax_sign": ("double p = exp(s[t] - mx) / den;", "double p = exp(mx - s[t]) / den;"),
    "naive_denominator_short": ("for (int64_t t = 0; t < S; ++t) den += exp(s[t] - mx);",
                                "for (int64_t t = 0; t + 1 < S; ++t) den += exp(s[t] - mx);"),
    "naive_scale_dropped": ("s[t] = dot * softmax_scale;", "s[t] = dot;"),
    "gather_slot_shifted": ("slot = t % PG;", "slot = (t + 1) % PG;"),
    "gather_ignores_block_table": ("int64_t page = bt_row[t / PG]", "int64_t page = t / PG"),
    "e4m3_bias_off_by_one": ("mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "fp8_scale_ignored": ("ckv[i] = oracle_e4m3_value(row[i]) * sigma;", "ckv[i] = oracle_e4m3_value(row[i]);"),
    "latent_rope_term_dropped": (
        "for (int r = 0; r < DR; ++r) dot += qr[r] * kvr[r];\n            s[i] = dot * softmax_scale;",
        "s[i] = dot * softmax_scale;"),
    "latent_lse_base2": ("const double l = n > 0 ? mx + log(den) : -INFINITY;",
                         "const double l = n > 0 ? mx + log2(den) : -INFINITY;"),
    "latent_last_token_dropped": ("if (t1 > seq_lens[b]) t1 = seq_lens[b];",
                                  "if (t1 > seq_lens[b] - 1) t1 = seq_lens[b] - 1;"),
    "absorb_w_uk_transposed": ("bf16_value(w_uk[((int64_t)h * DHC + d) * DC + c])",
                               "bf16_value(w_uk[((int64_t)h * DC + c) * DHC + d])"),
    "out_proj_wrong_head": ("bf16_value(w_uv[((int64_t)h * DHC + d) * DC + c])",
                            "bf16_value(w_uv[((int64_t)(h ^ 1) * DHC + d) * DC + c])"),
    "combine_unnormalised_weight": ("const double w = exp(lj - L);", "const double w = exp(lj - mx);"),
    "e4m3_encode_ties_away": ("c = (lo & 1) ? hi : lo; /* a tie: the even mantissa field */", "c = hi;"),
    "e4m3_encode_zero_sign_lost": ("const uint8_t sign = signbit(x) ? 0x80 : 0x00;",
                                   "const uint8_t sign = x < 0.0f ? 0x80 : 0x00;"),
    "e4m3_encode_overflow_to_nan": ("if (a >= 448.0) return sign | 0x7E;", "if (a > 448.0) return sign | 0x7F;"),
    "e4m3_encode_truncates": ("if (d_lo < d_hi)\n        c = lo;", "if (d_lo <= d_hi + 1e300)\n        c = lo;"),
    "quantize_scale_447": ("const float sigma = amax > 0.0f ? amax / 448.0f : 1.0f;",
                           "const float sigma = amax > 0.0f ? amax / 447.0f : 1.0f;"),
    "quantize_zero_row_scale": ("const float sigma = amax > 0.0f ? amax / 448.0f : 1.0f;",
                                "const float sigma = amax > 0.0f ? amax / 448.0f : 0.0f;"),
    "append_rope_from_latent": ("for (int j = 0; j < DR; ++j) row[DC + j] = r[j];",
                                "for (int j = 0; j < DR; ++j) row[DC + j] = c[j];"),
    "append_fp8_kr_shifted": ("kr[slot * DR + j] = r[j];", "kr[slot * DR + j] = r[(j + 1) % DR];"),
    "append_bad_slot_unreported": ("status = -1;\n            continue;", "status = 0;\n            continue;"),
    "bf16_widening_wrong": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = ((uint32_t)bits << 16) | 0x8000u;"),
    # NVFP4 (e2m1 codes with e4m3 block scales)
    "e2m1_subnormal_quarter": ("const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);",
                               "const double mag = e == 0 ? 0.25 * m : ldexp(1.0 + 0.5 * m, e - 1);"),
    "e2m1_bias_off_by_one": ("const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);",
                             "const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 2);"),
    "e2m1_ties_away": ("if (gap_above < gap_below || (gap_above == gap_below && (k & 1)))",
                       "if (gap_above <= gap_below)"),
    "e2m1_no_saturation": ("if (a >= 6.0) return sign | 0x7;", "if (a >= 7.0) return sign | 0x7;"),
    "nvfp4_sigma_without_six": ("const float sigma = amax > 0.0f ? amax / 2688.0f : 1.0f;",
                                "const float sigma = amax > 0.0f ? amax / 448.0f : 1.0f;"),
    "nvfp4_nibbles_swapped": ("const uint8_t code = (i & 1) ? (uint8_t)(row[i / 2] >> 4) : (uint8_t)(row[i / 2] & 0x0F);",
                              "const uint8_t code = (i & 1) ? (uint8_t)(row[i / 2] & 0x0F) : (uint8_t)(row[i / 2] >> 4);"),
    "nvfp4_block_of_32": ("ckv[i] = oracle_e2m1_value(code) * oracle_e4m3_value(bs[i / 16]) * sigma;",
                          "ckv[i] = oracle_e2m1_value(code) * oracle_e4m3_value(bs[i / 32]) * sigma;"),
    "nvfp4_block_scale_ignored": ("ckv[i] = oracle_e2m1_value(code) * oracle_e4m3_value(bs[i / 16]) * sigma;",
                                  "ckv[i] = oracle_e2m1_value(code) * sigma;"),
    "gather_fp8_scale_ignored": ("dst[i] = bf16_rne((float)oracle_e4m3_value(row[i]) * sigma);",
                                 "dst[i] = bf16_rne((float)oracle_e4m3_value(row[i]));"),
    "gather_nvfp4_nibbles_swapped": ("const uint8_t e2 = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);",
                                     "const uint8_t e2 = (i & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);"),
    # several new tokens per sequence
    "query_rows_causal_off_by_one": ("row_len[row] = seq_lens[b] - q + 1 + t;", "row_len[row] = seq_lens[b] - q + t;"),
    "query_rows_token_major": ("const int64_t row = (int64_t)b * q + t;", "const int64_t row = (int64_t)t * B + b;"),
    "query_rows_first_table_row": ("row_table[row] = b;", "row_table[row] = 0;"),
    "gather_bf16_truncates": ("return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);",
                              "return (uint16_t)(u >> 16);"),
    "gather_rows_shifted": ("uint16_t* dst = out + ((int64_t)cu_seqlens[b] + t) * DROW;",
                            "uint16_t* dst = out + ((int64_t)cu_seqlens[b] + (t + 1) % seq_lens[b]) * DROW;"),
    "nvfp4_block_scale_not_divided_by_six": ("const uint8_t s8 = oracle_e4m3_encode((bmax / sigma) / 6.0f);",
                                             "const uint8_t s8 = oracle_e4m3_encode(bmax / sigma);"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, mutant_dir):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique or missing"
    path_c = os.path.join(mutant_dir, f"{name}.c")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new))
    so = oracle.build(force=True, src=path_c, out=os.path.join(mutant_dir, f"{name}.so"))
    oracle._use_library(so)
    try:
        caught = None
        for check in pins.ALL_CHECKS:
            try:
                check()
            except (AssertionError, ValueError) as e:  # noqa: PERF203
                caught = (check.__name__, e)
                break
        assert caught is not None, f"no pin caught mutant {name}"
    finally:
        oracle._use_library(None)
