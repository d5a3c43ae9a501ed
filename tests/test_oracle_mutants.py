"""Planted mistakes in the oracle must each be caught by at least one pin.

Each mutant is a copy of ``oracle/mla_oracle.c`` with one plausible mistake
(a dropped term, a wrong sign, a wrong index, a transposed operand), compiled
into a temporary directory on the CPU.  The pin suite of ``oracle_pins`` is
run against it; the test passes when some pin fails.  This shows the pins
constrain every part of the oracle, not just that the oracle agrees with them.
"""

import os

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")

MUTANTS = {
    "drop_rope_score_term": (
        "acc += rd(q_pe, dqp, qrow * d_r + e) * rd(pool, dp, row + d_c + e);",
        "acc += 0.0 * rd(q_pe, dqp, qrow * d_r + e);"),
    "no_score_scale": ("s[j] = acc * scale;\n        if (s[j] > m) m = s[j];\n    }\n    double l",
                       "s[j] = acc;\n        if (s[j] > m) m = s[j];\n    }\n    double l"),
    "absorb_transposed_w_uk": (
        "dst[c] += qv * rd(w_uk, dw, wrow + c);",
        "dst[c] += qv * rd(w_uk, dw, (int64_t)i * d_h * d_c + ((int64_t)c * d_h + e) % ((int64_t)d_h * d_c));"),
    "rope_sign": ("x[2 * k] = a * cs - b * sn;", "x[2 * k] = a * cs + b * sn;"),
    "rope_frequency": ("pow(base, -2.0 * k / (double)d_r)", "pow(base, -1.0 * k / (double)d_r)"),
    "combine_unnormalised_weight": (
        "double w = exp(rd(lse_part, dpl, (int64_t)s * N + r) - L);",
        "double w = exp(rd(lse_part, dpl, (int64_t)s * N + r) - m);"),
    "ignore_page_table": (
        "int64_t pg = page_table[(int64_t)b * max_pages + j / page];\n        int64_t row = (pg * page + j % page) * width;\n        double acc",
        "int64_t pg = (int64_t)b * max_pages + j / page; (void)page_table;\n        int64_t row = (pg * page + j % page) * width;\n        double acc"),
    "out_proj_wrong_head": (
        "int64_t wrow = ((int64_t)i * d_h + e) * d_c;\n                int64_t orow",
        "int64_t wrow = ((int64_t)((i + 1) % H) * d_h + e) * d_c;\n                int64_t orow"),
    "causal_off_by_one": ("int64_t n = causal ? len - (T - 1 - t) : len;",
                          "int64_t n = causal ? len - (T - t) : len;"),
    "lse_without_max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "naive_value_uses_w_uk": ("av += rd(w_uv, dwv, wrow + c) * row[c];",
                              "av += rd(w_uk, dwk, wrow + c) * row[c];"),
    "query_rope_at_zero": ("d_r, (double)qpos, rope_base);", "d_r, 0.0, rope_base);"),
    "softmax_denominator": ("double a = exp(s[j] - m) / l;\n        if (a_out)",
                            "double a = exp(s[j] - m) / (l + 1.0);\n        if (a_out)"),
    "cache_rope_at_zero": ("orc_rope(row + d_c, d_r, (double)j, rope_base);",
                           "orc_rope(row + d_c, d_r, 0.0, rope_base);"),
    "query_head_rows_pe_first": (
        "if (e < d_h) q_nope[((int64_t)b * H + i) * d_h + e] = acc;\n"
        "                else q_pe[((int64_t)b * H + i) * d_r + (e - d_h)] = acc;",
        "if (e >= d_r) q_nope[((int64_t)b * H + i) * d_h + (e - d_r)] = acc;\n"
        "                else q_pe[((int64_t)b * H + i) * d_r + e] = acc;"),
    "spread_without_abs": ("dst[c] += a[j] * fabs(rd(pool, dp, row + c) - o[c]);",
                           "dst[c] += a[j] * (rd(pool, dp, row + c) - o[c]);"),
    "spread_about_zero": ("dst[c] += a[j] * fabs(rd(pool, dp, row + c) - o[c]);",
                          "dst[c] += a[j] * fabs(rd(pool, dp, row + c));"),
    "prefill_causal_off_by_one": ("int64_t n = causal ? (int64_t)t + 1 : L;",
                                  "int64_t n = causal ? (int64_t)t : L;"),
    "prefill_value_uses_w_uk": ("vx += rd(w_uv, dwv, wr + c) * row[c];",
                                "vx += rd(w_uk, dwk, wr + c) * row[c];"),
    "prefill_attn_rope_offset_ignored": (
        "acc += rd(q_pe, dqp, f * d_r + e) * rd(k_pe, dkp, (first + j) * k_pe_ld + k_pe_off + e);",
        "acc += rd(q_pe, dqp, f * d_r + e) * rd(k_pe, dkp, (first + j) * k_pe_ld + e);"),
    "prefill_attn_ignores_causal": ("int64_t n = causal ? t + (int64_t)1 : (int64_t)L;",
                                    "int64_t n = (int64_t)L + 0 * t;"),
    "prefill_attn_value_row_of_query": ("int64_t vr = (first + j) * H + i;", "int64_t vr = f;"),
    "project_kr_uses_w_dkv": ("acc += rd(w_kr, dw2, (int64_t)e * d + k) * rd(h, dh_t, hrow + k);",
                              "acc += rd(w_dkv, dw1, (int64_t)e * d + k) * rd(h, dh_t, hrow + k);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site of {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(str(path), str(tmp_path / "libmutant.so")))
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
            break
    assert failed, f"no pin caught mutant {name}"
