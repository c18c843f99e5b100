"""The oracle's pins must catch plausible mistakes.

Each mutant is a copy of the oracle source with one planted slip (on the CPU
only); the pin suite is run against it and must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "nvfp4_oracle.c")

MUTANTS = {
    "nibble_order_swapped": (
        "packed[i] = (uint8_t)(code[2 * i] | (code[2 * i + 1] << 4));",
        "packed[i] = (uint8_t)(code[2 * i + 1] | (code[2 * i] << 4));"),
    "e4m3_bias_off_by_one": (
        "mag = ldexp(1.0 + m / 8.0, e - 7);", "mag = ldexp(1.0 + m / 8.0, e - 8);"),
    "e2m1_subnormal_wrong": (
        "double mag = (e == 0) ? 0.5 * m :", "double mag = (e == 0) ? 1.0 * m :"),
    "ties_away_from_zero": (
        "return rint(a / spacing) * spacing;",
        "return floor(a / spacing + 0.5) * spacing;"),
    "scale_recipe_amax_over_4": (
        "orc_e4m3_encode(amax / (6.0 * g))", "orc_e4m3_encode(amax / (4.0 * g))"),
    "no_e2m1_saturation": ("if (v > 6.0) v = 6.0; /* satfinite */", ""),
    "v_uses_k_global_scale": (
        "double g = which == 0 ? c->k_global_scale : c->v_global_scale;\n  const uint8_t* data",
        "double g = c->k_global_scale;\n  const uint8_t* data"),
    "dropped_sm_scale": ("s[(j - j0) * rows + r] = sm_scale * acc;",
                         "s[(j - j0) * rows + r] = acc;"),
    "lse_in_log2": ("lse[r] = M[r] + log(Z[r]);", "lse[r] = M[r] + log2(Z[r]);"),
    "causal_top_left": ("limit[r] = causal ? (L - nq + i) : (L - 1);",
                        "limit[r] = causal ? (i) : (L - 1);"),
    "kv_head_modulo": ("(h_kv * G + g) * q_stride_head + d]",
                       "(g * c->num_kv_heads + h_kv) * q_stride_head + d]"),
    "merge_unnormalised": ("double w = exp(lse_partial[i] - lse);",
                           "double w = exp(lse_partial[i] - M);"),
    "slot_from_wrong_stride": ("slot * c->v_stride_slot", "slot * c->k_stride_slot"),
    "page_size_fixed_at_16": (
        "  pidx = pos / c->page_size;\n",
        "  pidx = pos / 16;\n"),
    "fp4qp_row_sum_without_p_scale": (
        "o[(int64_t)r * dv + d] / (kPScale * Z[r]);", "o[(int64_t)r * dv + d] / Z[r];"),
    "fp4qp_p_unquantised": ("      fp4_round16(pp, ph);\n",
                            "      memcpy(ph, pp, sizeof ph);\n"),
    "fp4qp_q_unquantised": ("        fp4_round16(x, qv + (int64_t)r * dk + d);\n",
                            "        memcpy(qv + (int64_t)r * dk + d, x, sizeof x);\n"),
    "fp4qp_mask_ignored_in_p": ("(j < L && j <= limit[r]) ? kPScale", "(j < L) ? kPScale"),
    "fp4qp_p_scaled_by_6_only": ("const double kPScale = 448.0 * 6.0;",
                                 "const double kPScale = 6.0;"),
    "fp4qp_causal_top_left": ("limit[r] = causal ? L - nq + i : L - 1;",
                              "limit[r] = causal ? i : L - 1;"),
    "fp4qp_lse_keeps_p_scale": ("-INFINITY : M[r] + log(Z[r]);",
                                "-INFINITY : M[r] + log(kPScale * Z[r]);"),
    "kv_len_page_size_fixed_at_16": (
        "  return (np - 1) * page_size + pt->last_page_len[b];",
        "  return (np - 1) * 16 + pt->last_page_len[b];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-w",
                           "-I", os.path.join(ROOT, "oracle"), str(mut), "-o",
                           str(so), "-lm"])
    env = dict(os.environ, NVFP4_ORACLE_SO=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p",
                        "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, "mutant %s survived the pins" % name
