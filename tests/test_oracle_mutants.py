"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is a copy of ``oracle/attn_oracle.c`` with one plausible error (a
dropped term, an off-by-one mask, a wrong head mapping, a transposed operand, a
wrong exponent bias ...), compiled on the CPU into a temporary library. The test
passes when at least one pin from ``oracle_pins`` fails on that mutant, which shows
the pins would notice the same mistake in the real oracle.
"""
import os

import pytest

import oracle
from oracle_pins import ORACLE_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "drop_scale": ("s[j - j_lo] = scale * dot;", "s[j - j_lo] = dot;"),
    "causal_excludes_diagonal": ("j_hi = pos + 1;", "j_hi = pos;"),
    "window_one_short": ("j_lo = pos - window_left;", "j_lo = pos - window_left + 1;"),
    "gqa_modulo_mapping": ("int64_t g = h / (Hq / Hkv);", "int64_t g = h % Hkv;"),
    "lse_drops_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "fp16_exponent_bias": ("e - 25);", "e - 24);"),
    "fp16_subnormal_scale": ("ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    "no_normalisation": ("double p = exp(s[j - j_lo] - m) / l;",
                         "double p = exp(s[j - j_lo] - m);"),
    "key_indexed_by_query_row": ("k + ((b * Lk + j) * Hkv + g) * d;",
                                 "k + ((b * Lk + (j + i) % Lk) * Hkv + g) * d;"),
    "values_read_from_keys": ("const uint16_t *vj = v + ", "const uint16_t *vj = k + "),
    "bf16_low_half": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    "max_not_subtracted_in_weights": ("double p = exp(s[j - j_lo] - m) / l;",
                                      "double p = exp(s[j - j_lo]) / l;"),
    "decode_queries_top_left": ("int64_t pos = Lk - Lq + i;", "int64_t pos = i;"),
    "decode_queries_off_by_one": ("int64_t pos = Lk - Lq + i;", "int64_t pos = Lk - Lq + i - 1;"),
    "key_range_start_ignored": ("        j_lo = key_lo;", "        j_lo = j_lo;"),
    "key_range_end_ignored": ("        j_hi = key_hi;", "        j_hi = j_hi;"),
    "merge_weights_unnormalised": ("double w = exp(lse_parts[p * nrows + r] - lse[r]);",
                                   "double w = exp(lse_parts[p * nrows + r] - m);"),
    "merge_lse_of_mean": ("lse[r] = m + log(total);", "lse[r] = m + log(total / nparts);"),
    "merge_first_part_only": ("        for (int64_t p = 0; p < nparts; ++p) {",
                              "        for (int64_t p = 0; p < 1; ++p) {"),
    "right_window_one_short": ("j_hi = pos + window_right + 1;", "j_hi = pos + window_right;"),
    "fp8_exponent_bias": ("m8 = ldexp((double)(f8 + 8), e8 - 10);",
                          "m8 = ldexp((double)(f8 + 8), e8 - 11);"),
    "fp8_subnormal_scale": ("m8 = ldexp((double)f8, -9);", "m8 = ldexp((double)f8, -10);"),
    "bwd_drops_D": ("double ds = p * (dp - D);", "double ds = p * dp;"),
    "bwd_dk_unscaled": ("dkj[c] += scale * ds * qi[c];", "dkj[c] += ds * qi[c];"),
    "bwd_dv_uses_dp": ("dvj[c] += p * doi[c];", "dvj[c] += dp * doi[c];"),
    "bwd_dq_uses_query": ("dqi[c] += scale * ds * widen16(krow[c], dtype);",
                          "dqi[c] += scale * ds * qi[c];"),
    "right_window_ignored": ("if (window_right >= 0 && pos + window_right + 1 < j_hi)",
                             "if (0 && pos + window_right + 1 < j_hi)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    src = tmp_path / f"mutant_{name}.c"
    src.write_text(text.replace(old, new))
    lib = oracle.load(oracle.build(str(src), str(tmp_path / f"lib_{name}.so"), force=True))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ORACLE_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
