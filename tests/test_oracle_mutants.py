"""Plant plausible mistakes in copies of the oracle and require the pins to catch
each one.  Shows that the pins constrain every part of the oracle's arithmetic."""
import os

import pytest

import oracle
from tests import _pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, mutated text) -- each a mistake a careful reader could make
MUTANTS = [
    ("e4m3_bias_off_by_one", "v = ldexp(8.0 + m, e - 10);", "v = ldexp(8.0 + m, e - 11);"),
    ("e4m3_subnormal_scale", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    ("e5m2_mantissa_width", "v = ldexp(4.0 + m, e - 17);", "v = ldexp(4.0 + m, e - 16);"),
    ("e2m1_subnormal", "0.5 * m", "1.0 * m"),
    ("e8m0_bias", "ldexp(1.0, c - 127)", "ldexp(1.0, c - 128)"),
    ("scale_block_width", "S[i * kb + k / 32]", "S[i * kb + k / 64]"),
    ("mn_major_read_transposed", "X[k * rows + i]", "X[i * K + k]"),
    ("nn_treated_as_nt", "int b_kcontig = (layout == LAYOUT_NT);", "int b_kcontig = 1;"),
    ("grouped_sx_rowmajor_in_group",
     "j->start_of[r] * j->KB + j->loc_of[r] + kb * j->msz_of[r]",
     "j->start_of[r] * j->KB + j->loc_of[r] * j->KB + kb"),
    ("grouped_sw_drops_nblock",
     "sW[((int64_t)g * (j->N / 128) + n / 128) * j->KB + kb]",
     "sW[((int64_t)g * (j->N / 128)) * j->KB + kb]"),
    ("grouped_block_boundary", "k < kb * 128 + 128", "k < kb * 128 + 64"),
    ("wide_half_order", "(l / 8) * 256 + (c / 4) * 128", "(l / 8) * 256 + (c % 2) * 128"),
    ("wide_row_quarter", "int64_t c = 4 * g + l / 32;", "int64_t c = 4 * g + l % 4;"),
    ("wide_chunk_kgroups", "kq = kg / 2, g = kg % 2", "kq = kg / 4, g = kg % 2"),
    ("wide_col_lane", "lane_col_byte(nn % 32, nn / 32, kb % 4)", "lane_col_byte(nn / 8, nn % 8, kb % 4)"),
    ("wide_col_one_quarter", "for (int64_t q = 0; q < 4; ++q)", "for (int64_t q = 0; q < 1; ++q)"),
    ("quant_emax", "fmt == FMT_E4M3 ? 8 : fmt == FMT_E5M2 ? 15 : 2", "fmt == FMT_E4M3 ? 7 : fmt == FMT_E5M2 ? 15 : 2"),
    ("quant_floor_log2", "return p - 1;", "return p;"),
    ("quant_ties_odd", "else c = (lo & 1) ? hi : lo;", "else c = (lo & 1) ? lo : hi;"),
    ("quant_ties_away", "else c = (lo & 1) ? hi : lo;", "else c = hi;"),
    ("quant_saturate_past_top", "    c = top;\n", "    c = top + 1;\n"),
    ("quant_sign_from_comparison", "if (signbit(v)) c |=", "if (v < 0) c |="),
    ("quant_nibble_order", "if ((k & 1) == 0) *byte", "if ((k & 1) == 1) *byte"),
    ("quant_colwise_scale_order", "scales[o * (len / 32) + b] = scode;", "scales[b * outer + o] = scode;"),
    ("quant_no_clamp_low", "if (e < -127) e = -127;", "if (e < -127) e = e + 256;"),
    ("group_scale_fmax", "amax / 448.0f", "amax / 512.0f"),
    ("group_sx_rowmajor", "sx[start * KB + l + kb * mg] = s;", "sx[start * KB + l * KB + kb] = s;"),
    ("group_block_rows", "for (int64_t t = 0; t < 128; ++t) {\n          const float m = fabsf(x[r * K + kb * 128 + t]);",
     "for (int64_t t = 0; t < 64; ++t) {\n          const float m = fabsf(x[r * K + kb * 128 + t]);"),
    ("group_scale_no_floor", "return s > tiny ? s : tiny;", "return s;"),
    ("bias_per_row", "D[i * N + n] + (bias ? (double)bias[n] : 0.0)", "D[i * N + n] + (bias ? (double)bias[i % N] : 0.0)"),
    ("gelu_tanh_scale", "0.5 * v * (1.0 + erf(v / sqrt(2.0)))", "0.5 * v * (1.0 + erf(v / 2.0))"),
    ("silu_sign", "v = v / (1.0 + exp(-v));", "v = v / (1.0 + exp(v));"),
    ("relu_leaky", "v = v > 0.0 ? v : 0.0;", "v = v > 0.0 ? v : 0.01 * v;"),
    ("bf16_exponent_bias", "v = ldexp(128.0 + m, e - 134);", "v = ldexp(128.0 + m, e - 133);"),
    ("bf16_subnormal_scale", "v = ldexp((double)m, -133);", "v = ldexp((double)m, -132);"),
    ("bf16_exponent_field", "e = (c >> 7) & 255, m = c & 127;", "e = (c >> 8) & 255, m = c & 127;"),
    ("bf16_sign_dropped", "  return s ? -v : v;\n}", "  return v;\n}"),
    ("bf16_row_group", "    grp_of[r] = g;\n", "    grp_of[r] = g > 0 ? g - 1 : 0;\n"),
    ("bf16_w_transposed", "const uint16_t* w = j->W + ((int64_t)g * j->N + n) * j->K;",
     "const uint16_t* w = j->W + (int64_t)g * j->N * j->K + n;"),
    ("bf16_k_tail_dropped", "for (int64_t k = 0; k < j->K; ++k) acc += xrow[k] * wrow[k];",
     "for (int64_t k = 0; k + 1 < j->K; ++k) acc += xrow[k] * wrow[k];"),
    ("block_sw_kmajor", "sw[(g * (N / 128) + nb) * (K / 128) + kb] = s;", "sw[(g * (K / 128) + kb) * (N / 128) + nb] = s;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor missing: {old}"
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(text.replace(old, new))
    lib = oracle.bind(oracle.compile_c(str(mutated), str(tmp_path / "libmutant.so")))
    failures = []
    for pin in _pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, KeyError, IndexError):
            failures.append(pin.__name__)
    assert failures, f"no pin caught mutant {name}"
