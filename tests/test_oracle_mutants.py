"""Plant plausible mistakes in copies of the oracle (on the CPU) and check
that at least one pin fails for each: a dropped term, a wrong sign, a
wrong index, a swapped nibble, a wrong constant.  This shows that the pins
in tests/oracle_pins.py constrain every step of the oracle."""
import os

import pytest

import oracle
from tests import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "mlq_oracle.c")

# (name, original text, mutated text); every mutant stays in bounds.
MUTANTS = [
    ("high_nibble_as_low", "(bytes16[j] >> 4) - 8", "(bytes16[j] & 0x0F) - 8"),
    ("offset_7_not_8", "(int)(bytes16[j] & 0x0F) - 8", "(int)(bytes16[j] & 0x0F) - 7"),
    ("nibble_halves_swapped", "w[j + 16] = (int8_t)((int)(bytes16[j] >> 4) - 8);",
     "w[j + 16] = (int8_t)((int)(bytes16[j] & 0x0F) - 8); w[j] = (int8_t)((int)(bytes16[j] >> 4) - 8);"),
    ("dropped_dx", "t = t * xd[b];", "t = t;"),
    ("wrong_dw_index", "wd[(size_t)r * nb + b]", "wd[b]"),
    ("wrong_x_block", "int32_t sumi = block_dot(w, xq + (size_t)b * ORACLE_QK);", "int32_t sumi = block_dot(w, xq);"),
    ("no_accumulate", "sum = sum + t;", "sum = t;"),
    ("id_128", "127.0f / amax", "128.0f / amax"),
    ("d_128", "amax / 127.0f", "amax / 128.0f"),
    ("round_not_signed", "copysignf(0.5f, x[j])", "0.5f"),
    ("clamp_126", "if (v >= 127.0f)       qq = 127;", "if (v >= 127.0f)       qq = 126;"),
    ("nan_not_zero", "else if (v != v)       qq = 0;", "else if (v != v)       qq = 1;"),
    ("fused_round", "float v = x[j] * id;                         /* one rounded multiply  */\n        v = v + copysignf(0.5f, x[j]);",
     "float v = fmaf(x[j], id, copysignf(0.5f, x[j]));"),
    ("round_half_even", "v = truncf(v);", "v = rintf(v - copysignf(0.5f, x[j]));"),
    ("dot_drops_last", "for (int j = 0; j < ORACLE_QK; ++j) s +=", "for (int j = 0; j < ORACLE_QK - 1; ++j) s +="),
    ("row_range_from_zero", "for (int r = r0; r < r1; ++r) {\n        float sum", "for (int r = 0; r < r1; ++r) {\n        float sum"),
    ("small_m_row_stride", "Y + (size_t)m * ldy", "Y + (size_t)m * rows"),
    ("rmsnorm_no_mean", "sqrt(ss / (double)n + (double)eps)", "sqrt(ss + (double)eps)"),
    ("rmsnorm_eps_outside", "sqrt(ss / (double)n + (double)eps)", "(sqrt(ss / (double)n) + (double)eps)"),
    ("softmax_no_max_in_sum", "sum += exp((double)x[i] - mx);", "sum += exp((double)x[i]);"),
    ("silu_sign", "a / (1.0 + exp(-a))", "a / (1.0 + exp(a))"),
    ("add_subtracts", "(double)y[j] + (double)x[j]", "(double)y[j] - (double)x[j]"),
    ("rope_freq_halved", "-2.0 * i / (double)head_dim", "-1.0 * i / (double)head_dim"),
    ("rope_sign", "a * c[i] - b * s[i]", "a * c[i] + b * s[i]"),
    ("rope_k_not_rotated", "for (int h = 0; h < n_kv_heads; ++h) rope_head", "for (int h = 0; h < 0; ++h) rope_head"),
    ("attention_no_scale", "p[t] = dot / sqrt((double)head_dim);", "p[t] = dot;"),
    ("attention_gqa_modulo", "const int g = h / group;", "const int g = h % n_kv_heads;"),
    ("q4k_min_added", "const float v = (t - u) * xd[B];", "const float v = (t + u) * xd[B];"),
    ("q4k_first_scale_only", "is += (int32_t)sm[b] * dot;", "is += (int32_t)sm[0] * dot;"),
    ("q4k_min_from_scales", "ms += (int32_t)sm[8 + b] * xbs[sb];", "ms += (int32_t)sm[b] * xbs[sb];"),
    ("q4k_high_nibble_low_x", "dot += (int32_t)(bytes[j] >> 4) * a[j + 16];",
     "dot += (int32_t)(bytes[j] >> 4) * a[j];"),
    ("q4k_dmin_row0", "(float)ms * wdmin[(size_t)r * nsb + B]", "(float)ms * wdmin[B]"),
    ("q4k_no_accumulate", "yr = yr + v;", "yr = v;"),
    ("q8k_bsum_drops_first", "for (int i = 0; i < ORACLE_QK; ++i) t += q[", "for (int i = 1; i < ORACLE_QK; ++i) t += q["),
    ("q8k_one_scale", "quantize_span(q + e0, d + (size_t)r * nsb + B, x + e0, ORACLE_QKK);",
     "quantize_span(q + e0, d + (size_t)r * nsb + B, x + e0, ORACLE_QK); quantize_span(q + e0 + ORACLE_QK, d + (size_t)r * nsb + B, x + e0 + ORACLE_QK, ORACLE_QKK - ORACLE_QK);"),
    ("half_bias_14", "v = ldexpf((float)(f + 1024), e - 25);", "v = ldexpf((float)(f + 1024), e - 24);"),
    ("half_subnormal_implicit", "if (e == 0)       v = ldexpf((float)f, -24);", "if (e == 0)       v = ldexpf((float)(f + 1024), -24);"),
    ("nbits_high_at_16", "(blkb[i] & 0x0F) : (blkb[i - blk / 2] >> 4)", "(blkb[i] & 0x0F) : (blkb[(i - blk / 2) % 16] >> 4)"),
    ("nbits_zp_sign", "return (int32_t)bp + 128 - z;", "return (int32_t)bp - 128 + z;"),
    ("nbits_zp_ignored", "const int z = zp ? zp[(size_t)r * nb + b] : 128;", "const int z = 128;"),
    ("nbits_x_block0", "* (int32_t)xq[(size_t)b * blk + i];\n            const size_t si", "* (int32_t)xq[i];\n            const size_t si"),
    ("nbits_scale_row0", "((const float *)scales)[si];", "((const float *)scales)[b];"),
    ("blk_bsum_drops_last", "for (int i = 0; i < blk; ++i) t += q[", "for (int i = 0; i < blk - 1; ++i) t += q["),
    ("attention_drops_last", "for (int t = 0; t < n_pos; ++t) {\n            const float *vt",
     "for (int t = 0; t < n_pos - 1; ++t) {\n            const float *vt"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    mpath = tmp_path / f"{name}.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.compile_c(str(mpath), str(tmp_path / f"lib_{name}.so"))
    O = oracle.Oracle(lib)
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(O)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
