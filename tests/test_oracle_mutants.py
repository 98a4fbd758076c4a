"""Plants plausible mistakes in a copy of the C oracle (on the CPU) and checks
that the pins catch every one: a pin that a wrong oracle also passes pins
nothing."""
import os
import shutil

import pytest

from oracle import oracle as orc
import oracle_pins

SRC = os.path.join(os.path.dirname(orc.__file__), "fa_oracle.c")

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("dropped_scale", "s[j] = scale * dot(qi, k + (size_t)j * d, d);", "s[j] = dot(qi, k + (size_t)j * d, d);"),
    ("causal_excludes_diagonal", "return causal ? i + 1 + (Nk - Nq) : Nk;",
     "return causal ? (i > 0 ? i + (Nk - Nq) : 1 + (Nk - Nq)) : Nk;"),
    ("lse_without_log_sum", "lse[(size_t)h * Nq + i] = M + log(l);", "lse[(size_t)h * Nq + i] = M;"),
    ("output_reads_k_not_v", "const double* vh = v + (size_t)h * Nk * d;", "const double* vh = k + (size_t)h * Nk * d;"),
    ("kv_causal_top_left", "return causal ? i + 1 + (Nk - Nq) : Nk;", "return causal ? i + 1 : Nk;"),
    ("kv_query_head_stride", "const double* qi = q + ((size_t)h * Nq + i) * d;", "const double* qi = q + ((size_t)h * Nk + i) * d;"),
    ("padding_row_off_by_one", "if (i >= a) { /* a padding row */", "if (i > a) { /* a padding row */"),
    ("padding_key_ignored", "if (j >= b) continue; /* a padding key */", "if (j >= Nk) continue; /* a padding key */"),
    ("bwd_kv_key_head_stride", "const size_t qb = (size_t)h * Nq * d, kb = (size_t)h * Nk * d;\n      const double* kj",
     "const size_t qb = (size_t)h * Nq * d, kb = (size_t)h * Nq * d;\n      const double* kj"),
    ("D_wrong_sign", "Di += s[j] * dp[j];", "Di -= s[j] * dp[j];"),
    ("dq_dropped_scale", "dqi[t] += scale * ds * kj[t];", "dqi[t] += ds * kj[t];"),
    ("dk_transposed_operand", "dkj[t] += scale * ds * qi[t];", "dkj[t] += scale * ds * kj[t];"),
    ("dv_uses_dS", "dvj[t] += p * dOi[t];", "dvj[t] += ds * dOi[t];"),
    ("bwd_causal_skips_diagonal", "for (int i = causal && j > off ? j - off : 0; i < a; ++i)",
     "for (int i = causal && j >= off ? j - off + 1 : 0; i < a; ++i)"),
    ("bwd_mask_reversed", "for (int i = causal && j > off ? j - off : 0; i < a; ++i)",
     "for (int i = 0; i < (causal ? (j - off + 1 > 0 ? j - off + 1 : 0) : a) && i < a; ++i)"),
    ("e4m3_exponent_bias_8", "v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3_round_truncates", "r = ldexp(nearbyint(ldexp(a, -q)), q);", "r = ldexp(floor(ldexp(a, -q)), q);"),
    ("fp8_sum_of_rounded_p", "wsum += wj;", "wsum += pj;"),
    ("fp8_dropped_v_scale", "oi[t] += pj * desc_v * oracle_e4m3_decode(vrow[t]);",
     "oi[t] += pj * oracle_e4m3_decode(vrow[t]);"),
    ("fp8_causal_skips_diagonal", "const int n = causal ? i + 1 : N;", "const int n = causal ? i : N;"),
    ("philox_nine_rounds", "for (int r = 0; r < 10; ++r) {", "for (int r = 0; r < 9; ++r) {"),
    ("dropout_mask_transposed", "{(unsigned int)j >> 2, (unsigned int)i >> 2, (unsigned int)bh, offset}",
     "{(unsigned int)i >> 2, (unsigned int)j >> 2, (unsigned int)bh, offset}"),
    ("dropout_unscaled", "? 256.0 / (256.0 - p256) : 0.0;", "? 1.0 : 0.0;"),
    ("dropout_dv_unmasked", "dvj[t] += p * z * dOi[t];", "dvj[t] += p * dOi[t];"),
    ("dropout_dp_unmasked", "dp[j] = drop_factor(seed, offset, h, i, j, p256) * dot(dOi, v + hb + (size_t)j * d, d);",
     "dp[j] = dot(dOi, v + hb + (size_t)j * d, d);"),
    ("dp_uses_o_index", "dp[j] = dot(dOi, v + kb + (size_t)j * d, d);", "dp[j] = dot(dOi, v + kb + (size_t)i * d, d);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / "fa_oracle_mutant.c"
    src.write_text(text.replace(old, new))
    so = orc.build(force=True, src=str(src), out=str(tmp_path / "libmutant.so"))
    lib = orc.load(so)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
