"""CPU: plant plausible mistakes in a copy of the oracle's C source and check
that the pins catch every one of them (a dropped term, a wrong sign or index,
a transposed operand, a wrong head mapping, a wrong address term)."""
import os
import tempfile

import pytest

import oracle as oracle_pkg
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "attn_oracle.c")

# (name, text in the committed source, replacement)
MUTANTS = [
    ("dropped_rescale", "for (int t = 0; t < d; ++t) oi[t] *= corr;", ""),
    ("causal_excludes_diagonal", "if (causal && j > diag) return 0;", "if (causal && j >= diag) return 0;"),
    ("window_wrong_sign", "j < diag - (long)window", "j < diag + (long)window"),
    ("gqa_interleaved_heads", "long hk = h / G;  /* contiguous", "long hk = h % Hkv;  /* contiguous"),
    ("no_max_in_lse", "*lse_i = m + log(l);", "*lse_i = log(l);"),
    ("scores_use_v", "s[j] = scale * dot(qi, kh + j * d, d);", "s[j] = scale * dot(qi, vh + j * d, d);"),
    ("missing_scale", "s[j] = scale * dot(qi, kh + j * d, d);", "s[j] = dot(qi, kh + j * d, d);"),
    ("merge_weight_sign", "double w = lc[c] * exp(mc[c] - M) / L;", "double w = lc[c] * exp(M - mc[c]) / L;"),
    ("decode_no_head_offset", "physical * block_stride + hk * (long)block_size * d + offset * token_stride",
     "physical * block_stride + offset * token_stride"),
    ("decode_offset_by_block", "long offset = t % block_size;", "long offset = t / block_size;"),
    ("no_final_divide", "for (long j = 0; j < Nk; ++j) p[j] /= l;\n    /* O = P V */", "/* O = P V */"),
    ("bwd_no_normalisation", "for (long j = 0; j < Nk; ++j) p[j] /= l;\n                        /* dP row",
     "/* dP row"),
    ("blocked_sum_not_corrected", "l[i - i0] = corr * l[i - i0] + lsum;", "l[i - i0] = l[i - i0] + lsum;"),
    ("bwd_dropped_row_term", "double ds = p[j] * (dp[j] - row);", "double ds = p[j] * dp[j];"),
    ("bwd_dk_from_k", "dkj[t] += scale * ds * qi[t];", "dkj[t] += scale * ds * kj[t];"),
    ("bwd_dq_missing_scale", "dqi[t] += scale * ds * kj[t];", "dqi[t] += ds * kj[t];"),
    ("bwd_dv_from_dp", "dvj[t] += p[j] * doi[t];", "dvj[t] += dp[j] * doi[t];"),
    ("paged_prefill_no_head_offset", "off * token_stride + hk * (long)block_size * d;", "off * token_stride;"),
    ("paged_prefill_top_left_alignment", "kh, vh, i, qn, kn, d, scale", "kh, vh, i, kn, kn, d, scale"),
    ("paged_prefill_offset_by_block", "off = t % block_size;", "off = t / block_size;"),
    ("blocksparse_pattern_ignored", "&&\n                            block_listed(row_ptr, col_idx, i / block_q, j / block_k))",
     "&& 1)"),
    ("blocksparse_dense_mask_ignored", "if (key_allowed(i, j, Nq, Nk, causal, window) &&\n                            block_listed",
     "if (j < Nk &&\n                            block_listed"),
    ("blocksparse_key_block_by_query_size", "i / block_q, j / block_k))", "i / block_q, j / block_q))"),
    ("e4m3_exponent_bias_8", "(double)mantissa / 8.0, exponent - 7)", "(double)mantissa / 8.0, exponent - 8)"),
    ("e4m3_subnormal_scale", "ldexp((double)mantissa / 8.0, -6);", "ldexp((double)mantissa / 8.0, -7);"),
    ("e4m3_no_nan_code", "if (exponent == 15 && mantissa == 7) return NAN;", ""),
    ("fp8_v_not_transposed", "vt8[(bh * d + t) * Nk + j]", "vt8[(bh * Nk + j) * d + t]"),
    ("fp8_missing_k_scale", "k[i] = k_descale * oracle_e4m3_value(k8[i]);", "k[i] = oracle_e4m3_value(k8[i]);"),
]


def test_mutants_are_distinct_edits():
    src = open(SRC).read()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, f"{name}: pattern must occur exactly once"


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib_path = os.path.join(tmp, "libmutant.so")
        oracle_pkg.compile_source(path, lib_path)
        orc = oracle_pkg.Oracle(oracle_pkg.load(lib_path))
        caught = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(orc)
            except (AssertionError, ValueError, FloatingPointError):
                caught.append(pin.__name__)
        assert caught, f"no pin caught the planted mistake '{name}'"
