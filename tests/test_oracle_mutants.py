"""Plausible mistakes planted in copies of the oracle's source must each trip at
least one pin.  The copies are compiled into a temporary directory; the oracle
itself is never modified."""
import os

import pytest

import oracle
import oracle_checks as C

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

# (name, text in the oracle, replacement)
MUTANTS = [
    ("window_off_by_one", "i - window + 1 > 0) ? i - window + 1", "i - window > 0) ? i - window"),
    ("gqa_modulo", "int kvh = h / G;\n                double *o = out + ((size_t)tok * Hq + h) * D;\n                for (int d = 0; d < D; d++) {",
     "int kvh = h % num_kv_heads;\n                double *o = out + ((size_t)tok * Hq + h) * D;\n                for (int d = 0; d < D; d++) {"),
    ("scale_divisor_128", "amax / 127.0f", "amax / 128.0f"),
    ("round_truncate", "nearbyintf(x[d] / scale)", "truncf(x[d] / scale)"),
    ("round_half_away", "nearbyintf(x[d] / scale)", "roundf(x[d] / scale)"),
    ("slot_offset_flipped", "int blk = s / S, off = s % S;", "int blk = s / S, off = S - 1 - s % S;"),
    ("table_walk_offset", "return ((long)phys * c->H + kvh) * c->S + j % c->S;",
     "return ((long)phys * c->H + kvh) * c->S + (j + 1) % c->S;"),
    ("missing_sm_scale", "s[j] = sm_scale * dot;", "s[j] = dot;"),
    ("query_position_shift", "int i = L - C + ci; /* position of this query */",
     "int i = L - C + ci + 1; /* position of this query */"),
    ("online_no_rescale", "l *= corr;", "l *= 1.0;"),
    ("merge_unweighted_l", "den += w * pl[p];", "den += pl[p];"),
    ("f16_exponent_bias", "e - 25", "e - 24"),
    ("bf16_shift", "(uint32_t)b << 16", "(uint32_t)b << 15"),
    ("f16_subnormal", "ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    ("clamp_126", "if (r > 127.0f)\n            r = 127.0f;", "if (r > 126.0f)\n            r = 126.0f;"),
    ("write_k_into_v", "void *cache = which ? v_cache : k_cache;", "void *cache = which ? k_cache : k_cache;"),
    ("dequant_no_scale", "out[d] = (double)codes[d] * scale;", "out[d] = (double)codes[d];"),
    ("linear_no_scale", "s += xv * ((double)codes[(size_t)i * k + j] * (double)scales[i]);",
     "s += xv * (double)codes[(size_t)i * k + j];"),
    ("linear_scale_of_next_channel", "s += xv * ((double)codes[(size_t)i * k + j] * (double)scales[i]);",
     "s += xv * ((double)codes[(size_t)i * k + j] * (double)scales[(i + 1) % n]);"),
    ("linear_bias_dropped", "            if (has_bias)\n                s +=", "            if (0)\n                s +="),
    ("linear_x_type_swapped",
     "double xv = x_dtype == PAO_BF16 ? pao_bf16_to_double(xb) : pao_f16_to_double(xb);",
     "double xv = x_dtype == PAO_BF16 ? pao_f16_to_double(xb) : pao_bf16_to_double(xb);"),
    ("weights_scale_slot_shift", "pao_quantize_row(row, k, codes + (size_t)i * k, scales + i);",
     "pao_quantize_row(row, k, codes + (size_t)i * k, scales + (i + 1) % n);"),
    ("causal_mask_off", "*hi = i < L - 1 ? i : L - 1;", "*hi = L - 1;"),
    ("window_of_one_ignored", "*lo = (window > 0 && i - window + 1 > 0)",
     "*lo = (window > 1 && i - window + 1 > 0)"),
    ("v_dequantised_with_k_scale", "(double)(which ? c->v_scale : c->k_scale)[r]",
     "(double)(which ? c->k_scale : c->k_scale)[r]"),
    ("v_scale_stored_in_k_scales", "float *sc = which ? v_scale : k_scale;",
     "float *sc = which ? k_scale : k_scale;"),
    ("online_acc_not_rescaled", "op[d] *= corr;", "op[d] *= 1.0;"),
    ("segment_last_key_dropped", "for (int j = j0; j <= j1; j++) {\n                            long r",
     "for (int j = j0; j < j1; j++) {\n                            long r"),
    ("merge_o_unweighted", "o[d] += w * po[(size_t)p * D + d];", "o[d] += po[(size_t)p * D + d];"),
    ("amax_signed", "float a = fabsf(x[d]);", "float a = x[d];"),
    ("negative_clamp_126", "if (r < -127.0f)\n            r = -127.0f;",
     "if (r < -126.0f)\n            r = -126.0f;"),
    ("linear_bias_as_f16", "s += x_dtype == PAO_BF16 ? pao_bf16_to_double(bias[i])",
     "s += x_dtype == PAO_F16 ? pao_bf16_to_double(bias[i])"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation site not found: " + name
    mut = tmp_path / ("pa_oracle_" + name + ".c")
    mut.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(force=True, src=str(mut), out=str(tmp_path / "lib.so")))
    for check in C.ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            return
    pytest.fail("no pin caught mutant " + name)
