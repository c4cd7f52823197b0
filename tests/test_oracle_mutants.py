"""The pins are strong enough: each plausible mistake planted in a copy of the oracle
source (a dropped term, a wrong sign, bias or index, swapped operands) makes at least
one pin fail.  The mistakes are planted only in throw-away copies, on the CPU."""
import os

import pytest

import oracle_pins
from oracle import oracle as O

MUTANTS = {
    "cutoff_off_by_one": ("int64_t cut = L - qlen + tok + 1;", "int64_t cut = L - qlen + tok;"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal_exp": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "bf16_bias": ("ldexp(1.0 + (double)m / 128.0, e - 127)",
                  "ldexp(1.0 + (double)m / 128.0, e - 126)"),
    "block_table_first_page_only": ("p / pb->page_size]", "0]"),
    "slot_shift": ("const int64_t slot = p % pb->page_size;",
                   "const int64_t slot = (p + 1) % pb->page_size;"),
    "per_token_scale_first_slot": ("scale_pt[tok_index]",
                                   "scale_pt[(phys * pb->num_kv_heads + h) * pb->page_size]"),
    "scalar_v_scale_dropped": ("return x * scale_scalar;", "return x;"),
    "sm_scale_dropped": ("scores[j] = pb->sm_scale * acc;", "scores[j] = acc;"),
    "v_reads_k": ("pb->v_cache, pb->v_scale, pb->v_scale_scalar",
                  "pb->k_cache, pb->k_scale, pb->k_scale_scalar"),
    "sparse_ignores_cutoff": ("if (p < lim) keys[n++] = p;", "if (p < L) keys[n++] = p;"),
    "sparse_padding_as_page0": ("if (sp < 0) continue;", "if (sp < 0) sp = 0;"),
    "head_map_transposed": ("const int head = h * g + i;",
                            "const int head = i * pb->num_kv_heads + h;"),
    "kv_head_stride_dropped": ("(phys * pb->num_kv_heads + h) * pb->page_size + o",
                               "(phys * pb->num_kv_heads) * pb->page_size + o"),
    "row_tok_reversed": ("const int64_t row = row0 + tok;",
                         "const int64_t row = row0 + (qlen - 1 - tok);"),
    "lse_without_max": ("smax + log(z)", "log(z)"),
    "softmax_sign": ("exp(scores[j] - smax)", "exp(smax - scores[j])"),
    "enc_ties_away": ("double m = nearbyint((ldexp(a, -ex) - 1.0) * 8.0);",
                      "double m = round((ldexp(a, -ex) - 1.0) * 8.0);"),
    "enc_truncates": ("double m = nearbyint((ldexp(a, -ex) - 1.0) * 8.0);",
                      "double m = floor((ldexp(a, -ex) - 1.0) * 8.0);"),
    "enc_subnormal_step": ("double m = nearbyint(ldexp(a, 9));",
                           "double m = nearbyint(ldexp(a, 8));"),
    "enc_no_saturation": ("if (a >= 448.0) return sign | 0x7E;", "if (a >= 480.0) return sign | 0x7F;"),
    "quant_scale_447": ("volatile float s = amax / 448.0f;", "volatile float s = amax / 447.0f;"),
    "quant_fp32_product": ("const double q = (double)bf16_to_f32(x[d]) / (double)s;",
                           "volatile float inv_m = 448.0f / amax;\n"
                           "    volatile float q_m = bf16_to_f32(x[d]) * inv_m;\n"
                           "    const double q = q_m;"),
    "quant_fp32_quotient": ("const double q = (double)bf16_to_f32(x[d]) / (double)s;",
                            "volatile float q_m = bf16_to_f32(x[d]) / s;\n"
                            "    const double q = q_m;"),
    "quant_slot_offset": ("const int64_t page = s / page_size, o = s % page_size;",
                          "const int64_t page = s / page_size, o = (s + 1) % page_size;"),
    "quant_head_stride": ("const int64_t row = (page * num_kv_heads + h) * page_size + o;",
                          "const int64_t row = (page * num_kv_heads) * page_size + o;"),
    "quant_v_from_k": ("quantize_row(v_new + src,", "quantize_row(k_new + src,"),
    "quant_skips_counted": ("      ++bad;\n      continue;", "      continue;"),
    "merge_exp_without_max": ("const double w = exp(l - M);", "const double w = exp(l);"),
    "merge_lse_without_max": ("lse[v] = M + log(z);", "lse[v] = log(z);"),
    "merge_unnormalised": ("for (int32_t d = 0; d < dim; ++d) o[d] /= z;", ""),
    "merge_first_part_only": ("      if (l == -INFINITY) continue;\n      const double w",
                              "      if (l == -INFINITY || i > 0) continue;\n      const double w"),
    "index_cutoff_off_by_one": ("int64_t lim = L - qlen + tok + 1;", "int64_t lim = L - qlen + tok;"),
    "index_natural_log": ("S[b] = m + log2(z);", "S[b] = m + log(z);"),
    "index_no_forced_page": ("if (nb > 0 && pb->topk > 0) sel[cnt++] = (int32_t)(nb - 1);", ""),
    "index_ties_to_higher": ("if (best < 0 || S[b] > S[best]) best = b;",
                             "if (best < 0 || S[b] >= S[best]) best = b;"),
    "index_scale_dropped": ("(double)pb->k_scale[(int64_t)phys * ps + o] : 1.0;", "1.0 : 1.0;"),
    "index_first_head_only": ("for (int64_t i = 0; i < n * H; ++i) z += exp2(s[i] - m);",
                              "for (int64_t i = 0; i < n; ++i) z += exp2(s[i] - m);"),
    "index_no_log2e": ("const double v = pb->sm_scale * log2e * acc;",
                       "const double v = pb->sm_scale * acc;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = O.source_text()
    assert old in src, f"mutation anchor for {name} not found"
    lib = O.OracleLib(O.build_variant(src.replace(old, new), str(tmp_path / f"m_{name}.so")))
    failed = []
    for pin in oracle_pins.PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
            break
    assert failed, f"no pin caught mutant {name}"
