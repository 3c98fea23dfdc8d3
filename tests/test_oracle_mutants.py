"""Each plausible mistake planted in a copy of the oracle must make some pin fail.

The copy lives in a temporary directory and is compiled on the CPU; the oracle in the
repository is never modified.  This shows that the pins in ``oracle_pins.py`` are sharp
enough to catch a dropped term, a wrong sign or index, a transposed operand and the like.
"""
import os
import shutil

import pytest

import oracle as O
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(O.__file__), "oracle.cpp")

MUTANTS = {
    "drop_relu": ("const double relu = dot > 0.0 ? dot : 0.0;", "const double relu = dot;"),
    "relu_wrong_side": ("const double relu = dot > 0.0 ? dot : 0.0;", "const double relu = dot < 0.0 ? dot : 0.0;"),
    "drop_k_scale": ("out[j - lo] = static_cast<double>(k_scale[j]) * head_sum;", "out[j - lo] = head_sum;"),
    "drop_weight": ("head_sum += relu * static_cast<double>(w[t * H + h]);", "head_sum += relu;"),
    "weight_of_token0": ("head_sum += relu * static_cast<double>(w[t * H + h]);",
                         "head_sum += relu * static_cast<double>(w[h]);"),
    "q_transposed": ("dot += tab[q[(t * H + h) * D + d]] * tab[k[j * D + d]];",
                     "dot += tab[q[(t * D + d) * H + h]] * tab[k[j * D + d]];"),
    "k_wrong_row": ("dot += tab[q[(t * H + h) * D + d]] * tab[k[j * D + d]];",
                    "dot += tab[q[(t * H + h) * D + d]] * tab[k[(j > 0 ? j - 1 : 0) * D + d]];"),
    "bias_8": ("mag = std::ldexp(1.0 + static_cast<double>(m) / 8.0, e - 7);",
               "mag = std::ldexp(1.0 + static_cast<double>(m) / 8.0, e - 8);"),
    "no_subnormals": ("mag = std::ldexp(static_cast<double>(m) / 8.0, -6);", "mag = 0.0;"),
    "sign_ignored": ("return s ? -mag : mag;", "return mag;"),
    "tie_to_higher_index": ("return a.second < b.second;", "return a.second > b.second;"),
    "ascending_scores": ("if (a.first != b.first) return a.first > b.first;",
                         "if (a.first != b.first) return a.first < b.first;"),
    "output_not_sorted": ("std::sort(sel.begin(), sel.end());", ""),
    "pad_with_zero": (": -1;", ": 0;"),
    "window_end_inclusive": ("b = clamp64(ke[rows[r]], 0, N);", "b = clamp64(ke[rows[r]] + 1, 0, N);"),
    "quant_ties_up": ("if (err < best_err || (err == best_err && (c & 1) == 0)) {", "if (err <= best_err) {"),
    "quant_sign_dropped": ("const uint8_t sign = std::signbit(y) ? 0x80 : 0x00;", "const uint8_t sign = 0x00;"),
    "quant_scale_240": ("const float s = m / 448.0f;", "const float s = m / 240.0f;"),
    "quant_no_division": ("e4m3_nearest(x[static_cast<size_t>(j)] / s)", "e4m3_nearest(x[static_cast<size_t>(j)])"),
    "attn_sink_dropped": ("double den = sink ? std::exp(static_cast<double>(sink[h]) - m) : 0.0;", "double den = 0.0;"),
    "attn_scale_dropped": ("s[a] = scale * dot;", "s[a] = dot;"),
    "attn_no_row_max": ("for (double v : s) m = std::max(m, v);", ""),
    "attn_value_of_first_key": ("o[d] += e * bf16(kv_bf16[list[a] * D + d]);", "o[d] += e * bf16(kv_bf16[list[0] * D + d]);"),
    "attn_minus_one_as_key0": ("if (idx[t * K + i] >= 0) list.push_back(idx[t * K + i]);",
                               "list.push_back(idx[t * K + i] >= 0 ? idx[t * K + i] : 0);"),
    "attn_repeats_merged": ("if (idx[t * K + i] >= 0) list.push_back(idx[t * K + i]);",
                            "if (idx[t * K + i] >= 0 && std::find(list.begin(), list.end(), idx[t * K + i]) == list.end()) list.push_back(idx[t * K + i]);"),
    "attn_head_transposed": ("dot += bf16(q_bf16[(t * H + h) * D + d])", "dot += bf16(q_bf16[(h * T + t) * D + d])"),
    "attn_bwd_value_term_dropped": ("g[d] += scale * ds * qv(t, h, d) + pj * dov(t, h, d);",
                                    "g[d] += scale * ds * qv(t, h, d);"),
    "attn_bwd_key_term_unscaled": ("g[d] += scale * ds * qv(t, h, d) + pj * dov(t, h, d);",
                                   "g[d] += ds * qv(t, h, d) + pj * dov(t, h, d);"),
    "attn_bwd_delta_added": ("const double ds = pj * (dprob(t, h, j) - delta[th]);",
                             "const double ds = pj * (dprob(t, h, j) + delta[th]);"),
    "attn_bwd_dq_unscaled": ("for (int64_t d = 0; d < D; ++d) g[d] += scale * ds * kvv(list[a], d);",
                             "for (int64_t d = 0; d < D; ++d) g[d] += ds * kvv(list[a], d);"),
    "attn_bwd_no_delta_in_dq": ("const double ds = std::exp(s[a] - m) / z * (dp[a] - dl);",
                                "const double ds = std::exp(s[a] - m) / z * dp[a];"),
    "attn_bwd_sink_ignored": ("double z = sink ? std::exp(static_cast<double>(sink[h]) - m) : 0.0;\n      for (size_t a",
                              "double z = 0.0;\n      for (size_t a"),
    "attn_bwd_dsink_sign": ("acc += -psink[static_cast<size_t>(t * H + h)]", "acc += psink[static_cast<size_t>(t * H + h)]"),
    "attn_bwd_repeats_once": ("if (idx[t * K + i] >= 0) occ[static_cast<size_t>(idx[t * K + i])].push_back({t, i});",
                              "if (idx[t * K + i] >= 0 && (i == 0 || idx[t * K + i - 1] != idx[t * K + i])) "
                              "occ[static_cast<size_t>(idx[t * K + i])].push_back({t, i});"),
    "window_not_clamped": ("const int64_t a = clamp64(ks[rows[r]], 0, N), b = clamp64(ke[rows[r]], 0, N);",
                           "const int64_t a = ks[rows[r]], b = ke[rows[r]] < N ? ke[rows[r]] : N;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"anchor for {name} no longer in oracle.cpp"
    mutated = src.replace(old, new)
    path = tmp_path / "oracle_mut.cpp"
    path.write_text(mutated)
    lib = O.load_library(O.build(force=True, src=str(path), out=str(tmp_path / "liboracle_mut.so")))
    failures = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError) as e:  # noqa: PERF203
            failures.append(pin.__name__)
    assert failures, f"no pin caught mutant {name}"
