"""Plant plausible mistakes in copies of the oracle and check that a pin catches each.

Each mutant is the oracle's C++ source with one edit (a dropped term, a wrong
index or sign, a swapped operand), compiled to a temporary shared object and run
against every pin on the CPU. The oracle itself is never modified.
"""
import os

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    "drop_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "group_modulo": ("const int64_t g = h / G;", "const int64_t g = h % n_kv_heads;"),
    "unnormalised_weights": ("const double p = std::exp(s[j] - l);",
                             "const double p = std::exp(s[j] - m);"),
    "lse_without_max": ("const double l = m + std::log(sum);\n            lse[bh] = l;",
                        "const double l = std::log(sum);\n            lse[bh] = l;"),
    "merge_lse_without_max": ("const double l = m + std::log(sum);\n        lse[r] = l;",
                              "const double l = std::log(sum);\n        lse[r] = l;"),
    "v_row_shifted": ("const uint16_t* v = v_pool + (int64_t(kv_indices[begin + j]) * n_kv_heads + g) * head_dim;",
                      "const uint16_t* v = v_pool + (int64_t(kv_indices[begin + (j + 1) % L]) * n_kv_heads + g) * head_dim;"),
    "k_layout_transposed": ("const uint16_t* k = k_pool + (int64_t(kv_indices[begin + j]) * n_kv_heads + g) * head_dim;",
                            "const uint16_t* k = k_pool + (int64_t(g) * pool_slots + kv_indices[begin + j]) * head_dim;"),
    "k_reads_v": ("for (int64_t d = 0; d < head_dim; ++d) dot += qd[d] * widen_bf16(k[d]);",
                  "for (int64_t d = 0; d < head_dim; ++d) dot += qd[d] * widen_bf16(k[d] ^ 0x8000);"),
    "merge_weight_vs_max": ("const double w = std::exp(lses[c * rows + r] - l);",
                            "const double w = std::exp(lses[c * rows + r] - m);"),
    "append_wrong_row": ("rows + i * row_elems,", "rows + ((i + 1) % n) * row_elems,"),
    "widen_truncates": ("uint32_t w = static_cast<uint32_t>(bits) << 16;",
                        "uint32_t w = static_cast<uint32_t>(bits & 0xFFFE) << 16;"),
    "prefill_position_ignores_prefix": ("const int64_t pos = L - C + (i - qo_indptr[b]);",
                                        "const int64_t pos = (i - qo_indptr[b]);"),
    "prefill_excludes_own_token": ("const int64_t n_seen = pos + 1;", "const int64_t n_seen = pos;"),
    "prefill_sees_next_token": ("const int64_t n_seen = pos + 1;",
                                "const int64_t n_seen = pos + 2 < L ? pos + 2 : L;"),
    "prefill_group_modulo": ("const int64_t kv_head = (ih % n_qo_heads) / G;",
                             "const int64_t kv_head = (ih % n_qo_heads) % n_kv_heads;"),
    "prefill_drop_scale": ("s[j] = qk * scale;", "s[j] = qk;"),
    "prefill_v_reads_k": ("orow[d] += w * widen_bf16(v_pool[row * head_dim + d]);",
                          "orow[d] += w * widen_bf16(k_pool[row * head_dim + d]);"),
    "prefill_weights_vs_max": ("const double w = std::exp(s[j] - log_denom);",
                               "const double w = std::exp(s[j] - smax);"),
    "query_head_offset": ("qd[d] = widen_bf16(q[bh * head_dim + d]);",
                          "qd[d] = widen_bf16(q[(b * n_qo_heads + (h ^ 1) % n_qo_heads) * head_dim + d]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_some_pin_catches_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut_src = tmp_path / "mutant.cpp"
    mut_src.write_text(src.replace(old, new))
    so = oracle.build(force=True, src=str(mut_src), out=str(tmp_path / "mutant.so"))
    orc = oracle.OracleLib(so)
    for pin in P.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            return  # caught
    pytest.fail(f"no pin caught mutant {name}")
