"""Planted mistakes in the oracle must be caught by its pins.

Each case copies oracle/oracle.cpp, plants one plausible mistake (a dropped term,
a wrong sign or index, a transposed operand), compiles the copy on the CPU and
runs the pins against it: at least one pin must fail.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.cpp")

MUTANTS = {
    "kv_head_modulo": ("int kvh = h / (p.Hq / p.Hkv);", "int kvh = h % p.Hkv;"),
    "scale_dropped": ("s[j - lo] = p.scale * acc;", "s[j - lo] = acc;"),
    "split_start_ceil": ("*lo = L * s / S;", "*lo = (L * s + S - 1) / S;"),
    "split_end_ceil": ("*hi = L * (s + 1) / S;", "*hi = (L * (s + 1) + S - 1) / S;"),
    "merge_weight_sign": ("double w = std::exp(ls[s] - tot);", "double w = std::exp(tot - ls[s]);"),
    "lse_max_dropped": ("*lse = m + std::log(z);", "*lse = std::log(z);"),
    "split_lse_max_dropped": ("double l = m + std::log(z);", "double l = std::log(z);"),
    "bhsd_heads_batch_swapped": ("(((int64_t)b * p.Hkv + kvh) * p.kv_rows + j)",
                                 "(((int64_t)kvh * p.B + b) * p.kv_rows + j)"),
    "varlen_rows_heads_swapped": ("(((int64_t)p.cu[b] + j) * p.Hkv + kvh)",
                                  "((int64_t)kvh * p.kv_rows + p.cu[b] + j)"),
    "f16_exponent_bias": ("e - 25);", "e - 24);"),
    "bf16_exponent_bias": ("e - 134);", "e - 133);"),
    "softmax_not_normalized": ("double pj = s[j] / z;", "double pj = s[j];"),
    "max_not_subtracted": ("s[j] = std::exp(s[j] - m);", "s[j] = std::exp(s[j]);"),
    "q_row_transposed": ("(((int64_t)b * p.tq + t) * p.Hq + h) * p.D",
                         "(((int64_t)h * p.tq + t) * p.B + b) * p.D"),
    "split_count_floor": ("int64_t sb = L == 0 ? 1 : (L + split_len - 1) / split_len;",
                          "int64_t sb = L == 0 ? 1 : (L + split_len / 2) / split_len;"),
    "split_count_cap_off_by_one": ("s_count[b] = (int32_t)(sb < max_splits ? sb : max_splits);",
                             "s_count[b] = (int32_t)(sb < max_splits ? sb : max_splits - 1);"),
    "token_sees_one_key_less": ("int64_t v = seq_len(p, b) - p.tq + t + 1;",
                                "int64_t v = seq_len(p, b) - p.tq + t;"),
    "split_ignores_causal_limit": ("if (hi > vis) hi = vis;", "if (false) hi = vis;"),
    "query_token_ignored": ("(((int64_t)b * p.tq + t) * p.Hq + h) * p.D",
                            "(((int64_t)b * p.tq) * p.Hq + h) * p.D"),
    # the row selector for several query tokens: the token index dropped, or token and head
    # swapped (the pin's shapes keep the swapped indices in range)
    "rows_mq_token_dropped": ("attend_row(p, rows_b[i], rows_t[i], rows_h[i], out + i * D, lse + i);",
                              "attend_row(p, rows_b[i], 0, rows_h[i], out + i * D, lse + i);"),
    "rows_mq_token_head_swapped": ("attend_row(p, rows_b[i], rows_t[i], rows_h[i], out + i * D, lse + i);",
                                   "attend_row(p, rows_b[i], rows_h[i], rows_t[i], out + i * D, lse + i);"),
    # per-sequence split counts with several tokens: the token index dropped from the split
    # step's row, or the sequence's count taken from its neighbour
    "var_mq_token_dropped": ("split_row(p, b, t, h, s_count[b], o, l);", "split_row(p, b, 0, h, s_count[b], o, l);"),
    "var_mq_count_of_neighbour": ("split_row(p, b, t, h, s_count[b], o, l);",
                                  "split_row(p, b, t, h, s_count[(b + 1) % B], o, l);"),
    "merge_skips_last_split": ("for (int s = 0; s < S; ++s) {\n            if (ls[s] == kNegInf) continue;",
                               "for (int s = 0; s + 1 < S; ++s) {\n            if (ls[s] == kNegInf) continue;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    count = src.count(old)
    assert count >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    path = tmp_path / "oracle_mutant.cpp"
    path.write_text(mutated)
    lib = oracle.load_library(oracle.compile_library(str(path), str(tmp_path / "libmut.so")))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
            break
    assert failed, f"planted mistake {name} passed every pin"
