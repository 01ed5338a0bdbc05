"""Each plausible slip in the oracle's C source trips at least one pin.

A copy of ``oracle/attention_ref.c`` with one planted mistake is compiled on
the CPU into a temporary library; the pins of ``oracle_pins`` run against it
and at least one must fail.  The real oracle is not touched.
"""
import os

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "attention_ref.c")

MUTANTS = {
    "drop_scale": ("s_row[j - j_first] = scale * dot;", "s_row[j - j_first] = dot;"),
    "causal_off_by_one": ("*j_last = i;", "*j_last = i + 1;"),
    "lse_without_max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "lse_log2": ("*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    "no_max_subtraction": ("p_row[t] = exp(s_row[t] - m);", "p_row[t] = exp(s_row[t]);"),
    "no_normalise": ("p_row[t] = p_row[t] / l;", "p_row[t] = p_row[t];"),
    "reversed_values": ("size_t vrow = kv_base + (size_t)(j_first + t) * (size_t)d;",
                        "size_t vrow = kv_base + (size_t)(j_last - t) * (size_t)d;"),
    "transposed_key_index": ("size_t krow = kv_base + (size_t)j * (size_t)d;",
                             "size_t krow = kv_base + (size_t)j;"),
    "skip_first_key_in_sum": ("double l = 0.0;\n  for (long t = 0; t < n_keys; ++t) {",
                              "double l = 0.0;\n  p_row[0] = 0.0;\n  for (long t = 1; t < n_keys; ++t) {"),
    "window_top_left": ("const long long diag = (long long)i + (long long)Nk - (long long)Nq;",
                        "const long long diag = (long long)i;"),
    "window_right_off_by_one": ("if (wr >= 0) *j_last = (long)(diag + wr < (long long)Nk ? diag + wr : (long long)Nk);",
                                "if (wr >= 0) *j_last = (long)(diag + wr + 1 < (long long)Nk ? diag + wr + 1 : (long long)Nk);"),
    "window_left_ignored": ("if (wl >= 0) *j_first", "if (wl >= 1 << 30) *j_first"),
    "sign_flip_logit": ("s_row[j - j_first] = scale * dot;", "s_row[j - j_first] = -scale * dot;"),
    "wrong_head_offset": ("size_t kv_base = (size_t)bh * (size_t)Nk * (size_t)d;",
                          "size_t kv_base = (size_t)(bh % 2) * (size_t)Nk * (size_t)d;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    # wrong_head_offset appears twice (all-rows and selected-rows entry points)
    assert text.count(old) >= 1, f"mutation anchor missing for {name}"
    mutated = text.replace(old, new)
    src = tmp_path / "mutant.c"
    src.write_text(mutated)
    lib_path = oracle.compile_oracle(str(src), str(tmp_path / "libmutant.so"))
    lib = oracle.load_library(lib_path)
    failures = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failures.append(pin.__name__)
        except Exception as e:  # a crash of the mutant counts as caught too
            failures.append(f"{pin.__name__}:{type(e).__name__}")
    assert failures, f"mutant {name} passed every pin"
