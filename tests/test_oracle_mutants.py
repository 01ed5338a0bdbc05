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
    "drop_scale": ("s_row[j] = scale * dot;", "s_row[j] = dot;"),
    "causal_off_by_one": ("n_keys = i + 1;", "n_keys = i + 2 < Nk ? i + 2 : Nk;"),
    "lse_without_max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "lse_log2": ("*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    "no_max_subtraction": ("p_row[j] = exp(s_row[j] - m);", "p_row[j] = exp(s_row[j]);"),
    "no_normalise": ("p_row[j] = p_row[j] / l;", "p_row[j] = p_row[j];"),
    "reversed_values": ("size_t vrow = kv_base + (size_t)j * (size_t)d;",
                        "size_t vrow = kv_base + (size_t)(n_keys - 1 - j) * (size_t)d;"),
    "transposed_key_index": ("size_t krow = kv_base + (size_t)j * (size_t)d;",
                             "size_t krow = kv_base + (size_t)j;"),
    "skip_first_key_in_sum": ("double l = 0.0;\n  for (long j = 0; j < n_keys; ++j) {",
                              "double l = 0.0;\n  p_row[0] = 0.0;\n  for (long j = 1; j < n_keys; ++j) {"),
    "sign_flip_logit": ("s_row[j] = scale * dot;", "s_row[j] = -scale * dot;"),
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
