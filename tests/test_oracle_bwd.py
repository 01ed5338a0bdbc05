"""The fp64 backward oracle against finite differences, autograd, closed forms
and invariants, plus planted mistakes that must trip a pin (CPU only)."""
import os

import pytest

from oracle import backward, compile_oracle
from oracle_bwd_pins import BWD_PINS

SRC = os.path.join(os.path.dirname(backward.__file__), "attention_bwd_ref.c")


@pytest.fixture(scope="module")
def bwd_lib():
    return backward.load_library()


@pytest.mark.parametrize("pin", BWD_PINS, ids=[p.__name__ for p in BWD_PINS])
def test_bwd_oracle_pin(pin, bwd_lib):
    pin(bwd_lib)


MUTANTS = {
    "drop_D": ("const double ds = p_row[j] * (dp_row[j] - D);", "const double ds = p_row[j] * dp_row[j];"),
    "dq_without_scale": ("for (long c = 0; c < d; ++c) dq_row[c] *= scale;", "(void)0;"),
    "dk_without_scale": ("for (size_t x = 0; x < (size_t)Nk * (size_t)d; ++x) dk_h[x] *= scale;", "(void)0;"),
    "dv_uses_ds": ("dv_h[(size_t)j * (size_t)d + (size_t)c] += p_row[j] *",
                   "dv_h[(size_t)j * (size_t)d + (size_t)c] += ds *"),
    "D_from_v_not_o": ("for (long c = 0; c < d; ++c) D += elem(dout, dtype, q_base + (size_t)c) * o_row[c];",
                       "for (long c = 0; c < d; ++c) D += elem(dout, dtype, q_base + (size_t)c) * o_row[0];"),
    "causal_off_by_one": ("if (causal && i + 1 < Nk) n = i + 1;", "if (causal && i + 2 < Nk) n = i + 2;"),
    "dk_uses_k": ("dk_h[(size_t)j * (size_t)d + (size_t)c] += ds * elem(q, dtype, q_base + (size_t)c);",
                  "dk_h[(size_t)j * (size_t)d + (size_t)c] += ds * elem(k, dtype, krow + (size_t)c);"),
    "softmax_unnormalised": ("for (long j = lo; j < n; ++j) p_row[j] /= l;", "(void)l;"),
    "window_left_off_by_one": ("if (wl >= 0 && i + s - wl > lo) lo = i + s - wl;",
                               "if (wl >= 0 && i + s - wl + 1 > lo) lo = i + s - wl + 1;"),
    "window_right_off_by_one": ("if (wr >= 0 && i + s + wr + 1 < n) n = i + s + wr + 1;",
                                "if (wr >= 0 && i + s + wr < n) n = i + s + wr;"),
    "window_top_left": ("const long s = Nk - Nq;", "const long s = 0;"),
    "window_sides_swapped": ("if (wl >= 0 && i + s - wl > lo) lo = i + s - wl;",
                             "if (wr >= 0 && i + s - wr > lo) lo = i + s - wr;"),
    "empty_window_sees_all": ("  if (n < lo) n = lo;", "  if (n < lo) {\n    lo = 0;\n    n = Nk;\n  }"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_bwd_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"anchor missing for {name}"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = backward.load_library(compile_oracle(str(src), str(tmp_path / "libmutant.so")))
    failures = []
    for pin in BWD_PINS:
        try:
            pin(lib)
        except AssertionError:
            failures.append(pin.__name__)
    assert failures, f"mutant {name} passed every pin"
