"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re
import subprocess

import pytest

import exact_attention_19_gb300 as fa
from exact_attention_19_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\*|void)\s+(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_entry_points():
    names = declared_functions()
    assert {"fa_fwd", "fa_strerror", "fa_version", "fa_fwd_status"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_version_and_strerror(lib):
    assert fa.fa_version() == 100
    assert fa.fa_strerror(0) == "ok"
    for code in range(1, 11):
        assert fa.fa_strerror(code) and fa.fa_strerror(code) != "unknown status"
    assert fa.fa_strerror(12345) == "unknown status"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def call(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, Nq=128, Nk=128, d=64, scale=0.125,
                causal=0, stream=None)
    args.update(kw)
    return fa.fa_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["H"],
                     args["Nq"], args["Nk"], args["d"], args["scale"], args["causal"], args["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(lse=None), 1),
    (dict(k=FAKE + 2), 2), (dict(lse=FAKE + 4), 2),
    (dict(d=96), 4), (dict(d=0), 4),
    (dict(B=0), 3), (dict(H=-1), 3), (dict(Nk=0), 3), (dict(Nq=-5), 3), (dict(causal=2), 3),
    (dict(causal=1, Nq=128, Nk=256), 5),
    (dict(scale=0.0), 9), (dict(scale=-1.0), 9), (dict(scale=float("inf")), 9), (dict(scale=float("nan")), 9),
    (dict(B=1 << 16, H=1 << 15), 3), (dict(B=1 << 12, H=1 << 12, Nq=1 << 20, Nk=1 << 20), 3),
])
def test_host_validation(lib, kw, code):
    assert call(**kw) == code


def test_empty_query_is_a_noop(lib):
    assert call(Nq=0) == 0
    assert call(Nq=0, q=None, o=None, lse=None) == 0
    assert call(Nq=0, k=None) == 1
