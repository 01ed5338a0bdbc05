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
    return sorted(set(re.findall(r"^\s*(?:int|const char\*|void|size_t)\s+(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_entry_points():
    names = declared_functions()
    assert {"fa_fwd", "fa_strerror", "fa_version", "fa_fwd_status", "fa_fwd_splitkv", "fa_splitkv_workspace_bytes",
            "fa_splitkv_heuristic"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_plain_c_consumer(lib, tmp_path):
    """include/fa.h is plain C: a C11 program compiled with -pedantic -Werror links
    libfa_gb300.so and gets the version, a message and a host-side argument error
    (no device work, so no GPU is needed)."""
    import shutil

    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
    src = tmp_path / "consumer.c"
    src.write_text(
        "#include <stdio.h>\n#include \"fa.h\"\n"
        "int main(void) {\n"
        "  printf(\"%d|%s|\", fa_version(), fa_strerror(FA_ERR_HEADDIM));\n"
        "  printf(\"%d\\n\", fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 128, 128, 96, 0.125f, 0, (cudaStream_t)0));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "consumer"
    lib_dir = os.path.dirname(fa.library_path())
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.dirname(HEADER),
                    "-I", cuda_inc, str(src), "-L", lib_dir, "-lfa_gb300", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.strip()
    version, message, status = out.split("|")
    assert int(version) == lib.fa_version()
    assert message == lib.fa_strerror(4).decode()
    assert int(status) == 1  # FA_ERR_NULL: null pointers are reported first


def test_version_and_strerror(lib):
    assert fa.fa_version() == 100
    assert fa.fa_strerror(0) == "ok"
    for code in range(1, 12):
        assert fa.fa_strerror(code) and fa.fa_strerror(code) != "unknown status"
    assert fa.fa_strerror(12345) == "unknown status"


def test_selftest_rejects_bad_arguments(lib):
    import ctypes

    w, n = ctypes.c_uint(), ctypes.c_ulonglong()
    assert lib.fa_selftest_wait(0, None, ctypes.byref(n), None) == 1  # FA_ERR_NULL
    assert lib.fa_selftest_wait(2, ctypes.byref(w), ctypes.byref(n), None) == 3  # FA_ERR_SHAPE


def test_probe_rejects_bad_arguments(lib):
    import ctypes

    assert lib.fa_probe_exp2(0, None, None) == 1  # FA_ERR_NULL, before any device call
    assert lib.fa_probe_exp2(2, ctypes.byref(ctypes.c_double()), None) == 3  # FA_ERR_SHAPE


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


def test_splitkv_workspace_size(lib):
    # n_kv = ceil(4096 / 128) = 32 tiles; 8 splits of 4 tiles; fp32 O [8, rows, 64] + L [8, rows]
    assert fa.fa_splitkv_workspace_bytes(1, 1, 4096, 4096, 64, 8) == 8 * 4096 * 65 * 4
    # 5 requested over 32 tiles -> 7 tiles per split -> 5 splits
    assert fa.fa_splitkv_workspace_bytes(2, 3, 100, 4096, 128, 5) == 5 * 600 * 129 * 4
    # more splits than tiles are capped at one split per tile
    assert fa.fa_splitkv_workspace_bytes(1, 1, 10, 200, 64, 16) == 2 * 10 * 65 * 4
    assert fa.fa_splitkv_workspace_bytes(1, 1, 10, 200, 96, 2) == 0
    assert fa.fa_splitkv_workspace_bytes(0, 1, 10, 200, 64, 2) == 0


@pytest.mark.parametrize("n_splits", [0, -1, 65])
def test_splitkv_rejects_split_count(lib, n_splits):
    st = fa.fa_fwd_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 64, 0.125, 0, n_splits, FAKE, 1 << 20, None)
    assert st == 3


def test_splitkv_host_validation(lib):
    st = fa.fa_fwd_splitkv(None, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 64, 0.125, 0, 2, FAKE, 1 << 20, None)
    assert st == 1
    st = fa.fa_fwd_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 96, 0.125, 0, 2, FAKE, 1 << 20, None)
    assert st == 4


def test_noalloc_host_validation(lib):
    st = fa.fa_fwd_splitkv_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 64, 0.125, 0, 0, None)
    assert st == 3
    # a request beyond the fixed array is refused before any device call
    st = fa.fa_fwd_splitkv_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 4096, 4096, 128, 0.125, 0, 8, None)
    assert st == 11


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(lse=None), 1), (dict(k=FAKE + 2), 2), (dict(d=96), 4), (dict(B=0), 3),
    (dict(causal=1, Nk=256), 5), (dict(scale=float("nan")), 9), (dict(Nq=0), 0),
    (dict(Nq=0, q=None, o=None, lse=None), 0),
    # oversized for the fixed array, but an argument error comes first
    (dict(q=None, H=64, Nq=4096, Nk=4096, d=128), 1), (dict(d=96, H=64, Nq=4096, Nk=4096), 4),
])
def test_noalloc_checks_match_workspace_entry_point(lib, kw, code):
    """The allocation-free call reports argument errors exactly as fa_fwd_splitkv
    does (the same checks in the same order), and Nq == 0 is a no-op that never
    touches the device, so both hold without a GPU."""
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, Nq=128, Nk=128, d=64, scale=0.125, causal=0,
             n_splits=4)
    a.update(kw)
    head = (a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"], a["scale"],
            a["causal"], a["n_splits"])
    assert fa.fa_fwd_splitkv_noalloc(*head, None) == code
    assert fa.fa_fwd_splitkv(*head, FAKE, 1 << 40, None) == code


def test_noalloc_single_slice_needs_no_array(lib):
    """One slice runs the plain kernel and uses no workspace, so a shape whose
    slice buffers would not fit the fixed array is not refused for that: the
    call gets past the size check (here to the device check, as no GPU is
    present or the fake pointers are not device memory)."""
    assert fa.fa_splitkv_workspace_bytes(1, 64, 4096, 4096, 128, 1) > fa.NOALLOC_SCRATCH_BYTES
    st = fa.fa_fwd_splitkv_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 4096, 4096, 128, 0.125, 0, 1, None)
    assert st in (6, 7, 10)  # FA_ERR_LAUNCH / FA_ERR_DEVICE / FA_ERR_POINTER, never FA_ERR_WORKSPACE


def test_window_host_validation(lib):
    assert fa.fa_fwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 256, 64, 0.125, -2, 0, None) == 3
    assert fa.fa_fwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 256, 64, 0.125, 0, -5, None) == 3
    assert fa.fa_fwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 256, 96, 0.125, 0, 0, None) == 4
    assert fa.fa_fwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 0, 256, 64, 0.125, 10, 0, None) == 0


def test_bwd_host_validation(lib):
    args = [FAKE] * 9
    assert fa.fa_bwd(*args, 1, 1, 128, 128, 64, 0.125, 0, FAKE, 1 << 20, None) != 1  # passes the NULL check
    assert fa.fa_bwd(None, *args[1:], 1, 1, 128, 128, 64, 0.125, 0, FAKE, 1 << 20, None) == 1
    assert fa.fa_bwd(*args, 1, 1, 128, 128, 64, 0.125, 0, None, 1 << 20, None) == 1
    assert fa.fa_bwd(*args, 1, 1, 128, 128, 96, 0.125, 0, FAKE, 1 << 20, None) == 4
    assert fa.fa_bwd(*args, 1, 1, 128, 256, 64, 0.125, 1, FAKE, 1 << 20, None) == 5
    assert fa.fa_bwd(*args, 1, 1, 0, 128, 64, 0.125, 0, FAKE, 1 << 20, None) == 3
    assert fa.fa_bwd(*args, 1, 1, 128, 128, 64, 0.125, 0, FAKE, 16, None) == 11
    assert fa.fa_bwd_workspace_bytes(2, 3, 200) == 2 * 6 * 256 * 4


def test_bwd_window_host_validation(lib):
    args = [FAKE] * 9
    assert fa.fa_bwd_window(*args, 1, 1, 128, 128, 64, 0.125, -2, 0, FAKE, 1 << 20, None) == 3
    assert fa.fa_bwd_window(*args, 1, 1, 128, 128, 64, 0.125, 0, -7, FAKE, 1 << 20, None) == 3
    assert fa.fa_bwd_window(None, *args[1:], 1, 1, 128, 128, 64, 0.125, 4, 0, FAKE, 1 << 20, None) == 1
    assert fa.fa_bwd_window(*args, 1, 1, 128, 128, 64, 0.125, 4, 0, None, 1 << 20, None) == 1
    assert fa.fa_bwd_window(*args, 1, 1, 128, 128, 96, 0.125, 4, 0, FAKE, 1 << 20, None) == 4
    assert fa.fa_bwd_window(*args, 1, 1, 0, 128, 64, 0.125, 4, 0, FAKE, 1 << 20, None) == 3
    assert fa.fa_bwd_window(*args, 1, 1, 128, 128, 64, float("nan"), 4, 0, FAKE, 1 << 20, None) == 9
    assert fa.fa_bwd_window(*args, 1, 1, 128, 128, 64, 0.125, 4, 0, FAKE, 16, None) == 11
    # a window needs no Nq == Nk: (-1, 0) with Nq != Nk passes every shape check
    st = fa.fa_bwd_window(*args, 1, 1, 128, 256, 64, 0.125, -1, 0, FAKE, 1 << 20, None)
    assert st not in (3, 5)
