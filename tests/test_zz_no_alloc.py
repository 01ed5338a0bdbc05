"""The allocation-free split-KV entry point (fa_fwd_splitkv_noalloc).

Some callers cannot allocate device memory (a host framework that owns the
whole device pool, a latency path that must not call cudaMalloc); this entry
point keeps its slice buffers in the library's own fixed device array, which
every call shares and which keeps whatever the previous call left in it.

The calls here run in a fixed order inside one test: first a large call that
fills most of the array with finite partial results, then a smaller causal
call with another slice count and head dimension (its empty causal slices
and its shorter partial rows sit where the first call left data), then a
one-slice call (the plain kernel, no array).  Each result is checked against
the fp64 oracle, and the causal one against the workspace entry point too, so
a partial left unwritten would read the first call's data and show up as a
mismatch with the oracle, not as a chance disagreement of two CUDA paths.

The file name makes pytest collect it last: a run that stops at the first
failure has already run every other test.  The test holds whether it runs
alone in a fresh process or after the rest of the suite.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_util import assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_19_gb300 as fa_mod
    from exact_attention_19_gb300 import build

    build.build()
    fa_mod.load()
    oracle.build()
    return fa_mod


def _to64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _noalloc(fa, w, n_splits, q, k, v):
    import torch

    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H,
                                   w.Nq, w.Nk, w.d, w.scale, int(w.causal), n_splits, stream)
    assert st == 0, fa.fa_strerror(st)
    torch.cuda.synchronize()
    st, word = fa.fa_fwd_status(None, clear=True)
    assert st == 0, f"kernel wait timed out, status word {word:#x}"
    return _to64(o), _to64(lse)


def _workspace(fa, w, n_splits, q, k, v):
    import torch

    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device="cuda")
    need = fa.fa_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, n_splits)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = fa.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H, w.Nq,
                           w.Nk, w.d, w.scale, int(w.causal), n_splits, ws.data_ptr(), need, stream)
    assert st == 0, fa.fa_strerror(st)
    torch.cuda.synchronize()
    return _to64(o), _to64(lse)


def test_noalloc_calls_in_a_row_match_the_oracle(fa):
    # (workload, requested slices): large first, then smaller, then one slice
    calls = [
        (synth.Workload("noalloc_large", 1, 2, 4096, 4096, 64, False, seed=71), 7),
        (synth.Workload("noalloc_causal", 2, 3, 1000, 1000, 128, True, sigma_q=4.0, seed=73), 5),
        (synth.Workload("noalloc_one_slice", 1, 2, 700, 900, 128, False, seed=75), 1),
    ]
    used = [fa.fa_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, s) for w, s in calls[:2]]
    # the first call fills most of the array, the second covers less of it
    assert fa.NOALLOC_SCRATCH_BYTES * 0.85 < used[0] <= fa.NOALLOC_SCRATCH_BYTES
    assert used[1] < used[0]
    for i, (w, n_splits) in enumerate(calls):
        qb, kb, vb = w.make()
        q, k, v = (to_device(x) for x in (qb, kb, vb))
        o, lse = _noalloc(fa, w, n_splits, q, k, v)
        o_ref, lse_ref = oracle.attention_fwd(qb, kb, vb, w.scale, w.causal)
        assert_close(o, lse, o_ref, lse_ref, f"noalloc call {i} ({w.name}, {n_splits} slices) vs oracle")
        if i == 1:
            o_ws, lse_ws = _workspace(fa, w, n_splits, q, k, v)
            assert_close(o, lse, o_ws, lse_ws, f"noalloc call {i} vs fa_fwd_splitkv")


def test_noalloc_rejects_oversized_request(fa):
    import torch

    # 16 heads x 4096 rows x 4 slices x 129 floats > 16 MiB
    B, H, N, d, n_splits = 1, 16, 4096, 128, 4
    assert fa.fa_splitkv_workspace_bytes(B, H, N, N, d, n_splits) > fa.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N,
                                   N, d, d ** -0.5, 0, n_splits, None)
    assert st == 11  # FA_ERR_WORKSPACE
