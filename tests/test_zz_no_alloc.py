"""The allocation-free split-KV entry point (fa_fwd_splitkv_noalloc).

Some callers cannot allocate device memory (a host framework that owns the
whole device pool, a latency path that must not call cudaMalloc); this entry
point keeps its slice buffers in the library's own fixed device array.  Its
output must match the workspace entry point (fa_fwd_splitkv) within the
parity tolerance, on two calls in a row, so that state left in the shared
array by one call cannot leak into the next.

The file name makes pytest collect it last: a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest

import synth
from parity_util import assert_close, o_err, lse_err, to_device

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
    return fa_mod


def _run_both(fa, w, n_splits):
    import torch

    q, k, v = (to_device(x) for x in w.make())
    stream = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr())
    shape = (w.B, w.H, w.Nq, w.Nk, w.d, w.scale, int(w.causal), n_splits)

    o_ws, l_ws = torch.empty_like(q), torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device="cuda")
    need = fa.fa_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, n_splits)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = fa.fa_fwd_splitkv(*args, o_ws.data_ptr(), l_ws.data_ptr(), *shape, ws.data_ptr(), need, stream)
    assert st == 0, fa.fa_strerror(st)

    o_na, l_na = torch.empty_like(q), torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd_splitkv_noalloc(*args, o_na.data_ptr(), l_na.data_ptr(), *shape, stream)
    assert st == 0, fa.fa_strerror(st)
    torch.cuda.synchronize()
    st, word = fa.fa_fwd_status(None, clear=True)
    assert st == 0, f"kernel wait timed out, status word {word:#x}"
    to64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    return to64(o_na), to64(l_na), to64(o_ws), to64(l_ws)


@pytest.mark.parametrize("case", [
    # (workload, slices): two calls in a row with different shapes and inputs
    [(synth.WORKLOADS["single_head_4096_d64"], 8),
     (synth.Workload("noalloc_causal", 2, 3, 1000, 1000, 128, True, sigma_q=4.0, seed=73), 5)],
])
def test_noalloc_matches_workspace_entry_point(fa, case):
    for w, n_splits in case:
        o, l, o_ref, l_ref = _run_both(fa, w, n_splits)
        assert_close(o, l, o_ref, l_ref, f"noalloc {w.name}")
        assert o_err(o, o_ref) <= 1e-2 and lse_err(l, l_ref) <= 1e-3


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
