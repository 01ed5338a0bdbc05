"""CUDA path vs the fp64 oracle on the same seeded bf16 inputs (GB300 only).

Every call goes through the C ABI (libfa_gb300.so via the ctypes binding).
Element-wise at sizes the oracle finishes in seconds (several tiles, ragged
tails); sampled rows at the full benchmark sizes in the launch configuration
the bench times.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from parity_util import assert_close, run_gpu, sample_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_19_gb300 as fa
    from exact_attention_19_gb300 import build

    build.build()
    fa.load()
    yield


_ORACLE_CACHE = {}


def _oracle_full(w: synth.Workload, q, k, v):
    key = (w.B, w.H, w.Nq, w.Nk, w.d, w.causal, w.sigma_q, w.seed)
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = oracle.attention_fwd(q, k, v, w.scale, w.causal)
    return _ORACLE_CACHE[key]


def _check_full(w: synth.Workload, n_splits=None):
    q, k, v = w.make()
    o, lse = run_gpu(q, k, v, w.scale, w.causal, n_splits)
    o_ref, lse_ref = _oracle_full(w, q, k, v)
    return assert_close(o, lse, o_ref, lse_ref, f"{w.name} n_splits={n_splits}")


# --- the three small workloads, every element ---------------------------------
# n_splits None: the library's choice (split-KV for the two single-head
# workloads); 1: the single-pass kernel.
@pytest.mark.parametrize("n_splits", [None, 1])
@pytest.mark.parametrize("name", ["single_head_256_d64", "single_head_4096_d64", "gpt2_small_causal_1024_d64"])
def test_workload_elementwise(name, n_splits):
    _check_full(synth.WORKLOADS[name], n_splits)


# --- ragged and odd shapes, every element --------------------------------------
RAGGED = [1, 2, 63, 65, 127, 129, 255, 257, 383, 1000]


@pytest.mark.parametrize("n_splits", [None, 1])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", RAGGED)
def test_ragged_square(n, d, causal, n_splits):
    _check_full(synth.Workload(f"ragged{n}", 1, 2, n, n, d, causal, seed=500 + n), n_splits)


# causal attention at d = 64 over at most 2048 keys runs one query tile per CTA
# (two CTAs per SM), longer key ranges two: both sides of the switch, every element
@pytest.mark.parametrize("n", [2047, 2048, 2049])
def test_causal_d64_tile_count_switch(n):
    _check_full(synth.Workload(f"switch{n}", 2, 3, n, n, 64, True, seed=900 + n), 1)


@pytest.mark.parametrize("n_splits", [None, 1])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nq,nk", [(100, 300), (513, 64), (1, 1000), (256, 129), (700, 4097)])
def test_rectangular_noncausal(nq, nk, d, n_splits):
    _check_full(synth.Workload(f"rect{nq}x{nk}", 2, 1, nq, nk, d, False, seed=900 + nq), n_splits)


# --- split-KV: forced slice counts, merge against the oracle ------------------
@pytest.mark.parametrize("n_splits", [2, 3, 5, 16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_forced(n_splits, d, causal):
    # 1000 keys = 8 K/V tiles (ragged tail): slices of 4, 3, 2 and 1 tiles; under
    # the causal mask the light query tiles see only some slices (empty partials)
    _check_full(synth.Workload("split", 2, 3, 1000, 1000, d, causal, seed=71), n_splits)


# d = 64 split-KV launches one query tile per CTA when the grid of tile pairs x
# slices would fill under half of the SMs or more than all of them, else pairs;
# these shapes land on each side on a 148- to 152-SM part
@pytest.mark.parametrize("shape", [
    (1, 1, 4096, False, 8),   # 128 pair CTAs: pairs
    (1, 1, 1000, False, 3),   # 12: single tiles
    (1, 3, 333, True, 2),     # 12: single tiles, causal (light tiles see one slice)
    (2, 1, 4097, False, 5),   # 170 > SMs: single tiles, one-row ragged tail
    (1, 1, 1024, True, 4),    # 16: single tiles, causal
    (2, 4, 2048, False, 2),   # 128: pairs
])
def test_splitkv_cta_shapes(shape):
    B, H, n, causal, n_splits = shape
    _check_full(synth.Workload(f"split_cta{n}", B, H, n, n, 64, causal, seed=73 + n), n_splits)


@pytest.mark.parametrize("d", [64, 128])
def test_splitkv_wide_logits(d):
    # the merge weights 2^(L_s - L) span many orders of magnitude
    _check_full(synth.Workload("split_wide", 1, 2, 2000, 2000, d, True, sigma_q=20.0, seed=72), 7)


def test_splitkv_workspace_errors():
    import torch

    import exact_attention_19_gb300 as fa

    q = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 256), dtype=torch.float32, device="cuda")
    need = fa.fa_splitkv_workspace_bytes(1, 1, 256, 256, 64, 2)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 256, 256, 64, 0.125, 0, 2)
    assert fa.fa_fwd_splitkv(*args, None, need, None) == 11
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need - 4, None) == 11
    host_ws = torch.empty(need, dtype=torch.uint8)
    assert fa.fa_fwd_splitkv(*args, host_ws.data_ptr(), need, None) == 10
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr() + 4, need, None) == 2
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need, None) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("d", [64, 128])
def test_multi_batch_head(d):
    _check_full(synth.Workload("bh", 3, 5, 200, 200, d, True, seed=31))
    _check_full(synth.Workload("bh", 2, 7, 130, 390, d, False, seed=32))


# thousands of short heads: grids of several thousand small CTAs (single-tile CTAs
# for the causal d = 64 case), causal scheduling groups far smaller than B * H,
# and a ragged second query tile of two rows in every head
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_many_short_heads(d, causal):
    _check_full(synth.Workload("many", 16, 128, 130, 130, d, causal, seed=40 + d + causal), 1)


# the persistent kernel (a single pass without a mask): more work units
# than multiprocessors, so each CTA streams several units through one K/V ring
# and one MMA stream; units whose second query tile is absent (Nq = 300: the
# second pair holds one tile) or two rows long, key counts that are not tile
# multiples, one key tile (S of the next unit issued in a unit's first step),
# and fewer units than multiprocessors
# (d = 64 takes the persistent kernel for up to 2048 keys: its two Q buffers
# per tile rotate across units)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", [(2, 80, 300, 1000), (1, 160, 256, 640), (3, 53, 130, 2000), (4, 40, 129, 100),
                                   (1, 3, 1000, 4097)])
def test_persistent_unit_stream(shape, d):
    B, H, nq, nk = shape
    _check_full(synth.Workload("persist", B, H, nq, nk, d, False, seed=50 + H + d), 1)
    _check_full(synth.Workload("persist_wide", B, H, nq, nk, d, False, sigma_q=8.0, seed=60 + H + d))


# causal d = 64 beyond 2048 keys: with at least 6 query-tile pairs per SM the
# persistent kernel under cluster launch control (a running CTA takes over the
# units of CTAs not yet started; units of 1 to N / 128 K/V tiles, a ragged last
# tile); with fewer, single query tiles (the last two shapes)
@pytest.mark.parametrize("shape", [(4, 64, 2200), (8, 16, 3000), (1, 20, 3000), (3, 7, 2049)])
def test_causal_d64_dynamic_schedule(shape):
    B, H, n = shape
    _check_full(synth.Workload("clc", B, H, n, n, 64, True, seed=70 + H), 1)
    _check_full(synth.Workload("clc_wide", B, H, n, n, 64, True, sigma_q=8.0, seed=80 + H), 1)


# causal d = 128 with at least 20 query-tile pairs per SM: the same dynamic
# schedule (16 x 48 heads of 1100 rows: 3840 pairs, a ragged last tile)
def test_causal_d128_dynamic_schedule():
    _check_full(synth.Workload("clc128", 16, 48, 1100, 1100, 128, True, seed=91), 1)


def test_causal_d64_dynamic_schedule_full_size():
    w = synth.WORKLOADS["long_8192_d64"].with_(name="long_8192_d64_causal", causal=True)
    q, k, v = w.make()
    o, lse = run_gpu(q, k, v, w.scale, True)
    rows = sample_rows(w.B, w.H, w.Nq, 300, seed=w.seed)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, rows, w.scale, True)
    assert_close(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, w.name)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    # row 0 of every head sees key 0 only: O = V[0] exactly
    assert np.array_equal(o[:, :, 0, :], synth.bf16_to_f32(v[:, :, 0, :]).astype(np.float64))


# --- degenerate and numerically hard cases -----------------------------------
@pytest.mark.parametrize("d", [64, 128])
def test_single_key(d):
    w = synth.Workload("nk1", 1, 3, 300, 1, d, False, seed=3)
    q, k, v = w.make()
    o, lse = run_gpu(q, k, v, w.scale, False)
    # closed form: O = V[0] exactly (bf16 V reproduced exactly), LSE = scale * q.k0
    vv = synth.bf16_to_f32(v).astype(np.float64)
    assert np.array_equal(o, np.broadcast_to(vv[:, :, :1, :], o.shape))
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, w.scale, False)
    assert_close(o, lse, o_ref, lse_ref, "nk1")


@pytest.mark.parametrize("causal", [False, True])
def test_zero_keys_give_uniform_weights(causal):
    n, d = 300, 128
    q = synth.normal_bf16(4, 0, (1, 1, n, d))
    k = np.zeros((1, 1, n, d), dtype=np.uint16)
    v = synth.normal_bf16(4, 2, (1, 1, n, d))
    o, lse = run_gpu(q, k, v, 1.0 / math.sqrt(d), causal)
    cnt = np.arange(1, n + 1) if causal else np.full(n, n)
    assert np.max(np.abs(lse[0, 0] - np.log(cnt))) < 1e-5
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, 1.0 / math.sqrt(d), causal)
    assert_close(o, lse, o_ref, lse_ref, "zero keys")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("sigma_q", [8.0, 30.0])
def test_wide_logits_force_rescaling(d, sigma_q):
    """Large, spread logits: the running maximum moves by far more than tau many times."""
    w = synth.Workload("wide", 1, 2, 1100, 1100, d, True, sigma_q=sigma_q, seed=41)
    _check_full(w)
    _check_full(w.with_(causal=False, seed=42))


def test_increasing_logits_rescale_every_tile():
    """Keys sorted so that every new tile raises each row's maximum."""
    n, d = 1024, 64
    rng = np.random.default_rng(8)
    q = np.zeros((1, 1, n, d), dtype=np.float32)
    q[..., 0] = 1.0
    k = np.zeros((1, 1, n, d), dtype=np.float32)
    k[..., 0] = np.linspace(-40.0, 40.0, n)  # logits grow along the key axis
    v = rng.normal(size=(1, 1, n, d)).astype(np.float32)
    bits = [synth.f32_to_bf16_bits(x) for x in (q, k, v)]
    for causal in (False, True):
        o, lse = run_gpu(*bits, 1.0, causal)
        o_ref, lse_ref = oracle.attention_fwd(*bits, 1.0, causal)
        assert_close(o, lse, o_ref, lse_ref, f"increasing causal={causal}")


def test_constant_values():
    w = synth.Workload("const", 1, 2, 777, 777, 128, True, seed=5)
    q, k, _ = w.make()
    v = np.full(k.shape, synth.f32_to_bf16_bits(np.float32([1.5]))[0], dtype=np.uint16)
    o, _ = run_gpu(q, k, v, w.scale, True)
    assert np.max(np.abs(o - 1.5)) <= 1.5 * 2 ** -8


def test_empty_query_rows_noop():
    import torch

    import exact_attention_19_gb300 as fa

    q = torch.zeros((1, 1, 0, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 1, 5, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = fa.fwd(q, k, k)
    assert o.shape == (1, 1, 0, 64) and lse.shape == (1, 1, 0)


def test_deterministic():
    w = synth.Workload("det", 2, 3, 1000, 1000, 128, True, seed=9)
    q, k, v = w.make()
    o1, l1 = run_gpu(q, k, v, w.scale, True)
    o2, l2 = run_gpu(q, k, v, w.scale, True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("mode", ["causal_d128", "full_d128", "full_d128_o16", "causal_d64_single_tile", "full_d64", "full_d64_o16",
                                  "window_d128", "split_d64", "split_causal_d128"])
def test_outputs_not_written_outside(mode):
    """O and LSE embedded in larger guard-filled buffers: the guards stay untouched.

    O goes out through tiled tensor stores of whole 128-row tiles; the last
    tile of every head here is ragged (333 rows), so the stores must drop the
    rows past Nq of the last head (past the buffer) and of every other head
    (the next head's rows).  Covers each kernel instantiation's epilogue.
    full_d128_o16 places O 16 bytes off a 32-byte boundary: the persistent
    kernel's 32-byte row stores must give way to 16-byte ones there."""
    import torch

    import exact_attention_19_gb300 as fa

    d = 64 if "d64" in mode else 128
    causal = "causal" in mode
    B, H, N = 2, 3, 333
    w = synth.Workload("guard", B, H, N, N, d, causal, seed=10)
    q, k, v = w.make()
    tq, tk, tv = to_device(q), to_device(k), to_device(v)
    n_o, n_l = q.size, B * H * N
    pad_o, pad_l = (4096 + 8 if mode.endswith("o16") else 4096), 64  # 8 bf16 = 16 bytes
    big_o = torch.full((n_o + 2 * pad_o,), 7.0, dtype=torch.bfloat16, device="cuda")
    big_l = torch.full((n_l + 2 * pad_l,), -3.0, dtype=torch.float32, device="cuda")
    o = big_o[pad_o:pad_o + n_o].view(q.shape)
    lse = big_l[pad_l:pad_l + n_l].view(B, H, N)
    kwargs = {}
    if mode.startswith("window"):
        kwargs["window"] = (100, 0)
    elif mode.startswith("split"):
        kwargs["n_splits"] = 3
    else:
        kwargs["n_splits"] = 1
    fa.fwd(tq, tk, tv, causal=causal, scale=w.scale, out=o, lse=lse, **kwargs)
    torch.cuda.synchronize()
    assert torch.all(big_o[:pad_o] == 7.0) and torch.all(big_o[pad_o + n_o:] == 7.0)
    assert torch.all(big_l[:pad_l] == -3.0) and torch.all(big_l[pad_l + n_l:] == -3.0)
    # every row inside was written (and is right) -- spot-check against the oracle
    rows = np.array([0, 127, 128, N - 1, N, 2 * N - 1, n_l - 1])
    o_ref, lse_ref = oracle.attention_rows(q, k, v, rows, w.scale, causal, window=kwargs.get("window"))
    o_s = o.float().cpu().numpy().astype(np.float64).reshape(-1, d)[rows]
    l_s = lse.cpu().numpy().astype(np.float64).reshape(-1)[rows]
    assert_close(o_s, l_s, o_ref, lse_ref, mode)


# --- device-side argument errors -------------------------------------------------
def test_host_pointer_rejected():
    import torch

    import exact_attention_19_gb300 as fa

    qh = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16)  # host memory
    qd = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(qd)
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd(qh.data_ptr(), qd.data_ptr(), qd.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 128, 128,
                   64, 0.125, 0, None)
    assert st == 10  # FA_ERR_POINTER


# --- full benchmark sizes, sampled rows --------------------------------------------
@pytest.mark.parametrize("name", ["long_8192_d128", "long_8192_d128_causal", "stress_32000_d128_causal"])
def test_full_size_sampled_rows(name):
    w = synth.WORKLOADS[name]
    q, k, v = w.make()
    o, lse = run_gpu(q, k, v, w.scale, w.causal)
    rows = sample_rows(w.B, w.H, w.Nq, 400, seed=w.seed)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, rows, w.scale, w.causal)
    o_s = o.reshape(-1, w.d)[rows]
    l_s = lse.reshape(-1)[rows]
    assert_close(o_s, l_s, o_ref, lse_ref, name)
    # properties over every row at full size
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    if w.causal:
        # row 0 of every head sees key 0 only: O = V[0] exactly, LSE = scale * q0.k0
        vv = synth.bf16_to_f32(v[:, :, 0, :]).astype(np.float64)
        assert np.array_equal(o[:, :, 0, :], vv)


# --- sliding windows (bottom-right aligned) and causal with Nq != Nk ----------
def _run_window(q, k, v, scale, window):
    import torch

    import exact_attention_19_gb300 as fa

    o, lse = fa.fwd(to_device(q), to_device(k), to_device(v), scale=scale, window=window)
    torch.cuda.synchronize()
    st, word = fa.fa_fwd_status(None, clear=True)
    assert st == 0, f"kernel wait timed out, status word {word:#x}"
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _assert_close_window(o, lse, o_ref, lse_ref, what):
    # rows that see no key: LSE = -inf and O = 0 on both sides, exactly
    empty = ~np.isfinite(lse_ref)
    assert np.array_equal(~np.isfinite(lse), empty), f"{what}: empty-row pattern differs"
    assert np.all(o[empty] == 0.0), f"{what}: O of an empty row is not 0"
    full = ~empty
    assert_close(o[full], lse[full], o_ref[full], lse_ref[full], what)


WINDOWS = [(-1, 0), (0, 0), (64, 0), (200, 50), (127, 128), (-1, 300), (5, -1), (1000, 1000)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("nq,nk", [(700, 700), (300, 1000), (1000, 300), (257, 129)])
def test_window_parity(nq, nk, window, d):
    w = synth.Workload("win", 2, 2, nq, nk, d, False, seed=61 + nq + nk)
    q, k, v = w.make()
    o, lse = _run_window(q, k, v, w.scale, window)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, w.scale, window=window)
    _assert_close_window(o, lse, o_ref, lse_ref, f"window {window} {nq}x{nk} d{d}")


# a window bounded on both sides with Nq <= Nk and at least 4 query-tile pairs
# per SM: the persistent kernel (tile 1's range may start one K/V tile after
# tile 0's; both are masked at both ends)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("window", [(200, 50), (0, 0), (127, 128), (1000, 1000), (5, 300)])
@pytest.mark.parametrize("shape", [(4, 64, 700, 700), (4, 80, 300, 1000)])
def test_window_persistent(shape, window, d):
    B, H, nq, nk = shape
    w = synth.Workload("winp", B, H, nq, nk, d, False, seed=71 + nq + nk + d)
    q, k, v = w.make()
    o, lse = _run_window(q, k, v, w.scale, window)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, w.scale, window=window)
    _assert_close_window(o, lse, o_ref, lse_ref, f"window {window} {B}x{H}x{nq}x{nk} d{d}")


def test_window_equal_to_causal_when_square():
    w = synth.Workload("wc", 1, 3, 1000, 1000, 128, True, seed=62)
    q, k, v = w.make()
    o_w, l_w = _run_window(q, k, v, w.scale, (-1, 0))
    o_c, l_c = run_gpu(q, k, v, w.scale, True, 1)
    assert np.array_equal(o_w, o_c) and np.array_equal(l_w, l_c)


def test_window_full_size_sampled_rows():
    # long-context shape with a 1024-key causal window: most K/V tiles skipped
    w = synth.WORKLOADS["long_8192_d128"]
    q, k, v = w.make()
    o, lse = _run_window(q, k, v, w.scale, (1024, 0))
    rows = sample_rows(w.B, w.H, w.Nq, 300, seed=63)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, rows, w.scale, window=(1024, 0))
    assert_close(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, "window 1024 at N=8192")


def test_window_rejects_bad_bounds():
    import torch

    import exact_attention_19_gb300 as fa

    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd_window(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 128, 128, 64,
                          0.125, -2, 0, None)
    assert st == 3
