"""bench.py host logic without a GPU: throughput aggregation, max over ranks
(two gloo ranks on CPU), traffic lookup and the oracle (reference) arm."""
import contextlib
import io
import json
import os
import socket

import numpy as np
import pytest

import bench
import synth


def test_aggregate_uses_slowest_rank():
    v, t = bench.aggregate([2.0, 4.0], [1e12, 1e12])
    assert t == 4.0 and v == pytest.approx(2e12 / 4e-3 / 1e12)


def test_visible_keys_and_sampling():
    w = synth.Workload("t", 1, 2, 10, 10, 64, True)
    rows = np.arange(20)
    assert bench.visible_keys(w, rows).tolist() == list(range(1, 11)) * 2
    # over all rows the counted FLOPs equal the full-causal count up to the diagonal half
    assert np.sum(4.0 * bench.visible_keys(w, rows) * 64) == pytest.approx(4 * 2 * 64 * (10 * 11 / 2))
    r = bench.sample_rows_even(w, 7)
    assert r[0] == 0 and r[-1] == 19 and len(set(r)) == len(r)


def test_window_flops_closed_forms():
    """Kept (row, key) pairs under a window, against closed forms: the causal
    triangle, the diagonal alone, a band, an open window, and Nq > Nk rows that
    keep nothing."""
    base = synth.Workload("w", 2, 3, 100, 100, 64, False)
    per_pair = 4.0 * 2 * 3 * 64
    assert bench.flops_of(base.with_(window=(-1, 0))) == per_pair * 100 * 101 / 2
    assert bench.flops_of(base.with_(window=(0, 0))) == per_pair * 100
    # band of 10 keys back: row i keeps min(i, 10) + 1 keys
    assert bench.flops_of(base.with_(window=(10, 0))) == per_pair * (sum(range(1, 11)) + 90 * 11)
    assert bench.flops_of(base.with_(window=(-1, -1))) == base.flops
    assert bench.flops_of(base.with_(window=(500, 500))) == base.flops
    # Nq = 100 > Nk = 30, diagonal window: only the last 30 rows keep a key (one each)
    tall = synth.Workload("t", 1, 1, 100, 30, 64, False, window=(0, 0))
    assert bench.flops_of(tall) == 4.0 * 64 * 30
    assert bench.pairs_of(tall) == 30
    keys = bench.visible_keys(tall, np.arange(100))
    assert np.all(keys[:70] == 0) and np.all(keys[70:] == 1)
    # no window: the metric's convention, halved under the causal mask
    assert bench.flops_of(base) == base.flops
    assert bench.flops_of(base.with_(causal=True)) == base.flops / 2


def test_kernel_name_follows_dispatch():
    w = synth.WORKLOADS["long_8192_d128"]
    assert bench.kernel_name(w, None) == "fa_fwd_persist_kernel"
    assert bench.kernel_name(w, 1) == "fa_fwd_persist_kernel"
    assert bench.kernel_name(w, 4) == "fa_fwd_kernel"
    assert bench.kernel_name(synth.WORKLOADS["long_8192_d128_causal"], None) == "fa_fwd_persist_kernel"
    assert bench.kernel_name(synth.WORKLOADS["stress_32000_d128_causal"], None) == "fa_fwd_kernel"
    assert bench.kernel_name(synth.WORKLOADS["single_head_4096_d64"], 1) == "fa_fwd_kernel"
    assert bench.kernel_name(synth.WORKLOADS["single_head_256_d64"], 1) == "fa_fwd_persist_kernel"
    assert bench.kernel_name(synth.WORKLOADS["gpt2_small_causal_1024_d64"], None) == "fa_fwd_kernel"
    assert bench.kernel_name(synth.WORKLOADS["long_8192_d64"].with_(causal=True), None) == "fa_fwd_persist_kernel"
    few = synth.WORKLOADS["long_8192_d64"].with_(causal=True, B=1, H=8)  # 256 pairs: under 6 per SM
    assert bench.kernel_name(few, None) == "fa_fwd_kernel"
    assert bench.kernel_name(w.with_(window=(64, 0)), None) == "fa_fwd_persist_kernel"
    assert bench.kernel_name(w.with_(window=(64, -1)), None) == "fa_fwd_kernel"
    assert bench.kernel_name(w.with_(window=(64, 0), B=1, H=8), None) == "fa_fwd_kernel"


def test_causal_flag_rejects_window():
    with pytest.raises(SystemExit):
        bench.main(["--causal", "--window", "64,0"])


def test_traffic_lookup(tmp_path, monkeypatch):
    h = bench.kernel_source_hash()
    f = tmp_path / "traffic.md"
    f.write_text(f"| long_8192_d128 | {h} | 123456 | 1 | 2 | 3 | cmd |\n| other | {h} | 7 | | | | |\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.read_traffic("long_8192_d128", h) == 123456.0
    assert bench.read_traffic("long_8192_d128", "0" * 16) is None
    assert bench.read_traffic("missing", h) is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [10.0, 30.0][rank]
        e2e = [7.0, 5.0][rank]
        tmax, emax = bench.max_over_ranks([elapsed, e2e], dist, "cpu")
        value, t = bench.aggregate([tmax] * world, [1e12 * 3] * world)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"tmax": tmax, "emax": emax, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r in res:
        assert r["tmax"] == 30.0 and r["emax"] == 7.0
        assert r["value"] == pytest.approx(2 * 3e12 / 30e-3 / 1e12)


def test_reference_arm_line(monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--workload",
                         "single_head_256_d64"])
    assert rc == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "single_head_256_d64"


def test_reference_arm_window_line(monkeypatch):
    """--window reaches the oracle leg: the line names the window and counts the
    kept pairs (a 16-key band over 256 rows: 16*17/2 + 240*17 pairs)."""
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--workload",
                         "single_head_256_d64", "--window", "16,0"])
    assert rc == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["config"]["window"] == [16, 0] and line["config"]["causal"] is False
    assert line["config"]["flops_per_step"] == 4.0 * 64 * (16 * 17 / 2 + 240 * 17)
    assert line["value"] > 0


def test_reference_arm_rejects_backward():
    with pytest.raises(SystemExit) as e:
        bench.main(["--impl", "reference", "--pass", "bwd"])
    assert e.value.code == 2


def test_reference_arm_other_ranks_silent(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert rc == 0 and buf.getvalue() == ""


def test_roofline_bound_follows_intensity():
    import synth

    peak, hbm = 1891.4, 6789.0
    # the long workload sits far above the ridge (about 279 FLOP per byte): tensor-bound
    w = synth.WORKLOADS["long_8192_d128"]
    r = bench.roofline_entry(w.flops, w.algorithmic_bytes, 1500.0, 400.0, peak, hbm)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and abs(r["frac"] - 1500.0 / peak) < 1e-12
    # the single-head N = 256 case (127 FLOP per byte) and the GPT-2 shape (254) are below it
    for name in ("single_head_256_d64", "gpt2_small_causal_1024_d64"):
        w = synth.WORKLOADS[name]
        r = bench.roofline_entry(w.flops, w.algorithmic_bytes, 1.0, 50.0, peak, hbm)
        assert r["bound"] == "hbm" and r["unit"] == "GB/s" and abs(r["frac"] - 50.0 / hbm) < 1e-12
        assert r["intensity_flop_per_byte"] < r["ridge_flop_per_byte"]


def test_e2e_entry_reports_the_faster_mode_and_both_figures():
    e = bench.e2e_entry(1000.0, 4.0, 500.0, 8.0, 100, 10, 5)
    assert e["mode"] == "pipelined" and e["value"] == 1000.0 and e["ms_per_step"] == 4.0
    assert e["serial_value"] == 500.0 and e["h2d_bytes_per_step"] == 100 and e["d2h_bytes_per_step"] == 10
    e = bench.e2e_entry(50.0, 0.08, 88.0, 0.05, 100, 10, 5)
    assert e["mode"] == "serial" and e["value"] == 88.0 and e["pipelined_value"] == 50.0


def test_bwd_algorithmic_bytes_counts_every_tensor_once():
    # 4 x 32 x 8192 x 128: eight bf16 tensors of 268,435,456 bytes (Q, K, V, O, dO read; dQ, dK, dV
    # written), LSE read (4 B per row), L and D written then read (16 B per row)
    w = synth.WORKLOADS["long_8192_d128"]
    rows = 4 * 32 * 8192
    assert bench.bwd_algorithmic_bytes(w) == 8 * 268435456 + 4 * rows + 16 * rows


def test_step_stats_percentiles():
    st = bench.step_stats([5.0, 1.0, 3.0, 2.0, 4.0])
    assert st == {"median": 3.0, "p10": 1.0, "p90": 5.0}
    assert bench.step_stats([]) is None


def test_timed_steps_without_flush_on_cpu_events():
    # the function's contract on a fake torch: one event per step boundary, totals add up
    class Ev:
        t = 0.0

        def __init__(self, enable_timing=True):
            self.stamp = None

        def record(self, stream=None):
            Ev.t += 1.0
            self.stamp = Ev.t

        def elapsed_time(self, other):
            return other.stamp - self.stamp

    class FakeCuda:
        Event = Ev

        @staticmethod
        def synchronize():
            pass

    class FakeTorch:
        cuda = FakeCuda

    total, per = bench.timed_steps(FakeTorch, lambda: None, 4, None, None)
    assert per == [1.0, 1.0, 1.0, 1.0] and total == 4.0
