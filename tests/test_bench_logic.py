"""bench.py host logic on the CPU: whole-job aggregation over ranks (gloo,
world size 2), clock summaries, argument rules, the reference arm's rank
handling, the roofline denominators and the traffic table lookup."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_aggregate_single_rank():
    """value from the median step; value_from_total from the K steps' total."""
    r = bench.aggregate(1.9, 10.0, 1, 2e12, 5, lambda x: x)
    assert r["ms_per_step"] == pytest.approx(1.9)
    assert r["value"] == pytest.approx(2e12 / 1.9e-3 / 1e12)
    assert r["value_from_total"] == pytest.approx(5 * 2e12 / 1e-2 / 1e12)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    r = bench.aggregate(local_ms[rank] / 4 - rank * 0.1, local_ms[rank], d.world, 1e12, 4, d.max)
    q.put((rank, r))
    d.close()


def test_aggregate_two_ranks_gloo():
    """Whole-job value = all ranks' flops over the slowest rank's time."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    local = [8.0, 12.0]
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, local, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(2))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        # medians 2.0 (rank 0) and 2.9 (rank 1): the slowest rank's median counts
        assert out[r]["ms_total"] == pytest.approx(12.0)
        assert out[r]["ms_per_step"] == pytest.approx(2.9)
        assert out[r]["value"] == pytest.approx(2 * 1e12 / 2.9e-3 / 1e12)
        assert out[r]["value_from_total"] == pytest.approx(2 * 1e12 * 4 / 12e-3 / 1e12)


def test_clock_summary_inside_windows():
    rows = [{"t": 10.0, "sm": 1800.0, "max": 2070.0, "reasons": {"sw_power_cap": "Not Active"}},
            {"t": 10.5, "sm": 2000.0, "max": 2070.0, "reasons": {"sw_power_cap": "Active"}},
            {"t": 20.0, "sm": 900.0, "max": 2070.0, "reasons": {"hw_slowdown": "Active"}}]
    c = bench.summarize_clocks(rows, [(9.9, 10.6)])
    assert c["samples"] == 2 and c["sm_mhz"] == 1900.0
    assert c["reasons"] == ["sw_power_cap"]
    c2 = bench.summarize_clocks(rows, [(30.0, 30.1)])
    assert c2["samples"] == 3
    assert bench.summarize_clocks([], [(0, 1)])["sm_mhz"] is None


def test_rejected_clock_records():
    """hw_slowdown / thermal reasons void a window (it is measured again);
    sw_power_cap does not; clocks far below max with no reason do."""
    assert bench.rejected({"reasons": ["sw_power_cap"], "sm_mhz": 1900.0, "sm_max_mhz": 2070.0}) is None
    assert bench.rejected({"reasons": [], "sm_mhz": 2070.0, "sm_max_mhz": 2070.0}) is None
    assert "hw_slowdown" in bench.rejected({"reasons": ["hw_slowdown"], "sm_mhz": 900.0,
                                            "sm_max_mhz": 2070.0})
    assert "sw_thermal_slowdown" in bench.rejected({"reasons": ["sw_power_cap", "sw_thermal_slowdown"],
                                                    "sm_mhz": 1500.0, "sm_max_mhz": 2070.0})
    assert "no reason" in bench.rejected({"reasons": [], "sm_mhz": 1200.0, "sm_max_mhz": 2070.0})
    assert bench.rejected({"reasons": [], "sm_mhz": None, "sm_max_mhz": None}) is None


def test_args_rules():
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1 and a.impl == "ours"
    q = bench.parse_args(["--quick"])  # every workload once, still >= 3 warm-up steps
    assert q.steps == 1 and q.warmup == 3 and q.no_cpu and q.no_e2e and not q.no_modes


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_mode_peaks():
    """Measured cuBLAS rates of this run take precedence for TF32 (and 3xTF32)
    and FP8; without them the BF16 burst times the nominal ratio."""
    peaks = {"bf16_tflops": 2000.0, "sm_max_mhz": 2000.0}
    assert bench.mode_peak("bf16", peaks, 100)[1] == 2000.0
    assert bench.mode_peak("tf32", peaks, 100)[1] == pytest.approx(2000.0 * 1.1 / 2.25)
    b, p, how = bench.mode_peak("tf32", peaks, 100, {"tf32": 1040.0, "fp8": 3500.0})
    assert p == 1040.0 and how.startswith("measured in this run")
    assert bench.mode_peak("3xtf32", peaks, 100, {"tf32": 1040.0})[1] == 1040.0
    assert bench.mode_peak("e5m2", peaks, 100, {"fp8": 3500.0})[1] == 3500.0
    assert bench.mode_peak("e4m3", peaks, 100, {"tf32": 1040.0})[2].startswith("fallback")
    assert bench.nominal_peak("e4m3", peaks) == pytest.approx(4000.0)
    b, p, _ = bench.mode_peak("simt", peaks, 100)
    assert b == "alu" and p == pytest.approx(100 * 128 * 2 * 2000e6 / 1e12)


def test_traffic_table_respects_source_hash():
    """A recorded DRAM-traffic figure applies only to the sources it was
    captured on; otherwise the line carries null and says why."""
    sha = bench.source_sha("tf32")
    table = {("tf32", "w1"): {"bytes": 1234, "sha": sha, "command": "ncu ..."},
             ("simt", "w1"): {"bytes": 99, "sha": "000000000000", "command": "ncu ..."}}
    v, src = bench.recorded_traffic("tf32", "w1", table)
    assert v == 1234.0 and src["command"] == "ncu ..."
    v, why = bench.recorded_traffic("simt", "w1", table)
    assert v is None and "stale" in why
    v, why = bench.recorded_traffic("tf32", "other", table)
    assert v is None and "no ncu capture" in why
    assert bench.source_sha("simt") != sha


def test_reference_line_shape(capsys):
    """The reference arm prints one JSON line with the contract's keys (run on
    a tiny sample: 1 step)."""
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "cpu_baseline", "e2e", "config"):
        assert k in line
    assert line["impl"] == "reference" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_cpu_oracle_small_workloads_times_both_thread_counts():
    """The small-workload oracle timings of cpu_baseline: one entry per small
    workload, one and all host threads, and the thread count restored."""
    import oracle

    n = oracle.max_threads()
    out = bench.cpu_oracle_small()
    assert set(out) == {"square-64 fp32", "square-1024 fp32", "ragged 1000x1013x997 fp32"}
    for row in out.values():
        assert len(row) == (2 if n > 1 else 1) and all(v >= 0 for v in row.values())
    assert oracle.max_threads() == n
