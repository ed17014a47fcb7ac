"""bench.py's output on CPU: the result line is the last line of stdout,
is short, and carries every key the measurement contract names; side rows
go out first, one JSON line each."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402


def _line():
    num, plan = bench.resnet50_plan(oracle.plan_buckets)
    cpu = {"value": 12.0, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": "first 6,515,688 elements of each of the 5 buckets x 8 replicas (32,578,440 elements per "
                     "pass), 17 passes in 10.2 s, numpy single-threaded on 16 host cores",
           "c_oracle": {"single_thread_GBps": 12.1, "threads_GBps": 171.0, "threads": 16}}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3,
              "window": "nearest samples to a short timed region", "power_w_max": 700.0}
    return bench.headline(value=7000.0, world=1, K=20, W=5, elapsed_ms=2.6, plan=plan, num=num, peak=6669.2,
                          peak_kind="measured", achieved=6650.0, avg_launch_ms=0.0277, traffic=1.74e8,
                          traffic_note=None, cpu=cpu, e2e_copy=230.0, e2e_zero=235.0, h2d_gbs=210.0,
                          host_check=True, e2e_steps=5, clocks=clocks, step_streams=5)


def test_headline_is_short_and_complete():
    line = _line()
    s = json.dumps(line, separators=(",", ":"))
    assert len(s) <= bench.HEADLINE_MAX_BYTES, len(s)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in line, key
    assert line["metric"] == bench.METRIC
    assert "workload" in line["config"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in line["roofline"], key
    assert abs(line["roofline"]["frac"] - 6650.0 / 6669.2) < 1e-12
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in line["cpu_baseline"], key
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in line["e2e"], key
    assert line["e2e"]["h2d_bytes_per_step"] >= 8 * 25_557_032 * 4   # every replica's gradients, every step
    assert line["gpu_launches"] == 20 * 5


def test_rows_first_headline_last(capsys, tmp_path):
    out = tmp_path / "rows.jsonl"
    bench.emit_row("sgd_gpt2_small", {"ms": 0.55, "GBps": 7250.0}, str(out))
    for i in range(200):                           # a long sweep must not push the result line out of the tail
        bench.emit_row("sweep_flat_fp32", {"bytes_per_replica": 1 << 30, "replicas": 16, "i": i}, str(out))
    bench.emit_headline(_line())
    lines = capsys.readouterr().out.strip().split("\n")
    assert len(lines) == 202
    last = json.loads(lines[-1])
    assert last["metric"] == bench.METRIC and last["value"] == 7000.0
    assert all("row" in json.loads(x) for x in lines[:-1])
    assert len(lines[-1]) <= bench.HEADLINE_MAX_BYTES
    assert len(out.read_text().strip().split("\n")) == 201


def test_overlong_headline_is_refused():
    line = _line()
    line["config"]["padding"] = "x" * bench.HEADLINE_MAX_BYTES
    try:
        bench.emit_headline(line)
    except RuntimeError:
        return
    raise AssertionError("an over-long result line was printed")
