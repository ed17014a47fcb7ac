"""bench.py's multi-rank host logic on CPU (gloo, world size 2): the timed
region's time is the slowest rank's, the job rate counts every rank's bytes,
and under torchrun only rank 0 prints the result line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [12.5, 30.25][rank]                   # rank 1 is the slow one
    mx = bench.dist_max(local_ms, world)
    rate = bench.weak_scaling_rate(world, 1e9, 10, mx)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, mx, rate))


def test_dist_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, rate in res:
        assert mx == 30.25
        assert rate == pytest.approx(2 * 1e9 * 10 / 30.25e-3 / 1e9)


def test_weak_scaling_rate_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(7.0, 1) == 7.0
    assert bench.weak_scaling_rate(1, 920053152, 4000, 555.0) == pytest.approx(920053152 * 4000 / 0.555 / 1e9)


def test_torchrun_reference_arm_two_ranks_prints_once():
    """--impl reference under torchrun: rank 0 times the oracle and prints one
    line (n_gpus = 2, impl = reference); rank 1 exits 0 without output."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "GB/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_rows_option_names_every_group():
    """`--rows` selects side-row groups by name: the names its help text
    lists are exactly the groups bench_rows guards, so no group can be
    skipped by a misspelt name in either place."""
    import inspect
    import re
    sys.path.insert(0, ROOT)
    import bench
    guarded = set(re.findall(r'if want\("(\w+)"\)', inspect.getsource(bench.bench_rows)))
    src = inspect.getsource(bench.parse_args)
    help_text = "".join(re.findall(r'"([^"]*)"', src[src.index('"--rows"'):src.index("return p.parse_args")]))
    listed = set(re.findall(r"\b([a-z0-9]+) \(", help_text)) | set(re.findall(r"\b(syncbn|sampler|sweep)\b", help_text))
    assert guarded == {"linear", "gpt2", "accum", "orders", "syncbn", "sampler", "sweep"}, guarded
    assert guarded <= listed, (guarded, listed)
    old = sys.argv
    try:
        sys.argv = ["bench.py", "--rows", "syncbn,sampler"]
        assert bench.parse_args().rows == "syncbn,sampler"
        sys.argv = ["bench.py"]
        assert bench.parse_args().rows is None
    finally:
        sys.argv = old
