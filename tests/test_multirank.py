"""The benchmark's multi-rank host logic across two gloo ranks on the CPU.

Each GPU runs a whole replica of the decode step (the path has no exchange
step); the ranks meet only on the host: a barrier on both sides of the timed
region, the slowest rank's time, and the whole-job throughput over all ranks.
These tests run that logic as two processes over gloo on 127.0.0.1, and the
launcher that bench.py --gpus N uses when it is started as a plain script.
"""
import contextlib
import io
import json
import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

WORLD = 2


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import time
    import torch.distributed as dist
    env = {"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
           "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)}
    os.environ.update(env)
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.init_ranks(w, "gloo")
    try:
        # barrier: no rank leaves before the slowest arrives
        if rank == 1:
            time.sleep(0.3)
        t0 = time.monotonic()
        bench.barrier(w)
        waited = time.monotonic() - t0
        # each rank's own time differs; every rank gets the largest
        ms_own = [3.5, 7.25][rank]
        ms = bench.max_over_ranks(ms_own, w)
        value = bench.whole_job_gbs(w, 1_000_000, 10, ms)
        # the reference arm runs on rank 0 alone: other ranks print nothing
        buf = io.StringIO()
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                bench.reference_arm(types.SimpleNamespace(steps=1, warmup=0, gpus=w), r, w)
        bench.barrier(w)
        with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
            json.dump([ms, value, waited, buf.getvalue()], f)
    finally:
        bench.finish_ranks(w)
        assert not dist.is_initialized()


def test_dist_env_parsing():
    assert bench.dist_env({}) == (0, 1, 0)
    assert bench.dist_env({"RANK": "3", "WORLD_SIZE": "4"}) == (3, 4, 3)
    assert bench.dist_env({"RANK": "5", "WORLD_SIZE": "8", "LOCAL_RANK": "1"}) == (5, 8, 1)
    for bad in ({"RANK": "2", "WORLD_SIZE": "2"}, {"WORLD_SIZE": "0"},
                {"RANK": "-1", "WORLD_SIZE": "2"}):
        with pytest.raises(ValueError):
            bench.dist_env(bad)


def test_single_rank_needs_no_process_group():
    import torch.distributed as dist
    bench.init_ranks(1, "gloo")
    assert not dist.is_initialized()
    bench.barrier(1)
    assert bench.max_over_ranks(2.5, 1) == 2.5
    bench.finish_ranks(1)


def test_whole_job_value_scales_with_ranks():
    one = bench.whole_job_gbs(1, 58_000_000, 100, 1.7)
    assert one == pytest.approx(58_000_000 * 100 / 1.7e-3 / 1e9)
    # weak scaling: N replicas doing the same work in the same time deliver N times the bytes
    assert bench.whole_job_gbs(4, 58_000_000, 100, 1.7) == pytest.approx(4 * one)
    with pytest.raises(ValueError):
        bench.whole_job_gbs(1, 1, 1, 0.0)


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(WORLD, port, str(tmp_path)), nprocs=WORLD,
                       join=True, start_method="spawn")
    rows = []
    for r in range(WORLD):
        with open(tmp_path / ("rank%d.txt" % r)) as f:
            ms, value, waited, printed = json.load(f)
        rows.append((ms, value, waited, printed))
    for ms, value, _, printed in rows:
        assert ms == 7.25                      # the slowest rank's time, on every rank
        assert value == pytest.approx(WORLD * 1_000_000 * 10 / 7.25e-3 / 1e9)
        assert printed == ""
    assert rows[0][2] > 0.2                    # rank 0 waited at the barrier for rank 1


def test_launcher_command_and_world_check():
    cmd = bench.local_ranks_command(["--gpus", "4", "--steps", "3"], 4, 29123)
    assert cmd[:3] == [sys.executable, "-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--master-addr=127.0.0.1" in cmd
    assert "--master-port=29123" in cmd
    assert cmd[-4:] == ["--gpus", "4", "--steps", "3"]
    assert os.path.samefile(cmd[-5], os.path.join(ROOT, "bench.py"))
    bench.check_world(2, 2)
    with pytest.raises(SystemExit):
        bench.check_world(2, 1)


def test_gpus_2_without_a_launcher_starts_two_ranks():
    """bench.py --gpus 2 run as a plain script starts two local ranks of
    itself under torch.distributed.run; with --impl reference rank 0 alone
    prints its line, which carries n_gpus 2, and both ranks exit 0."""
    import subprocess
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-seconds", "0.2"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
