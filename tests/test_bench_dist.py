"""The benchmark's multi-process logic on CPU: two gloo ranks (the path a
torchrun launch with N > 1 takes), without a GPU."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        step_ms = 1.0 + rank                      # rank 1 is the slower one
        worst = bench.max_over_ranks(step_ms, dist, "cpu")
        e2e = bench.max_over_ranks(float("nan") if rank == 1 else 3.0, dist, "cpu")
        value = bench.job_tflops(2e12, world, worst)
        with open(f"{out_path}.{rank}", "w") as f:
            json.dump({"worst": worst, "value": value, "e2e_nan": e2e != e2e}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_with_two_gloo_ranks(tmp_path):
    port = _free_port()
    out = str(tmp_path / "r")
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    res = [json.load(open(f"{out}.{r}")) for r in range(2)]
    for r in res:
        assert r["worst"] == 2.0                  # every rank sees the slowest rank's time
        assert r["value"] == pytest.approx(2e12 * 2 / 2e-3 / 1e12)   # both ranks' FLOPs over it
        assert r["e2e_nan"]                       # a failed measurement on one rank is not hidden


def _dead_rank_main(rank, world, port, out_path, mode="exit"):
    """Rank 1 leaves between steps (no kernel or collective in flight): it
    exits ("exit"), or stays alive without joining the next collective
    ("stall").  Rank 0 must learn of it in its next collective, with an
    error, not a hang: at once when the peer's connection closes, after the
    process group's timeout when the peer is silent."""
    import time
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["RANK"], os.environ["WORLD_SIZE"] = str(rank), str(world)
    sys.path.insert(0, ROOT)
    import bench
    d = bench.init_distributed("gloo", timeout_s=5)
    d.barrier()                                   # one healthy step together
    if rank == 1:
        if mode == "stall":
            time.sleep(9)                         # alive, but never reaches the collective
        os._exit(0)                               # the rank is gone; nothing of it is in flight
    t0 = time.monotonic()
    try:
        bench.max_over_ranks(1.0, d, "cpu")
        outcome = "returned"
    except Exception as ex:                       # the survivor's next collective fails
        outcome = type(ex).__name__
    with open(f"{out_path}.0", "w") as f:
        json.dump({"outcome": outcome, "seconds": time.monotonic() - t0}, f)
    os._exit(0)                                   # no clean shutdown with a dead peer


@pytest.mark.parametrize("mode,limit_s", [("exit", 4.0), ("stall", 8.5)])
def test_a_dead_rank_ends_the_survivors_next_collective_with_an_error(tmp_path, mode, limit_s):
    port = _free_port()
    out = str(tmp_path / "d")
    mp.spawn(_dead_rank_main, args=(2, port, out, mode), nprocs=2, join=True)
    res = json.load(open(f"{out}.0"))
    assert res["outcome"] != "returned"
    assert res["seconds"] < limit_s                # the 5 s timeout, not the backend's default


def test_process_group_timeout_is_bounded():
    sys.path.insert(0, ROOT)
    import bench
    assert 60 <= bench.PG_TIMEOUT_S <= 600


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, None, "cpu") == 1.5
    assert bench.job_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", "tiny", "--steps", "2", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
