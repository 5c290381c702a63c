"""bench.py's multi-rank host plumbing, run as world-size-2 process groups over
gloo on the CPU: rank/world discovery from the launcher's environment, the
barrier, the max-over-ranks step time and the whole-job throughput built from
it, and the reference arm that only rank 0 runs and prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_env(rank: int, world: int, port: int) -> dict:
    return {"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank), "WORLD_SIZE": str(world),
            "LOCAL_RANK": str(rank)}


def _worker(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(_rank_env(rank, world, port))
    sys.path.insert(0, ROOT)
    import bench
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    bench.barrier()
    step_ms = [2.0, 5.0][rank]                      # rank 1 is the slow one
    slowest = bench.max_over_ranks(step_ms)
    res = {"rank": r, "world": w, "slowest": slowest, "value": bench.job_throughput(2048, w, slowest)}
    bench.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)
    torch.distributed.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo(tmp_path):
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        res = json.loads((tmp_path / f"rank{rank}.json").read_text())
        assert res["rank"] == rank and res["world"] == 2
        assert res["slowest"] == 5.0                              # every rank sees the max
        assert res["value"] == pytest.approx(2 * 2048 / 5e-3)     # both ranks' tokens over the slowest step


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.dist_env() == (0, 1, 0)
        assert bench.max_over_ranks(3.5) == 3.5                   # no process group: identity
        assert bench.job_throughput(2048, 1, 2.0) == pytest.approx(2048 / 2e-3)
    finally:
        os.environ.update(env)


def test_reference_arm_runs_on_rank0_only():
    """Launched like torchrun with two ranks: rank 0 times the oracle and prints one JSON line,
    rank 1 exits 0 without output."""
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, **_rank_env(rank, 2, port))
        procs.append(subprocess.Popen(
            [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1",
             "--warmup", "3"], cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE))
    outs = [p.communicate(timeout=600) for p in procs]
    for p, (_, err) in zip(procs, outs):
        assert p.returncode == 0, err.decode()[-2000:]
    lines = [ln for ln in outs[0][0].decode().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
    assert res["cpu_baseline"]["kind"] == "oracle"
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["e2e"]["d2h_bytes_per_step"] == 0
    assert outs[1][0].decode().strip() == ""
