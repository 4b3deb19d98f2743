"""The benchmark's multi-rank path on CPU: two gloo ranks (127.0.0.1), weak
scaling over replicas: whole-job throughput = units of all ranks / the max
step time over ranks; no collective on the data path."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    d = bench.init_dist(ws, "gloo")
    try:
        units = [3.0e9, 5.0e9][rank]
        ms = [10.0, 40.0][rank]
        bench.barrier(d)
        value, ms_job = bench.whole_job(d, units, ms, torch.device("cpu"))
        q.put((rank, ws, r, value, ms_job))
    finally:
        d.destroy_process_group()


def test_two_rank_weak_scaling_uses_max_time_and_total_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ws, r, value, ms_job in got:
        assert ws == 2 and r == rank
        assert ms_job == pytest.approx(40.0)
        assert value == pytest.approx((3.0e9 + 5.0e9) / 0.040)


def test_single_rank_needs_no_process_group():
    import bench
    value, ms = bench.whole_job(None, 8.0e9, 20.0, torch.device("cpu"))
    assert ms == 20.0 and value == pytest.approx(4.0e11)


def test_gpus_flag_launches_that_many_ranks():
    """bench.py --gpus 2 (outside torchrun) re-runs itself as two ranks under torch.distributed.run;
    the reference arm (CPU only: the oracle on host threads) prints one line, from rank 0, with n_gpus 2."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--rows", "2", "--ref-sample", "8192", "--steps", "1", "--warmup", "0", "--chunk", "4096"],
                       capture_output=True, text=True, timeout=300, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2
