"""The N > 1 path of bench.py on the CPU, with world_size-2 gloo process groups.

Requests are independent, so ranks run independent replicas with no collective on the data
path. Only the timing is combined: the whole-job rate is the units all ranks processed over
the slowest rank's time. Under torchrun, the reference arm runs on rank 0 alone and prints
one line; the other ranks exit cleanly.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [10.0, 20.0][rank]                         # rank 1 is the slower one
    rate, ms = bench.whole_job_rate(dist, local_ms, units_per_rank_step=9, steps=3, ws=world)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"rate": rate, "ms": ms}, f)
    dist.destroy_process_group()


def test_whole_job_rate_takes_the_slowest_rank(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        got = json.load(open(tmp_path / f"r{r}.json"))
        assert got["ms"] == 20.0
        assert got["rate"] == pytest.approx(9 * 3 * 2 / 0.020)


def test_whole_job_rate_single_process():
    sys.path.insert(0, ROOT)
    import bench
    rate, ms = bench.whole_job_rate(None, 30.0, units_per_rank_step=576, steps=10, ws=1)
    assert ms == 30.0 and rate == pytest.approx(576 * 10 / 0.030)


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
    assert j["config"]["workload"] == "b64k8v262144"
