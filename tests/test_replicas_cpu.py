"""Multi-process (world size 2, gloo on CPU) checks of the replica path of bench.py:
every rank runs an independent replica with no data-path collective; the job's time is
the slowest rank's and its throughput counts the tokens of every rank; the reference
arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_WORKER = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import torch
import torch.distributed as dist
import bench
rank = int(os.environ["RANK"]); world = int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo")
ms = [3.0, 7.5][rank]
job_ms = bench.max_over_ranks(ms, world, "cpu")
tps = bench.job_tokens_per_s(64, world, job_ms)
dist.barrier()
print(json.dumps({"rank": rank, "job_ms": job_ms, "tps": tps}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time_and_sum_tokens(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(_WORKER)
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script), ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=120)
        assert p.returncode == 0, e
        outs.append(json.loads(o.strip().splitlines()[-1]))
    for o in outs:
        assert o["job_ms"] == 7.5
        assert abs(o["tps"] - 2 * 64 / 7.5e-3) < 1e-6


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        workload, layers, kv_len, seed, steps, warmup, gpus = "tiny", None, None, 0, 1, 0, 2

    bench.run_reference(A, rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.0, 1, "cpu") == 4.0
    assert bench.job_tokens_per_s(64, 1, 8.0) == pytest.approx(8000.0)
