"""The multi-rank path of bench.py on CPU: two gloo ranks (one process per
rank, rendezvous on 127.0.0.1) each report a different local time; every
rank must see the slowest one, and the whole-job rate must count the work of
both ranks over that time (weak scaling: a replica per rank, no exchange)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_s = [0.75, 1.25][rank]
    slowest = bench.rank_max(local_s, "cpu")
    rate = bench.whole_job_rate(10.0, 4, world, slowest)
    out[rank] = (slowest, rate, bench.dist_env())
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        slowest, rate, env = out[rank]
        assert slowest == pytest.approx(1.25)
        assert rate == pytest.approx(10.0 * 4 * 2 / 1.25)
        assert env == (rank, world, rank)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.rank_max(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(2.0, 3, 1, 1.5) == pytest.approx(4.0)


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference times the CPU oracle and prints one JSON line
    with the contract's keys (run on CPU, tiny workload)."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "fp32_256", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s"
    assert line["value"] > 0 and line["higher_is_better"] is True
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "config", "cpu_baseline",
                "e2e"):
        assert key in line
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
