"""The multi-rank timing path of bench.py on CPU with gloo (world size 2)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.dist_max(10.0 + rank, "cpu")          # rank 1 is the slowest
    rate = bench.whole_job_rate(world, 100.0, ms)
    dist.barrier()
    with open(os.path.join(out_dir, "r%d" % rank), "w") as f:
        f.write("%r %r\n" % (ms, rate))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for rank in range(world):
        ms, rate = map(float, open(tmp_path / ("r%d" % rank)).read().split())
        assert ms == 11.0                       # every rank sees the max
        assert rate == pytest.approx(2 * 100.0 / 11e-3)


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(3.5) == 3.5
    assert bench.whole_job_rate(1, 50.0, 2.0) == pytest.approx(25000.0)


def test_reference_arm_prints_one_contract_line():
    """bench.py --impl reference (the fp64 oracle on the host cores) runs
    without a GPU and prints one JSON line with the contract's keys."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 1
    assert line["value"] > 0 and line["unit"] == "TFLOPS" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "fwdbwd_causal_peaked_b2_h16_n8192_d128"
