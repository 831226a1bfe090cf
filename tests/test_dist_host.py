"""The multi-process path of bench.py on the CPU, world size 2 over gloo.

The layers and images are independent, so N ranks run N replicas with no data
exchange; the only collective is the max over ranks of the timed totals.  These
tests run that reduction in two gloo processes, check the whole-job rate, and
launch the reference arm under torchrun: rank 0 alone prints its line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    got = bench.reduce_max(values[rank], dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(got))


def test_reduce_max_over_two_gloo_ranks(tmp_path):
    values = [3.25, 7.5]
    mp.start_processes(_rank_main, args=(2, _free_port(), values, str(tmp_path)), nprocs=2,
                       join=True, start_method="spawn")
    got = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(2)]
    assert got == [7.5, 7.5]


def test_single_rank_needs_no_collective():
    assert bench.reduce_max(4.0, None, "cpu") == 4.0


def test_job_rate_is_weak_scaling():
    # two replicas of 1 TFLOP in the slowest rank's 2 ms: 1000 TFLOP/s
    assert bench.job_rate(1e12, 2, 2.0, 1e12) == pytest.approx(1000.0)
    assert bench.job_rate(1e12, 1, 2.0, 1e12) == pytest.approx(500.0)


def test_reference_arm_under_torchrun_prints_on_rank0_only():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "bcast",
           "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
