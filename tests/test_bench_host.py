"""Host-side logic of the benchmark, on CPU.

The N > 1 path as world-size-2 gloo process groups: the path has no exchange step
(every (sequence, KV head) block is independent), so N GPUs run N replicas of the
workload; the only collective is the maximum of the timed region over the ranks, and
the reported value is the units all ranks processed per second of that slowest time
(weak scaling). The reference arm runs on rank 0 alone. And the prefill leg's CPU
baseline on a small prompt.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
    value = bench.whole_job_rate(16 * 256, world, ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
        json.dump({"ms": ms, "value": value}, fh)


def test_timed_region_is_the_slowest_rank_and_value_is_whole_job(tmp_path):
    import torch.multiprocessing as mp

    world = 2
    port = _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True, start_method="spawn")
    res = [json.load(open(os.path.join(tmp_path, f"rank{r}.json"))) for r in range(world)]
    assert all(r["ms"] == 15.0 for r in res)  # every rank holds the maximum
    assert all(abs(r["value"] - 16 * 256 * 2 / 15e-3) < 1e-6 for r in res)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.whole_job_rate(100, 1, 1000.0) == 100.0


def test_reference_arm_does_no_work_off_rank_zero():
    """Under torchrun the reference arm's ranks other than 0 exit 0 without output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_prefill_cpu_baseline_runs_on_a_small_prompt():
    """The prefill leg's CPU baseline (the oracle on host cores, sampled, scaled by the
    causal work) on a small prompt: one object of the bench contract's cpu_baseline form."""
    import numpy as np

    sys.path.insert(0, ROOT)
    import bench

    rng = np.random.default_rng(0)
    n = 128 + 128 * 2 + 40
    k = rng.standard_normal((n, 2, 128)).astype(np.float16)
    v = rng.standard_normal((n, 2, 128)).astype(np.float16)
    q = rng.standard_normal((n, 8, 128)).astype(np.float16)
    r = bench.prefill_cpu_baseline(k, v, q, positions_sample=16, head=1)
    assert r["kind"] == "oracle" and r["unit"] == "prompt tokens/s" and r["value"] > 0 and r["cores"] >= 1
