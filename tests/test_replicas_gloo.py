"""Host-side logic of the multi-GPU benchmark, run as gloo ranks on the CPU.

The path does not shard across GPUs here (every logical rank lives in one
GPU's memory), so N GPUs run N independent replicas: the only cross-rank
operations are the barrier and the max-time / sum-of-units reduction of the
benchmark, tested here with world_size 2.
"""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (rank, rank, world)
    dist.barrier()
    ms, units = bench.reduce_over_ranks(1.5 + rank, 1000.0 * (rank + 1), world)
    q.put((rank, ms, units))
    dist.barrier()
    dist.destroy_process_group()


def test_max_time_and_summed_units_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, units in res:
        assert ms == 2.5          # the slowest rank's time
        assert units == 3000.0    # units of all ranks


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.0, 7.0, 1) == (3.0, 7.0)
    nb = bench.algorithmic_bytes(32768, 7168, 8, 294656)
    # the bytes the prefill step must move (padding rows excluded)
    assert nb["dispatch_bf16"] == 32768 * 7168 * 2 + 32768 * 8 * 4 + 32768 * 8 * 7168 * 2
    assert nb["combine"] == 32768 * 8 * 7168 * 2 + 2 * 32768 * 8 * 4 + 32768 * 7168 * 2
    assert nb["dispatch_fp8"] == 32768 * 7168 * 2 + 32768 * 8 * 4 + 32768 * 8 * (7168 + 56 * 4)
