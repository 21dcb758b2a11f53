"""Multi-rank host logic on CPU (gloo, world_size 2): rows shard across ranks
with no data-path collective; timing is reduced with a max over ranks; the
reference arm runs on rank 0 only."""
import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(float(rank + 1) * 1.5, world, torch.device("cpu"))
    bench.barrier(world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29611
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get() for _ in range(2))
    assert res == {0: 3.0, 1: 3.0}


@pytest.mark.slow
def test_reference_arm_two_ranks_prints_once():
    env = dict(os.environ)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29623", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "tiny4x1024_f32", "--ref-rows", "4"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_reference_arm_verification_workload():
    """The reference arm of the verification bench: the oracle over all
    sequences of the workload per step, one JSON line with the contract's
    keys."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
           "--warmup", "3", "--workload", "verify256x4x128256_f32"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "sequences/s" and d["value"] > 0
    assert d["config"]["workload"] == "verify256x4x128256_f32"


def _shard_worker(rank, world, port, q):
    """One rank of the job: its shard of the workload (the helper bench.py
    uses for --gpus N), run through the oracle, gathered over gloo."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch
    import gpu_helpers as H
    from top_selection_stats_gb300 import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = workloads.random_case(41, 12, 3001, dtype="bf16", mask_frac=0.3)
    shard = workloads.rank_shard(case, rank, world)
    r = H.oracle_run(shard, threads=1)
    mine = {k: torch.as_tensor(np.ascontiguousarray(r[k]).astype(np.int64))
            for k in ("status", "token", "kept_count", "kept_mask")}
    out = {}
    for k, t in mine.items():
        parts = [torch.empty_like(t) for _ in range(world)]
        dist.all_gather(parts, t)
        out[k] = torch.cat(parts).numpy()
    if rank == 0:
        q.put(out)
    dist.barrier()
    dist.destroy_process_group()


def test_row_shards_over_two_ranks_equal_the_single_rank_job():
    """world_size 2 (gloo, CPU): each rank runs its contiguous shard; the
    shards' results, concatenated, equal one rank running the whole job."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import gpu_helpers as H
    from top_selection_stats_gb300 import workloads
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, 29631, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = q.get(timeout=300)
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    case = workloads.random_case(41, 12, 3001, dtype="bf16", mask_frac=0.3)
    whole = H.oracle_run(workloads.global_job(case, 2), threads=1)
    for k in ("status", "token", "kept_count", "kept_mask"):
        assert np.array_equal(got[k], np.asarray(whole[k]).astype(np.int64)), k
    # the two shards draw differently (their offsets differ)
    assert not np.array_equal(got["token"][:12], got["token"][12:])
