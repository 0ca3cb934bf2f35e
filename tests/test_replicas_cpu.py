"""The multi-GPU path is replicas only (the layer needs no exchange): check
the benchmark's rank combination and the reference arm's rank handling with
two gloo ranks on the CPU."""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _worker(rank, ws, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import bench
    r, w, d = bench.dist_init(backend="gloo")
    assert (r, w) == (rank, ws) and d is not None
    d.barrier()
    total_ms, value = bench.combine_ranks(times[rank], 100, w, d, torch.device("cpu"))
    out[rank] = (total_ms, value)
    d.barrier()
    d.destroy_process_group()


def test_combine_ranks_takes_the_slowest_rank_gloo():
    ws, port = 2, 29517
    times = [12.5, 20.0]                 # ms for 100 steps on each rank
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(ws, port, times, out), nprocs=ws, join=True)
        res = dict(out)
    for rank in range(ws):
        total_ms, value = res[rank]
        assert total_ms == 20.0                   # the slowest rank
        assert value == pytest.approx(20.0 * 1e3 / 100 / ws)   # µs per step of the whole job


def test_combine_ranks_single_process():
    import bench
    total_ms, value = bench.combine_ranks(7.0, 70, 1, None, torch.device("cpu"))
    assert total_ms == 7.0 and value == pytest.approx(100.0)


def test_reference_arm_non_zero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT="29519")
    # rank 1 of the reference arm returns before any work or collective
    import bench  # noqa: F401  (import check)
    code = ("import sys; sys.argv=['bench.py','--impl','reference','--steps','1','--warmup','0'];"
            "import bench; bench.dist_init = lambda backend='nccl': (1, 2, None); bench.main()")
    p = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_reference_arm_prints_one_contract_line():
    """N = 1: the reference arm (the oracle on the host cores) prints one JSON
    line with the contract's keys and its own e2e and cpu_baseline."""
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["higher_is_better"] is False and d["value"] > 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert "workload" in d["config"]
