"""bench.py's multi-replica host logic on CPU: two ranks over gloo (the GPU runs
use NCCL with one replica per GPU; the path does not shard, so there is no data
exchange, only the barrier and the max over ranks of the step time)."""
import json
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup()
    dist = bench.dist_init(w, local, use_gpu=False)
    bench.barrier(dist, use_gpu=False)
    step_s = 0.010 * (rank + 1)  # rank 1 is the slower one
    slowest = bench.allreduce_max(dist, step_s, use_gpu=False)
    value = bench.job_rate(w, 100, slowest)
    bench.barrier(dist, use_gpu=False)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "slowest": slowest, "value": value}, f)


def test_two_gloo_ranks_agree_on_the_slowest_step(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn",
                       join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, g in enumerate(got):
        assert g["world"] == 2 and g["rank"] == r
        assert g["slowest"] == pytest.approx(0.020)
        # whole-job rate: both replicas' units over the slowest step
        assert g["value"] == pytest.approx(2 * 100 / 0.020)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.dist_init(1, 0, use_gpu=False) is None
    assert bench.allreduce_max(None, 3.5, use_gpu=False) == 3.5
    bench.barrier(None, use_gpu=False)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    """Under torchrun every rank runs bench.py; only rank 0 times the oracle."""
    import bench
    bench.run_reference(None, None, [1], world=2, rank=1)
    assert capsys.readouterr().out == ""
