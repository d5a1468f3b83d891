"""Expert parallelism (weight_only_int4_moe_gb300.ep) on the host: the dispatch
plan, and the whole dispatch -> local layer -> combine path over two gloo ranks,
each holding half of the experts and its own tokens.  The local layer here is
the oracle restricted to the rank's experts, so the result must equal the
single-process oracle on the same tokens up to fp64 summation order.  (On GPUs
the local layer is the library's forward; that path has one GPU per run here and
is not measured.)"""
import json
import os
import socket

import numpy as np
import pytest

from weight_only_int4_moe_gb300 import ep, inputs

E, K, H, I = 8, 2, 256, 128


def test_plan_orders_pairs_by_destination_and_drops_invalid_ids():
    ids = np.array([[5, 0], [3, 6], [-1, 4], [7, 8], [1, 1]])
    plan = ep.DispatchPlan(ids, E, 2)  # rank 0: experts 0..3, rank 1: 4..7
    # valid pairs in flat order: 0:5 1:0 2:3 3:6 5:4 6:7 8:1 9:1 (4: -1 and 7: 8 dropped)
    assert plan.send_counts.tolist() == [4, 4]
    assert plan.send_pairs.tolist() == [1, 2, 8, 9, 0, 3, 5, 6]  # stable within a rank
    assert plan.send_tokens.tolist() == [0, 1, 4, 4, 0, 1, 2, 3]
    assert plan.local_ids.tolist() == [0, 3, 1, 1, 1, 2, 0, 3]
    with pytest.raises(ValueError):
        ep.DispatchPlan(ids, 9, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = inputs.make_weights(E, H, I, 77)  # every rank draws the same weight set
    M = 12 + 5 * rank
    t = inputs.make_tokens(inputs.MoEConfig("ep", E, K, H, I, (M,), "uniform", 0, 80 + rank), M)
    ids = t["topk_ids"].copy()
    if rank == 1:
        ids[3, 1] = E + 5  # dropped, as in the single-GPU layer
    if rank == 0:
        ids[:, :] = ids % (E // world)  # rank 0 routes only to its own experts
    per = E // world
    lo = rank * per
    local = {k: w[k][lo:lo + per] for k in ("q13", "s13", "q2", "s2")}

    def local_forward(rows, rids, rw):
        if rows.shape[0] == 0:
            return torch.zeros((0, H), dtype=torch.float64)
        out, _ = oracle.moe_forward(rows.numpy().view(np.uint16), local["q13"], local["s13"],
                                    local["q2"], local["s2"], rids.numpy(), rw.numpy())
        return torch.from_numpy(out)

    x = torch.from_numpy(t["x"].view(np.int16))
    got = ep.ep_forward(x, torch.from_numpy(ids), torch.from_numpy(t["topk_weights"]), E,
                        local_forward).numpy()
    ref, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], ids,
                                t["topk_weights"])
    rms = float(np.sqrt(np.mean(ref ** 2)))
    plan = ep.DispatchPlan(ids, E, world)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max_over_rms": float(np.abs(got - ref).max()) / rms, "rms": rms,
                   "send_counts": plan.send_counts.tolist()}, f)


def test_two_ranks_match_the_single_process_oracle(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn",
                       join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert got[0]["send_counts"][1] == 0       # rank 0 sent nothing to rank 1
    assert sum(got[1]["send_counts"]) == 17 * K - 1  # one pair of rank 1 dropped
    for g in got:
        assert g["rms"] > 0
        assert g["max_over_rms"] <= 1e-12, g
