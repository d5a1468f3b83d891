"""Expert parallelism on the GPU: the library's row kernels of the dispatch and
the combine (moe_ep_gather, moe_ep_combine), and the whole expert-parallel layer
(plan, dispatch, the library's forward on the rank's experts, combine) on one
GPU as a one-rank NCCL group, against the single-process oracle."""
import socket

import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import inputs
from helpers import assert_parity

pytestmark = pytest.mark.gpu


def _ops():
    from weight_only_int4_moe_gb300 import ops
    return ops


def test_gather_copies_rows_and_zeroes_bad_indices():
    import torch
    ops = _ops()
    rng = np.random.default_rng(5)
    R, H = 37, 264
    src = rng.integers(-2 ** 15, 2 ** 15, size=(R, H), dtype=np.int16)
    rows = rng.integers(0, R, size=301).astype(np.int32)
    rows[[3, 77]] = [R, -1]  # outside the source: zeroed and reported
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = ops.moe_ep_gather(torch.from_numpy(src).cuda(), torch.from_numpy(rows).cuda(),
                            bad=bad).cpu().numpy()
    want = src[np.clip(rows, 0, R - 1)].copy()
    want[[3, 77]] = 0
    assert np.array_equal(got, want)
    assert int(bad.item()) == 1
    empty = ops.moe_ep_gather(torch.from_numpy(src).cuda(),
                              torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert tuple(empty.shape) == (0, H)


def test_combine_adds_repeated_rows_and_drops_bad_indices():
    import torch
    ops = _ops()
    rng = np.random.default_rng(6)
    n, H, M = 500, 512, 23
    src = rng.standard_normal((n, H)).astype(np.float32)
    rows = rng.integers(0, M, size=n).astype(np.int32)
    rows[[0, 9]] = [M + 3, -2]  # dropped and reported
    out0 = rng.standard_normal((M, H)).astype(np.float32)
    out = torch.from_numpy(out0).cuda()
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.moe_ep_combine(torch.from_numpy(src).cuda(), torch.from_numpy(rows).cuda(), out, bad=bad)
    want = out0.astype(np.float64)
    keep = (rows >= 0) & (rows < M)
    np.add.at(want, rows[keep], src[keep].astype(np.float64))
    got = out.cpu().numpy().astype(np.float64)
    # fp32 atomic sums in any order: within a few ulps of the fp64 sum of the terms
    tol = 1e-6 * (np.abs(out0).max() + np.abs(src).max() * np.bincount(rows[keep]).max())
    assert np.abs(got - want).max() <= tol
    assert int(bad.item()) == 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_expert_parallel_layer_on_one_gpu_matches_the_oracle():
    """The full expert-parallel path with one rank: every pair is dispatched to
    this rank through the NCCL all-to-all, its x row gathered by
    moe_ep_gather, run through the library's forward with one slot per row,
    sent back and combined by moe_ep_combine."""
    import torch
    import torch.distributed as dist
    from weight_only_int4_moe_gb300 import ep
    ops = _ops()
    E, K, H, I, M = 16, 4, 512, 256, 45
    w = inputs.make_weights(E, H, I, 91)
    t = inputs.make_tokens(inputs.MoEConfig("ep", E, K, H, I, (M,), "uniform", 0, 92), M)
    ids = t["topk_ids"].copy()
    ids[7, 2] = E + 1  # dropped, as in the single-GPU layer
    pw = ops.PackedWeights(w, E, H, I, K)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1)
    try:
        x = torch.from_numpy(t["x"].view(np.int16)).cuda().view(torch.bfloat16)
        got = ep.ep_forward(x, torch.from_numpy(ids).cuda(),
                            torch.from_numpy(t["topk_weights"]).cuda(), E,
                            ep.gpu_local_forward(pw))
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    ref, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], ids,
                                t["topk_weights"])
    assert_parity(got.cpu().numpy(), ref, "expert-parallel layer, one rank")
