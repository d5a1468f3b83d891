"""Expert parallelism: the MoE layer with its experts split over the ranks of a
process group ("From PCIe to NVLink", section "Part I: Laying the Foundation":
the serving system shards the 384 experts over the GPUs, EP8 / EP4).

Rank r holds experts [r * E / G, (r + 1) * E / G) of G ranks, and its own
tokens.  One call:

1. plan (host): every (token, slot) pair goes to the rank that holds its
   expert; pairs are sent in destination order (stable, so in flat pair order
   within a destination), with the expert's local index there;
2. dispatch: the pair counts, then each pair's x row, local expert id and
   routing weight, by all-to-all;
3. the local layer on the received rows, one routing slot per row (top_k = 1,
   the pair's own weight): each row's weighted expert output;
4. combine: the rows go back by the reverse all-to-all and each is added into
   its token's output.

The collectives are torch.distributed's all_to_all_single (NCCL between GPUs,
gloo on the host).  `local_forward` computes step 3: on the GPU, the library's
forward on the rank's own packed experts (`gpu_local_forward`).  On CUDA tensors
the row movement of steps 2 and 4 runs in the library's kernels
(`moe_ep_gather`: the x row of every sent pair; `moe_ep_combine`: the returned
rows added into their tokens' output rows); torch indexes only the per-pair
routing weights.  Host tensors (the gloo path) use torch's indexing for the
same two steps.  Ids outside [0, E) are dropped, as in the single-GPU layer.
"""
from __future__ import annotations

import numpy as np
import torch


class DispatchPlan:
    """Where each routing pair of this rank goes.

    send_pairs  flat pair indices (t * top_k + j) in send order
    send_tokens their tokens
    local_ids   their experts' indices on the destination rank
    send_counts pairs per destination rank
    """

    def __init__(self, topk_ids: np.ndarray, E: int, world: int):
        if E % world:
            raise ValueError(f"{E} experts do not split evenly over {world} ranks")
        ids = np.asarray(topk_ids, dtype=np.int64)
        self.M, self.top_k = ids.shape
        flat = ids.reshape(-1)
        per = E // world
        valid = np.nonzero((flat >= 0) & (flat < E))[0]
        dest = flat[valid] // per
        order = np.argsort(dest, kind="stable")
        self.send_pairs = valid[order]
        self.send_tokens = self.send_pairs // self.top_k
        self.local_ids = (flat[self.send_pairs] - dest[order] * per).astype(np.int32)
        self.send_counts = np.bincount(dest, minlength=world).astype(np.int64)
        self.experts_per_rank = per


def _a2a(out_rows, t: torch.Tensor, send_counts, recv_counts, group):
    import torch.distributed as dist
    out = t.new_empty((out_rows,) + tuple(t.shape[1:]))
    dist.all_to_all_single(out, t.contiguous(), [int(c) for c in recv_counts],
                           [int(c) for c in send_counts], group=group)
    return out


def exchange_counts(send_counts: np.ndarray, device, group) -> np.ndarray:
    """Pairs this rank receives from each rank."""
    import torch.distributed as dist
    s = torch.as_tensor(send_counts, dtype=torch.int64, device=device)
    r = torch.empty_like(s)
    dist.all_to_all_single(r, s, group=group)
    return r.cpu().numpy()


def dispatch(plan: DispatchPlan, x: torch.Tensor, topk_weights: torch.Tensor, group):
    """Sends each pair's x row, local expert id and weight to the expert's rank.
    Returns (rows [R, H], ids int32 [R, 1], weights fp32 [R, 1], recv_counts)."""
    dev = x.device
    recv_counts = exchange_counts(plan.send_counts, dev, group)
    R = int(recv_counts.sum())
    tok = torch.as_tensor(plan.send_tokens, device=dev)
    if x.is_cuda and x.element_size() == 2:
        from . import ops
        send_x = ops.moe_ep_gather(x, tok)
    else:
        send_x = x.index_select(0, tok)
    send_ids = torch.as_tensor(plan.local_ids, device=dev)
    send_w = topk_weights.reshape(-1).index_select(0, torch.as_tensor(plan.send_pairs, device=dev))
    # 2-byte rows (bf16 x) travel as int32 pairs: not every backend moves 16-bit
    # integers, and the bits are all that matter here
    packed = send_x.element_size() == 2 and send_x.shape[-1] % 2 == 0
    rows = _a2a(R, send_x.view(torch.int32) if packed else send_x, plan.send_counts,
                recv_counts, group)
    if packed:
        rows = rows.view(x.dtype)
    ids = _a2a(R, send_ids, plan.send_counts, recv_counts, group)
    w = _a2a(R, send_w, plan.send_counts, recv_counts, group)
    return rows, ids.view(R, 1), w.view(R, 1), recv_counts


def combine(plan: DispatchPlan, rows_out: torch.Tensor, recv_counts, group) -> torch.Tensor:
    """Returns the weighted expert outputs to their pairs' ranks and sums each
    token's pairs: out [M, H]."""
    back = _a2a(len(plan.send_pairs), rows_out, recv_counts, plan.send_counts, group)
    out = torch.zeros((plan.M, rows_out.shape[1]), dtype=rows_out.dtype, device=rows_out.device)
    tok = torch.as_tensor(plan.send_tokens, device=rows_out.device)
    if back.is_cuda and back.dtype == torch.float32:
        from . import ops
        ops.moe_ep_combine(back, tok, out)
    else:
        out.index_add_(0, tok, back)
    return out


def ep_forward(x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor, E: int,
               local_forward, group=None) -> torch.Tensor:
    """The MoE layer with experts split over the group: out [M, H] for this
    rank's tokens.  local_forward(rows, ids [R, 1], weights [R, 1]) returns the
    weighted outputs [R, H] of the rank's own experts (see gpu_local_forward)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    plan = DispatchPlan(topk_ids.cpu().numpy(), E, world)
    rows, ids, w, recv_counts = dispatch(plan, x, topk_weights, group)
    rows_out = local_forward(rows, ids, w)
    return combine(plan, rows_out, recv_counts, group)


def gpu_local_forward(packed_weights, workspace=None):
    """local_forward for ep_forward on a GPU: the library's forward on this
    rank's packed experts (shape.E = the experts of one rank), one routing slot
    per received row."""
    from . import ops
    sh = packed_weights.shape
    local = ops.Shape.of(sh.E, 1, sh.hidden, sh.inter, ops.MOE_OUT_F32, sh.weight_format, sh.flags)

    def run(rows, ids, w):
        if rows.shape[0] == 0:
            return torch.zeros((0, sh.hidden), dtype=torch.float32, device=rows.device)
        return ops.moe_int4_forward(rows, packed_weights.w13, packed_weights.w13_scales,
                                    packed_weights.w2, packed_weights.w2_scales, ids, w, local,
                                    workspace=workspace)
    return run
