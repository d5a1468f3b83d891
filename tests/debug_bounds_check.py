"""Run by test_debug_bounds_gpu.py in a process of its own with
MOE_INT4_DEBUG_BOUNDS=1: the forward through the debug-bounds build of the
library (index checks on every routing buffer read back by a kernel) on shapes
that cover each block-height regime, a multi-block align, the routed entry
point, dropped invalid ids and MXFP4 weights.  Each output must match the
oracle and no check may fire (MOE_DEVERR_BOUNDS clear).  Prints one line per
case; exits non-zero on the first failure."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
from helpers import assert_parity  # noqa: E402
from weight_only_int4_moe_gb300 import build, inputs, ops  # noqa: E402

CASES = [
    # E, k, H, I, M, routing   (block height from the forward's own policy)
    (8, 2, 256, 128, 16, "uniform"),       # 16, single-block align
    (16, 4, 384, 256, 37, "uniform"),      # 32
    (16, 4, 384, 256, 96, "uniform"),      # 64 (scalar combine)
    (8, 2, 256, 128, 160, "uniform"),      # 96
    (4, 1, 256, 128, 300, "uniform"),      # 128
    (64, 6, 512, 256, 700, "skewed"),      # multi-block align, skewed routing
    (8, 2, 512, 256, 1000, "uniform"),     # wide 192
    (128, 8, 1024, 512, 200, "uniform"),   # round-robin waves then the split part
    (384, 8, 256, 128, 90, "uniform"),     # 16, separate plan: the per-block down kernel
]


def run_case(E, k, H, I, M, routing, seed, flags=0):
    import torch
    w = inputs.make_weights(E, H, I, 900 + seed)
    pw = ops.PackedWeights(w, E, H, I, k)
    pw.shape = ops.Shape.of(E, k, H, I, flags=flags)
    t = inputs.make_tokens(inputs.MoEConfig("dbg", E, k, H, I, (M,), routing, 0, 950 + seed), M)
    x = torch.from_numpy(t["x"].view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.from_numpy(t["topk_ids"]).cuda()
    tw = torch.from_numpy(t["topk_weights"]).cuda()
    ws = ops.alloc_workspace(M, pw.shape)
    out = pw.forward(x, ids, tw, workspace=ws)
    torch.cuda.synchronize()
    flags, dropped = ops.moe_int4_get_errors(ws)
    assert flags == 0 and dropped == 0, (E, k, H, I, M, hex(flags), dropped)
    ref, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], t["topk_ids"],
                                t["topk_weights"])
    m = assert_parity(out.cpu().numpy(), ref, f"E{E} M{M}")
    plan = "small-batch" if ops.moe_int4_gemv(M, pw.shape) else (
        f"block_m={ops.moe_int4_block_m(M, pw.shape)}" +
        (", per-block down" if ops.moe_int4_block_down(M, pw.shape) else ""))
    print(f"E={E} k={k} H={H} I={I} M={M} {plan} "
          f"max/rms={m['max_over_rms']:.2e} rel_l1={m['rel_l1']:.2e}", flush=True)
    return w, pw


def run_invalid_ids(flags):
    """Out-of-range ids are dropped and reported (MOE_DEVERR_BAD_EXPERT_ID);
    the bounds checks stay quiet."""
    import torch
    E, k, H, I, M = 16, 4, 384, 256, 37
    w = inputs.make_weights(E, H, I, 990)
    pw = ops.PackedWeights(w, E, H, I, k)
    pw.shape = ops.Shape.of(E, k, H, I, flags=flags)
    t = inputs.make_tokens(inputs.MoEConfig("dbg", E, k, H, I, (M,), "uniform", 0, 991), M)
    bad = t["topk_ids"].copy()
    bad[::5, 1] = E + 2
    bad[3::7, 0] = -1
    x = torch.from_numpy(t["x"].view(np.int16)).cuda().view(torch.bfloat16)
    ws = ops.alloc_workspace(M, pw.shape)
    out = pw.forward(x, torch.from_numpy(bad).cuda(), torch.from_numpy(t["topk_weights"]).cuda(),
                     workspace=ws)
    torch.cuda.synchronize()
    flags, dropped = ops.moe_int4_get_errors(ws)
    assert flags == ops.MOE_DEVERR_BAD_EXPERT_ID, hex(flags)
    assert dropped == int(((bad < 0) | (bad >= E)).sum()), dropped
    ref, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], bad,
                                t["topk_weights"])
    assert_parity(out.cpu().numpy(), ref, "invalid ids")
    print(f"invalid ids (plan flags {pw.shape.flags:#x}): flags={flags:#x} dropped={dropped}",
          flush=True)


def run_routed(flags):
    import torch
    E, k, H, I, M = 32, 4, 384, 256, 29
    w = inputs.make_weights(E, H, I, 995)
    pw = ops.PackedWeights(w, E, H, I, k)
    pw.shape = ops.Shape.of(E, k, H, I, flags=flags)
    rng = np.random.default_rng([9, 5])
    xb = inputs.bf16_bits_from_f32(rng.standard_normal((M, H), dtype=np.float32))
    lg = rng.standard_normal((M, E), dtype=np.float32)
    ws = ops.alloc_workspace(M, pw.shape)
    out, ids, tw = ops.moe_int4_forward_routed(
        torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16), pw.w13, pw.w13_scales,
        pw.w2, pw.w2_scales, torch.from_numpy(lg).cuda(), pw.shape, workspace=ws)
    torch.cuda.synchronize()
    flags, dropped = ops.moe_int4_get_errors(ws)
    assert flags == 0 and dropped == 0, hex(flags)
    ref_ids, _ = oracle.route(lg, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    ref, _ = oracle.moe_forward(xb, w["q13"], w["s13"], w["q2"], w["s2"], ref_ids,
                                tw.cpu().numpy())
    assert_parity(out.cpu().numpy(), ref, "routed")
    print("routed: ok", flush=True)


def run_mxfp4():
    """The MXFP4 kernels (the same pipeline with the other dequant) under the
    same checks."""
    import torch
    E, k, H, I, M = 8, 2, 512, 256, 1000
    w = inputs.make_weights_mxfp4(E, H, I, 996)
    pw = ops.PackedWeights(w, E, H, I, k, fmt="mxfp4")
    t = inputs.make_tokens(inputs.MoEConfig("dbg", E, k, H, I, (M,), "uniform", 0, 997), M)
    x = torch.from_numpy(t["x"].view(np.int16)).cuda().view(torch.bfloat16)
    ws = ops.alloc_workspace(M, pw.shape)
    out = pw.forward(x, torch.from_numpy(t["topk_ids"]).cuda(),
                     torch.from_numpy(t["topk_weights"]).cuda(), workspace=ws)
    torch.cuda.synchronize()
    flags, dropped = ops.moe_int4_get_errors(ws)
    assert flags == 0 and dropped == 0, hex(flags)
    ref, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], t["topk_ids"],
                                t["topk_weights"], fmt="mxfp4")
    assert_parity(out.cpu().numpy(), ref, "mxfp4")
    print("mxfp4: ok", flush=True)


def main():
    assert ops.debug_bounds(), "run with MOE_INT4_DEBUG_BOUNDS=1"
    ops.load_library()
    assert ops.library_path() == build.DEBUG_LIB
    # every case through the tensor-core kernels, and through the matrix-vector
    # kernels (small-batch or per-block down) where the default plan picks them
    for i, case in enumerate(CASES):
        run_case(*case, seed=i, flags=ops.MOE_FLAG_NO_GEMV)
        E, k, H, I, M, _ = case
        sh = ops.Shape.of(E, k, H, I)
        if ops.moe_int4_gemv(M, sh) or ops.moe_int4_block_down(M, sh):
            run_case(*case, seed=i)
    for flags in (ops.MOE_FLAG_NO_GEMV, 0):
        run_invalid_ids(flags)
        run_routed(flags)
    run_mxfp4()
    print("debug-bounds: all cases clean", flush=True)


if __name__ == "__main__":
    main()
