"""The bounded pipeline waits, on the GPU, through the debug-bounds build (run
as a child process by test_timeout_gpu.py; MOE_INT4_DEBUG_BOUNDS=1).

That build's host hook MOE_INT4_DEBUG_SKIP_STAGE=i makes CTA 0 of the first GEMM
kernel leave the copy of its weight stage i out: the mbarrier that the stage's
copy would complete is never completed, so the wait for it must run out (about
50 ms in this build), set MOE_DEVERR_TIMEOUT and wind the grid down.  Nothing
faults and nothing traps.  The call must return, report the flag, and leave the
context usable: a normal forward right after it matches the oracle."""
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
from weight_only_int4_moe_gb300 import build, inputs, ops  # noqa: E402
from helpers import assert_parity  # noqa: E402


def run(flags, label):
    import torch
    E, k, H, I, M = 8, 2, 7168, 512, 32  # CTA 0 streams about a dozen gate/up stages
    w = inputs.make_weights(E, H, I, 1001)
    pw = ops.PackedWeights(w, E, H, I, k)
    pw.shape = ops.Shape.of(E, k, H, I, flags=flags)
    t = inputs.make_tokens(inputs.MoEConfig("to", E, k, H, I, (M,), "uniform", 0, 1002), M)
    x = torch.from_numpy(t["x"].view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.from_numpy(t["topk_ids"]).cuda()
    tw = torch.from_numpy(t["topk_weights"]).cuda()
    ws = ops.alloc_workspace(M, pw.shape)

    os.environ["MOE_INT4_DEBUG_SKIP_STAGE"] = "5"
    t0 = time.perf_counter()
    pw.forward(x, ids, tw, workspace=ws)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    del os.environ["MOE_INT4_DEBUG_SKIP_STAGE"]
    fl, _ = ops.moe_int4_get_errors(ws)
    assert fl & ops.MOE_DEVERR_TIMEOUT, hex(fl)
    assert dt < 20.0, dt  # the waits gave up, in tens of milliseconds each

    # the context is still usable: a clean call matches the oracle
    ops.moe_int4_clear_errors(ws)
    out = pw.forward(x, ids, tw, workspace=ws)
    torch.cuda.synchronize()
    assert ops.moe_int4_get_errors(ws) == (0, 0)
    ref, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], t["topk_ids"],
                                t["topk_weights"])
    assert_parity(out.cpu().numpy(), ref, label)
    print(f"{label}: timeout reported after {dt * 1e3:.0f} ms, next call clean", flush=True)


def main():
    assert ops.debug_bounds(), "run with MOE_INT4_DEBUG_BOUNDS=1"
    ops.load_library()
    assert ops.library_path() == build.DEBUG_LIB
    run(ops.MOE_FLAG_NO_GEMV, "fused decode kernel")
    run(ops.MOE_FLAG_UNFUSED, "separate kernels")
    print("timeouts: all cases reported and recovered", flush=True)


if __name__ == "__main__":
    main()
