"""The forward inside a CUDA graph.  moe_int4_forward and moe_int4_forward_routed
are stream-ordered, allocate nothing and read every routing-dependent size
(bucket lengths, block count, schedule) on the device, so one capture replays
correctly for new inputs of the same M: new tokens, a new routing, new routing
weights.  Each replay is checked against the oracle on the inputs it read."""
import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import inputs
from helpers import assert_parity

pytestmark = pytest.mark.gpu


def _ops():
    from weight_only_int4_moe_gb300 import ops
    return ops


def _tokens(E, k, H, I, M, seed, routing="uniform"):
    cfg = inputs.MoEConfig("graph", E, k, H, I, (M,), routing, 0, seed)
    return inputs.make_tokens(cfg, M)


def _oracle(w, t, tokens=None):
    out, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], t["topk_ids"],
                                t["topk_weights"], tokens=tokens)
    return out


def _capture(fn):
    """Run fn once on a side stream (first-call set-up stays outside the
    capture), then capture it into a graph."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("E,k,H,I,M,routing,plan", [
    (16, 4, 384, 256, 5, "uniform", "default"),      # 20 pairs: the small-batch kernels
    (16, 4, 384, 256, 37, "uniform", "default"),     # 148 pairs, L2-resident experts: the same
    (16, 4, 384, 256, 37, "uniform", "tensor"),      # ragged M, single-block align
    (64, 6, 512, 256, 700, "skewed", "default"),     # multi-block align, skewed routing
    (8, 2, 512, 256, 1000, "uniform", "default"),    # wide blocks of 192 rows
    (384, 8, 256, 128, 90, "uniform", "default"),    # 16-row blocks: the per-block down kernel
])
def test_forward_graph_replays_new_inputs(E, k, H, I, M, routing, plan):
    import torch
    ops = _ops()
    w = inputs.make_weights(E, H, I, 300 + E)
    pw = ops.PackedWeights(w, E, H, I, k)
    if plan == "tensor":
        pw.shape = ops.Shape.of(E, k, H, I, flags=ops.MOE_FLAG_NO_GEMV)
    ws = ops.alloc_workspace(M, pw.shape)
    x = torch.empty((M, H), dtype=torch.int16, device="cuda")
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((M, k), dtype=torch.float32, device="cuda")
    out = torch.empty((M, H), dtype=torch.float32, device="cuda")

    def load(t):
        x.copy_(torch.from_numpy(np.ascontiguousarray(t["x"]).view(np.int16)))
        ids.copy_(torch.from_numpy(np.ascontiguousarray(t["topk_ids"], dtype=np.int32)))
        tw.copy_(torch.from_numpy(np.ascontiguousarray(t["topk_weights"], dtype=np.float32)))

    load(_tokens(E, k, H, I, M, 40, routing))
    g = _capture(lambda: pw.forward(x.view(torch.bfloat16), ids, tw, out=out, workspace=ws))
    for seed in (41, 42, 43):
        t = _tokens(E, k, H, I, M, seed, routing)
        load(t)
        g.replay()
        torch.cuda.synchronize()
        assert_parity(out.cpu().numpy(), _oracle(w, t), f"graph replay seed {seed}")


def test_routed_forward_graph_replays_new_logits():
    """Router logits in, routing and output out: the routing of each replay is
    the router oracle's, bit for bit, and the output matches the MLP oracle."""
    import torch
    ops = _ops()
    E, k, H, I, M = 32, 4, 384, 256, 29
    w = inputs.make_weights(E, H, I, 501)
    pw = ops.PackedWeights(w, E, H, I, k)
    ws = ops.alloc_workspace(M, pw.shape)
    x = torch.empty((M, H), dtype=torch.int16, device="cuda")
    logits = torch.empty((M, E), dtype=torch.float32, device="cuda")
    out = torch.empty((M, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((M, k), dtype=torch.float32, device="cuda")

    def draw(seed):
        rng = np.random.default_rng([7, seed])
        xb = inputs.bf16_bits_from_f32(rng.standard_normal((M, H), dtype=np.float32))
        lg = rng.standard_normal((M, E), dtype=np.float32)
        x.copy_(torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)))
        logits.copy_(torch.from_numpy(lg))
        return xb, lg

    draw(0)
    g = _capture(lambda: ops.moe_int4_forward_routed(
        x.view(torch.bfloat16), pw.w13, pw.w13_scales, pw.w2, pw.w2_scales, logits, pw.shape,
        out=out, topk_ids=ids, topk_weights=tw, workspace=ws))
    for seed in (1, 2):
        xb, lg = draw(seed)
        g.replay()
        torch.cuda.synchronize()
        ref_ids, ref_w = oracle.route(lg, k)
        np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
        np.testing.assert_allclose(tw.cpu().numpy(), ref_w, rtol=1e-5, atol=0)
        t = {"x": xb, "topk_ids": ref_ids, "topk_weights": tw.cpu().numpy()}
        assert_parity(out.cpu().numpy(), _oracle(w, t), f"routed graph replay seed {seed}")
