"""The router on the GPU (moe_route, and fused with the align in
moe_int4_forward_routed) against the router oracle: expert ids bit for bit (the
selection is decided by exact fp32 comparisons of the logits, ties to the lower
index), weights within fp32 rounding of the fp64 softmax, and the routed layer
within the layer's parity bounds."""
import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import inputs
from helpers import assert_parity

pytestmark = pytest.mark.gpu

W_RTOL = 2e-6  # fp32 expf / divide against the fp64 softmax


def _ops():
    from weight_only_int4_moe_gb300 import ops
    return ops


def _logits(M, E, seed):
    return np.random.default_rng([11, M, E, seed]).standard_normal((M, E), dtype=np.float32)


@pytest.mark.parametrize("M,E,k", [
    (1, 384, 8), (9, 384, 8), (90, 384, 8), (1000, 384, 8),  # decode and verify sizes
    (17, 1024, 32), (33, 32, 32), (64, 37, 5), (5, 1, 1), (3, 2, 2), (0, 384, 8)])
def test_route_matches_oracle(M, E, k):
    import torch
    ops = _ops()
    lg = _logits(M, E, 1)
    ids, w = ops.moe_route(torch.from_numpy(lg).cuda(), k)
    torch.cuda.synchronize()
    rid, rw = oracle.route(lg, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=W_RTOL, atol=0)


def test_route_ties_and_extremes():
    import torch
    ops = _ops()
    rng = np.random.default_rng(3)
    lg = rng.integers(-2, 3, (200, 160)).astype(np.float32)  # many exact ties
    lg[5] = 0.0                                               # all equal
    lg[6, ::7] = 80.0                                         # exp range
    lg[7] = -np.arange(160, dtype=np.float32) * 30.0          # tiny weights underflow
    for k in (1, 4, 8, 32):
        ids, w = ops.moe_route(torch.from_numpy(lg).cuda(), k)
        torch.cuda.synchronize()
        rid, rw = oracle.route(lg, k)
        np.testing.assert_array_equal(ids.cpu().numpy(), rid)
        np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=W_RTOL, atol=1e-30)


ROUTED = [
    # E, k, H, I, M, seed: fused route+align (M <= 32, P <= 4096), router kernel +
    # single-block align (M > 32), router kernel + multi-block align (P > 4096)
    (8, 2, 256, 128, 16, 0), (16, 4, 384, 256, 37, 1), (32, 4, 256, 128, 300, 2),
    (64, 6, 512, 256, 700, 3), (384, 8, 256, 128, 9, 4)]


@pytest.mark.parametrize("plan", ["default", "tensor"])
@pytest.mark.parametrize("E,k,H,I,M,seed", ROUTED)
def test_forward_routed_matches_oracle(E, k, H, I, M, seed, plan):
    """The router in front of the default plan (the small-batch kernels at
    these sizes where they apply) and of the tensor-core kernels (the fused
    route + align, or the router kernel and the align)."""
    import torch
    ops = _ops()
    w = inputs.make_weights(E, H, I, 600 + seed)
    pw = ops.PackedWeights(w, E, H, I, k)
    if plan == "tensor":
        pw.shape = ops.Shape.of(E, k, H, I, flags=ops.MOE_FLAG_NO_GEMV)
    rng = np.random.default_rng([12, seed])
    x = inputs.bf16_bits_from_f32(rng.standard_normal((M, H), dtype=np.float32))
    lg = _logits(M, E, seed)
    out, ids, tw = ops.moe_int4_forward_routed(
        torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16), pw.w13, pw.w13_scales,
        pw.w2, pw.w2_scales, torch.from_numpy(lg).cuda(), pw.shape)
    torch.cuda.synchronize()
    rid, rw = oracle.route(lg, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(tw.cpu().numpy(), rw, rtol=W_RTOL, atol=0)
    ref, _ = oracle.moe_forward(x, w["q13"], w["s13"], w["q2"], w["s2"], rid, rw)
    assert_parity(out.float().cpu().numpy(), ref, f"routed E{E} k{k} M{M} {plan}")


def test_forward_routed_equals_forward_on_its_routing():
    """The routed layer is the layer applied to the routing it returns."""
    import torch
    ops = _ops()
    E, k, H, I, M = 64, 6, 512, 256, 120
    w = inputs.make_weights(E, H, I, 650)
    pw = ops.PackedWeights(w, E, H, I, k)
    rng = np.random.default_rng(13)
    x = torch.from_numpy(inputs.bf16_bits_from_f32(
        rng.standard_normal((M, H), dtype=np.float32)).view(np.int16)).cuda().view(torch.bfloat16)
    lg = torch.from_numpy(_logits(M, E, 9)).cuda()
    out_r, ids, tw = ops.moe_int4_forward_routed(x, pw.w13, pw.w13_scales, pw.w2, pw.w2_scales,
                                                 lg, pw.shape)
    out_f = pw.forward(x, ids, tw)
    torch.cuda.synchronize()
    a, b = out_r.float().cpu().numpy(), out_f.float().cpu().numpy()
    # equal up to the order of the fp32 atomic adds of the top-k combine
    np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-5 * float(np.abs(b).max()))
