"""The edges of the fp16 operand domain, on the GPU.

The tensor cores multiply fp16 operands: x is converted from bf16, the weights
(q - 8) * scale are formed in fp16, and the SwiGLU intermediate is stored as
fp16.  Inside fp16's exact range the forward must meet the oracle bound with no
flag raised; an x element or an intermediate beyond +-65504 must raise
MOE_DEVERR_RANGE, and moe_int4_pack must count every scale whose dequantised
weights are not exact in fp16."""
import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import inputs
from helpers import assert_parity, gpu_forward

pytestmark = pytest.mark.gpu

E, K, H, I, M = 8, 2, 256, 128, 24
# the default plan at this size is the small-batch kernels; "tensor" forces the
# tensor-core kernels, which have their own conversions and range checks
PLANS = ["default", "tensor"]


def _ops():
    from weight_only_int4_moe_gb300 import ops
    return ops


def _tokens(seed, x_scale=1.0):
    cfg = inputs.MoEConfig("edge", E, K, H, I, (M,), "uniform", 0, 800 + seed)
    t = dict(inputs.make_tokens(cfg, M))
    x = inputs.f32_from_bf16_bits(t["x"]) * np.float32(x_scale)
    t["x"] = inputs.bf16_bits_from_f32(x)
    return t


def _forward(w, t, plan="default"):
    ops = _ops()
    pw = ops.PackedWeights(w, E, H, I, K)
    if plan == "tensor":
        pw.shape = ops.Shape.of(E, K, H, I, flags=ops.MOE_FLAG_NO_GEMV)
    assert ops.moe_int4_gemv(M, pw.shape) == (plan == "default")
    ws = ops.alloc_workspace(M, pw.shape)
    got = gpu_forward(pw, t, workspace=ws)
    flags, _ = ops.moe_int4_get_errors(ws)
    return pw, got, flags


@pytest.mark.parametrize("plan", PLANS)
def test_edge_of_exact_range_meets_the_bound(plan):
    """Scales down at 2^-14 (the smallest normal fp16) and x up to +-3e4: the
    operands are exact, the intermediate stays in range, and the result meets
    the bound with no flag raised."""
    rng = np.random.default_rng(41)
    w = inputs.make_weights(E, H, I, 41)
    for name in ("s13", "s2"):
        s = rng.uniform(2.0 ** -14, 2.0 ** -12, size=w[name].shape).astype(np.float32)
        s.flat[::97] = 2.0 ** -14  # the boundary itself
        w[name] = inputs.bf16_bits_from_f32(s)
    t = _tokens(1, x_scale=3000.0)
    x = inputs.f32_from_bf16_bits(t["x"])
    x[:, 7] = 30000.0  # one large element per token
    x[::3, 100] = -30000.0
    t["x"] = inputs.bf16_bits_from_f32(x)
    a = oracle.moe_intermediate(t["x"], w["q13"], w["s13"], t["topk_ids"], np.arange(M * K))
    assert np.abs(a).max() < 65504  # the case stays inside the range
    pw, got, flags = _forward(w, t, plan)
    assert pw.inexact_scales == 0
    assert flags == 0, hex(flags)
    ref, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], t["topk_ids"],
                                t["topk_weights"])
    assert_parity(got, ref, "edge of the exact range")


@pytest.mark.parametrize("plan", PLANS)
def test_x_beyond_fp16_range_raises_the_flag(plan):
    ops = _ops()
    w = inputs.make_weights(E, H, I, 42)
    t = _tokens(2)
    x = inputs.f32_from_bf16_bits(t["x"])
    x[5, 17] = 1.0e5  # finite in bf16, beyond fp16
    t["x"] = inputs.bf16_bits_from_f32(x)
    _, _, flags = _forward(w, t, plan)
    assert flags & ops.MOE_DEVERR_RANGE


@pytest.mark.parametrize("plan", PLANS)
def test_intermediate_beyond_fp16_range_raises_the_flag(plan):
    """x in range (|x| < 1e4) but SiLU(g) * u beyond 65504."""
    ops = _ops()
    w = inputs.make_weights(E, H, I, 43)
    t = _tokens(3, x_scale=2000.0)
    assert np.abs(inputs.f32_from_bf16_bits(t["x"])).max() < 65504
    ref_a = oracle.moe_intermediate(t["x"], w["q13"], w["s13"], t["topk_ids"],
                                    np.arange(M * K))
    assert np.abs(ref_a).max() > 65504  # the case really leaves the range
    _, _, flags = _forward(w, t, plan)
    assert flags & ops.MOE_DEVERR_RANGE


@pytest.mark.parametrize("plan", PLANS)
def test_normal_inputs_raise_no_range_flag(plan):
    w = inputs.make_weights(E, H, I, 44)
    _, _, flags = _forward(w, _tokens(4), plan)
    assert flags == 0


def test_pack_counts_inexact_scales():
    """Exactly the non-zero scales outside [2^-14, 2729] (and non-finite ones)
    are counted; the largest bf16 inside is 2720, the next one 2736."""
    import torch
    ops = _ops()
    rng = np.random.default_rng(45)
    q = inputs._random_nibble_bytes(rng, (1, 256, 32))
    s = rng.uniform(0.005, 0.02, size=(1, 256, 2)).astype(np.float32)
    inside = [0.0, -0.0, 2.0 ** -14, -(2.0 ** -14), 2720.0, -2720.0]
    outside = [2.0 ** -15, 1e-6, -1e-7, 2736.0, -9000.0, 1e5, np.inf, -np.inf, np.nan]
    vals = inside + outside
    s.flat[: len(vals)] = vals
    bits = inputs.bf16_bits_from_f32(s)
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.moe_int4_pack(torch.from_numpy(q).cuda(), torch.from_numpy(bits.view(np.int16)).cuda(),
                      True, inexact=cnt)
    torch.cuda.synchronize()
    assert int(cnt.item()) == len(outside)
