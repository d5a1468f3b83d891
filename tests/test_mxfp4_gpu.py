"""MXFP4 experts (E2M1 codes, one E8M0 scale per 32) on the GPU: the packed
scale factors, and moe_int4_forward with shape.weight_format = MOE_W_MXFP4
against the MXFP4 oracle across block-height regimes, element by element."""
import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import inputs
from helpers import assert_parity, gpu_forward

pytestmark = pytest.mark.gpu


def _ops():
    from weight_only_int4_moe_gb300 import ops
    return ops


def _factor_bits(e):
    """fp16 bits of 2^(e - 127), the packed factor of an E8M0 code e, clamped to
    the supported range [103, 140] -- from its definition, on the host."""
    x = min(13, max(-24, int(e) - 127))
    return (x + 15) << 10 if x >= -14 else 1 << (x + 24)


def test_packed_scales_are_the_fp16_factors_and_out_of_range_codes_are_counted():
    import torch
    ops = _ops()
    E, N, K = 2, 256, 128
    rng = np.random.default_rng(4)
    q = torch.from_numpy(rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)).cuda()
    s = rng.integers(103, 141, (E, N, K // 32), dtype=np.uint8)
    s[0, 0, 0], s[0, 0, 1] = 103, 140  # the ends of the range
    s[0, 3, 1] = 255   # NaN code
    s[1, 7, 0] = 141   # above the range
    s[1, 9, 2] = 102   # below
    sd = torch.from_numpy(s).cuda()
    _, packed_s, bad = ops.moe_mxfp4_pack(q, sd, True)
    torch.cuda.synchronize()
    assert int(bad.item()) == 3
    # The scale layout is the INT4 one: an INT4 pack of distinct marker scales
    # shows which packed slot holds which group.
    n_groups = E * N * (K // 32)
    marker = (0x3C00 + np.arange(n_groups)).astype(np.uint16).reshape(E, N, K // 32)
    _, packed_m = ops.moe_int4_pack(q, torch.from_numpy(marker.view(np.int16)).cuda(), True)
    torch.cuda.synchronize()
    pm = packed_m.cpu().numpy().view(np.uint16)
    ps = packed_s.cpu().numpy().view(np.uint16)
    # the markers are bf16 values in fp16's normal range: their fp16 bits are exact
    mf = inputs.f32_from_bf16_bits(marker.ravel()).astype(np.float16).view(np.uint16)
    pos_of = {int(v): i for i, v in enumerate(mf)}
    assert len(pos_of) == len(mf)
    s_flat = s.ravel()
    for j in range(len(pm)):
        g = pos_of[int(pm[j])]
        assert ps[j] == _factor_bits(s_flat[g]), (j, g, s_flat[g])


SHAPES = [
    # E, k, H, I, M, seed
    (8, 2, 256, 128, 16, 0),      # block 16
    (16, 4, 384, 256, 37, 1),     # block 32, ragged
    (16, 4, 384, 256, 96, 2),     # block 64
    (4, 1, 256, 128, 300, 3),     # block 128
    (64, 6, 512, 256, 700, 4),    # multi-block align
    (8, 2, 512, 256, 1000, 5),    # wide 192
    (4, 2, 384, 256, 300, 6),     # wide 192, three down row tiles
    (384, 8, 256, 128, 90, 7),    # default plan: separate, per-block down kernel
]


@pytest.mark.parametrize("plan", ["default", "tensor"])
@pytest.mark.parametrize("E,k,H,I,M,seed", SHAPES)
def test_mxfp4_forward_matches_oracle(E, k, H, I, M, seed, plan):
    """Each shape through the default plan (the small-batch kernels where they
    apply) and through the tensor-core kernels."""
    ops = _ops()
    w = inputs.make_weights_mxfp4(E, H, I, 40 + seed)
    pw = ops.PackedWeights(w, E, H, I, k, fmt="mxfp4")
    assert pw.shape.weight_format == ops.MOE_W_MXFP4
    if plan == "tensor":
        pw.shape = ops.Shape.of(E, k, H, I, weight_format=ops.MOE_W_MXFP4,
                                flags=ops.MOE_FLAG_NO_GEMV)
    t = inputs.make_tokens(inputs.MoEConfig("mx", E, k, H, I, (M,), "uniform", 0, 60 + seed), M)
    got = gpu_forward(pw, t)
    ref, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], t["topk_ids"],
                                t["topk_weights"], fmt="mxfp4")
    print(assert_parity(got, ref, f"mxfp4 E{E} M{M} {plan}"))


def test_the_two_formats_agree_on_weights_both_hold():
    """INT4 (q - 8 = m, scale 0.5) and MXFP4 (E2M1 code of m, scale 2^-1) copies
    of the same weights: the two forwards agree to fp32 rounding."""
    ops = _ops()
    E, k, H, I, M = 8, 2, 256, 128, 40
    rng = np.random.default_rng(8)
    m_set = np.array([0, 1, -1, 2, -2, 3, -3, 4, -4, 6, -6])
    code_of = {0: 0, 1: 2, 2: 4, 3: 5, 4: 6, 6: 7}

    def draw(shape):
        m = rng.choice(m_set, size=shape)
        qi = (m + 8).astype(np.uint8)
        qf = np.vectorize(lambda v: code_of[abs(int(v))] | (8 if v < 0 else 0))(m).astype(np.uint8)
        pack = lambda c: (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
        return pack(qi), pack(qf)

    i13, f13 = draw((E, 2 * I, H))
    i2, f2 = draw((E, H, I))
    wi = {"q13": i13, "s13": np.full((E, 2 * I, H // 32), 0x3F00, np.uint16),
          "q2": i2, "s2": np.full((E, H, I // 32), 0x3F00, np.uint16)}
    wf = {"q13": f13, "s13": np.full((E, 2 * I, H // 32), 126, np.uint8),
          "q2": f2, "s2": np.full((E, H, I // 32), 126, np.uint8)}
    t = inputs.make_tokens(inputs.MoEConfig("mx", E, k, H, I, (M,), "uniform", 0, 77), M)
    oi = gpu_forward(ops.PackedWeights(wi, E, H, I, k), t)
    of = gpu_forward(ops.PackedWeights(wf, E, H, I, k, fmt="mxfp4"), t)
    scale = np.abs(oi).max()
    np.testing.assert_allclose(of, oi, rtol=0, atol=1e-5 * scale)


@pytest.mark.slow
def test_mxfp4_k26_shapes_sampled():
    """The K2.6 layer shapes (hidden 7168, inter 2048, top-8) with 48 MXFP4
    experts at M = 90, in the forward's own launch configuration: every output
    finite, sampled tokens against the oracle."""
    ops = _ops()
    E, k, H, I, M = 48, 8, 7168, 2048, 90
    w = inputs.make_weights_mxfp4(E, H, I, 123)
    pw = ops.PackedWeights(w, E, H, I, k, fmt="mxfp4")
    t = inputs.make_tokens(inputs.MoEConfig("mx", E, k, H, I, (M,), "uniform", 0, 124), M)
    got = gpu_forward(pw, t)
    assert np.all(np.isfinite(got))
    toks = np.sort(np.random.default_rng(5).choice(M, size=4, replace=False))
    ref, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], t["topk_ids"],
                                t["topk_weights"], tokens=toks, fmt="mxfp4")
    print(assert_parity(got[toks], ref, "mxfp4 K2.6 shapes E48 M90"))
