"""Checks of the seeded input recipe (CPU only)."""
import numpy as np

from weight_only_int4_moe_gb300 import inputs


def test_bf16_rounding_is_rne():
    vals = np.array([1.0, 1.00390625, 1.01171875, -3.5, 0.0, 1e-3], dtype=np.float32)
    b = inputs.bf16_bits_from_f32(vals)
    # 1 + 2^-8 is a tie between 1 and 1+2^-7: ties to even -> 1.0 (0x3F80)
    assert b[0] == 0x3F80 and b[1] == 0x3F80
    # 1 + 3*2^-8 is a tie between 1+2^-7 (odd) and 1+2^-6 (even) -> 0x3F82
    assert b[2] == 0x3F82
    assert inputs.f32_from_bf16_bits(b[3]) == -3.5
    back = inputs.f32_from_bf16_bits(b)
    assert np.all(np.abs(back - vals) <= np.abs(vals) * 2 ** -8)


def test_weights_shapes_ranges_and_determinism():
    w = inputs.make_weights(4, 64, 32, 3)
    assert w["q13"].shape == (4, 64, 32) and w["s13"].shape == (4, 64, 2)
    assert w["q2"].shape == (4, 64, 16) and w["s2"].shape == (4, 64, 1)
    s = inputs.f32_from_bf16_bits(w["s13"])
    assert s.min() >= 0.0049 and s.max() <= 0.0201
    w2 = inputs.make_weights(4, 64, 32, 3)
    for k in w:
        np.testing.assert_array_equal(w[k], w2[k])
    nib = np.concatenate([w["q13"].reshape(-1) & 15, w["q13"].reshape(-1) >> 4])
    assert set(np.unique(nib).tolist()) == set(range(16))


def test_routing_uniform():
    cfg = inputs.WORKLOADS["tiny"]
    t = inputs.make_tokens(cfg, 16)
    ids, w = t["topk_ids"], t["topk_weights"]
    assert ids.shape == (16, 2) and w.shape == (16, 2)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-6)
    assert np.all(w[:, 0] >= w[:, 1])
    assert all(len(set(r)) == 2 for r in ids.tolist())


def test_routing_skewed_share():
    cfg = inputs.WORKLOADS["k26_verify"]
    small = inputs.MoEConfig("s", 384, 8, 64, 64, (256,), "skewed", 1, 2)
    t = inputs.make_tokens(small, 256)
    assert abs(t["hot_share"] - 0.5) <= 0.011
    assert len(t["hot"]) == 77
    assert cfg.routing == "skewed"


def test_router_logits_reproduce_the_routings():
    """Routing the generated router logits gives the generator's routings
    (uniform and skewed recipes)."""
    for cfg, M in ((inputs.WORKLOADS["tiny"], 16), (inputs.MoEConfig("s", 64, 8, 128, 128, (40,), "skewed", 2, 9), 40)):
        pool = [inputs.make_tokens(cfg, M)["topk_ids"]] + [ids for ids, _ in inputs.routing_pool(cfg, M, 2)]
        for ids, lg in zip(pool, inputs.router_logits_pool(cfg, M, 2)):
            rid, _ = inputs.route(lg, cfg.top_k)
            np.testing.assert_array_equal(rid, ids)


def test_dequantised_int4_weights_are_exact_in_fp16():
    """The kernels form (q - 8) * scale in fp16 as one FMA,
    (16 + q) * s + fp16(-24 * s), rounded once.  For a bf16 scale s in
    [2^-14, 2729] the addend -24 * s is exact in fp16 and so is the result
    (8 + 3 significant bits): checked here over every positive bf16 value of
    that range and every q, the FMA's exact sum rounded to fp16 once."""
    bits = np.arange(0x3880, 0x4530, dtype=np.uint16)        # 2^-14 .. 2816 (exclusive)
    s = inputs.f32_from_bf16_bits(bits).astype(np.float64)
    s = s[(s >= 2.0 ** -14) & (s <= 2729.0)]
    assert s.min() == 2.0 ** -14 and s.max() == 2720.0
    addend = (-24.0 * s).astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(addend, -24.0 * s)           # exact
    q = np.arange(16, dtype=np.float64)[:, None]
    fma = ((16.0 + q) * s[None, :] + addend[None, :])          # exact in fp64
    got = fma.astype(np.float16).astype(np.float64)            # one rounding
    np.testing.assert_array_equal(got, (q - 8.0) * s[None, :])
    # the next bf16 value, 2736, makes the addend overflow: -24 * 2736 = -65664
    with np.errstate(over="ignore"):
        assert not np.isfinite(np.float16(-24.0 * 2736.0))
