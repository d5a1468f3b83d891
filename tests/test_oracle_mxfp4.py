"""The MXFP4 weight format of the oracle (e2m1(q) * 2^(e - 127), one E8M0 scale
per 32 along K), pinned to things other than its own formula: the E2M1 value
table of the OCP Microscaling specification (tests/golden/e2m1_values.json),
PyTorch's float8_e8m0fnu decoder for the scales, a dense numpy MLP on weights
dequantised from those two, and exact agreement with the INT4 path on weights
both formats represent identically."""
import json
import os

import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_values.json")


def _table():
    d = json.load(open(GOLDEN))
    vals = np.array([d["values"][str(c)] for c in range(16)], dtype=np.float64)
    return d, vals


def test_e2m1_matches_the_specification_table():
    d, vals = _table()
    got = np.array([oracle.e2m1(c) for c in range(16)])
    np.testing.assert_array_equal(got, vals)
    assert np.signbit(oracle.e2m1(8))  # -0
    ch = d["characteristic"]
    pos = got[:8]
    assert pos.max() == ch["max_normal"]
    assert pos[2] == ch["min_normal"]  # exponent field 1, mantissa 0
    assert pos[1] == ch["max_subnormal"] == ch["min_subnormal"]


def test_e2m1_sign_symmetry_and_order():
    v = [oracle.e2m1(c) for c in range(16)]
    for c in range(8):
        assert v[c + 8] == -v[c]
    assert all(a < b for a, b in zip(v[:7], v[1:8]))


def test_e8m0_matches_the_library_decoder():
    torch = pytest.importorskip("torch")
    codes = np.arange(255, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([oracle.e8m0(int(c)) for c in codes])
    np.testing.assert_array_equal(got, lib)
    assert np.isnan(oracle.e8m0(255))
    assert oracle.e8m0(127) == 1.0 and oracle.e8m0(128) == 2.0 and oracle.e8m0(126) == 0.5


def _dequant_numpy(q, s, vals):
    """[E, N, K] weights from canonical nibbles and E8M0 bytes, with the table
    values and the library scale decoder."""
    import torch
    lo = (q & 0x0F).astype(np.int64)
    hi = (q >> 4).astype(np.int64)
    codes = np.stack([lo, hi], axis=-1).reshape(q.shape[0], q.shape[1], -1)
    scale = torch.from_numpy(np.ascontiguousarray(s)).view(torch.float8_e8m0fnu).to(
        torch.float64).numpy()
    return vals[codes] * np.repeat(scale, 32, axis=2)


def test_weight_entries_match_numpy():
    pytest.importorskip("torch")
    _, vals = _table()
    w = inputs.make_weights_mxfp4(3, 64, 32, 5)
    W = _dequant_numpy(w["q13"], w["s13"], vals)
    rng = np.random.default_rng(1)
    for _ in range(200):
        e, n, k = rng.integers(0, 3), rng.integers(0, 64), rng.integers(0, 64)
        assert oracle.weight_fmt("mxfp4", w["q13"], w["s13"], e, n, k) == W[e, n, k]


def test_top1_weight1_is_the_dense_mlp():
    """top_k = 1 with weight 1: each token's output is one expert's dense MLP,
    computed here with numpy matmuls on independently dequantised weights."""
    pytest.importorskip("torch")
    _, vals = _table()
    E, H, I, M = 4, 64, 32, 9
    w = inputs.make_weights_mxfp4(E, H, I, 7)
    rng = np.random.default_rng(3)
    x = inputs.bf16_bits_from_f32(rng.standard_normal((M, H), dtype=np.float32))
    ids = rng.integers(0, E, (M, 1)).astype(np.int32)
    tw = np.ones((M, 1), dtype=np.float32)
    out, dropped = oracle.moe_forward(x, w["q13"], w["s13"], w["q2"], w["s2"], ids, tw,
                                      fmt="mxfp4")
    assert dropped == 0
    W13 = _dequant_numpy(w["q13"], w["s13"], vals)
    W2 = _dequant_numpy(w["q2"], w["s2"], vals)
    xf = inputs.f32_from_bf16_bits(x).astype(np.float64)
    for t in range(M):
        e = ids[t, 0]
        g = W13[e, :I] @ xf[t]
        u = W13[e, I:] @ xf[t]
        a = g / (1 + np.exp(-g)) * u
        np.testing.assert_allclose(out[t], W2[e] @ a, rtol=1e-12, atol=1e-12)


def test_agrees_exactly_with_int4_on_shared_values():
    """Weights m / 2 with m in {0, +-1, +-2, +-3, +-4, +-6}, which both formats
    hold exactly -- INT4 as q - 8 = m with scale 0.5, MXFP4 as the E2M1 code of
    m with scale 2^-1 -- give bit-identical oracle outputs."""
    E, H, I, M, k = 3, 64, 32, 5, 2
    rng = np.random.default_rng(11)
    m_set = np.array([0, 1, -1, 2, -2, 3, -3, 4, -4, 6, -6])
    code_of = {0: 0, 1: 2, 2: 4, 3: 5, 4: 6, 6: 7}  # E2M1 code of |m|

    def draw(shape):
        m = rng.choice(m_set, size=shape)
        q_int4 = (m + 8).astype(np.uint8)
        q_fp4 = np.array([code_of[abs(int(v))] | (8 if v < 0 else 0) for v in m.ravel()],
                         dtype=np.uint8).reshape(shape)
        return q_int4, q_fp4

    def pack(codes):  # canonical nibble order: even k in the low nibble
        return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)

    i13, f13 = draw((E, 2 * I, H))
    i2, f2 = draw((E, H, I))
    s13_i = np.full((E, 2 * I, H // 32), 0x3F00, dtype=np.uint16)  # bf16 0.5
    s2_i = np.full((E, H, I // 32), 0x3F00, dtype=np.uint16)
    s13_f = np.full((E, 2 * I, H // 32), 126, dtype=np.uint8)  # E8M0 2^-1
    s2_f = np.full((E, H, I // 32), 126, dtype=np.uint8)
    x = inputs.bf16_bits_from_f32(rng.standard_normal((M, H), dtype=np.float32))
    ids = rng.integers(0, E, (M, k)).astype(np.int32)
    tw = rng.uniform(0.1, 1.0, (M, k)).astype(np.float32)
    out_i, _ = oracle.moe_forward(x, pack(i13), s13_i, pack(i2), s2_i, ids, tw)
    out_f, _ = oracle.moe_forward(x, pack(f13), s13_f, pack(f2), s2_f, ids, tw, fmt="mxfp4")
    assert np.abs(out_i).max() > 0
    np.testing.assert_array_equal(out_f, out_i)
