"""Pins for the oracle (CPU only).

The oracle is checked against things other than itself: exact bf16 values,
hand-derived closed forms (tests/golden/closed_form_cases.json), an independent
all-experts dense formulation built from numpy matmul, the special case top_k=1
with weight 1 (one dense dequantised MLP), linearity in the routing weights,
invariance to unrouted experts and to the slot order, and brute-force sorting
for the align buffers.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


# ----------------------------------------------------------------------------
# independent numpy formulation (library matmul, all experts, dense masks)
# ----------------------------------------------------------------------------
def np_unpack(q):
    lo = (q & 0x0F).astype(np.int64)
    hi = (q >> 4).astype(np.int64)
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def np_dequant(q, s):
    vals = np_unpack(q).astype(np.float64) - 8.0
    sc = inputs.f32_from_bf16_bits(s).astype(np.float64)
    return vals * np.repeat(sc, 32, axis=-1)


def np_dense_moe(x_bits, w, ids, tw):
    x = inputs.f32_from_bf16_bits(x_bits).astype(np.float64)
    W13 = np_dequant(w["q13"], w["s13"])
    W2 = np_dequant(w["q2"], w["s2"])
    E, twoI, H = W13.shape
    I = twoI // 2
    M = x.shape[0]
    out = np.zeros((M, H))
    for e in range(E):
        gu = x @ W13[e].T
        g, u = gu[:, :I], gu[:, I:]
        a = g / (1.0 + np.exp(-g)) * u
        y = a @ W2[e].T
        coef = np.where(ids == e, tw.astype(np.float64), 0.0).sum(axis=1)
        out += coef[:, None] * y
    return out


def tiny_case(seed=0, M=16, E=8, k=2, H=256, I=128):
    cfg = inputs.MoEConfig("t", E, k, H, I, (M,), "uniform", seed, 100 + seed)
    w = inputs.make_weights(E, H, I, 1000 + seed)
    t = inputs.make_tokens(cfg, M)
    return w, t


def run_oracle(w, t, **kw):
    return oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"],
                              t["topk_ids"], t["topk_weights"], **kw)


def rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


# ----------------------------------------------------------------------------
# scalar conventions
# ----------------------------------------------------------------------------
def test_bf16_exact_values():
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x3C23) == 163.0 / 16384.0
    assert oracle.bf16_to_double(0x3C80) == 2.0 ** -6
    assert oracle.bf16_to_double(0x0000) == 0.0


def test_nibble_order():
    row = np.array([0x21, 0xF0, 0x8A], dtype=np.uint8)
    assert [oracle.nibble(row, k) for k in range(6)] == [1, 2, 0, 15, 10, 8]


def test_dequant_formula_endpoints():
    q = np.full((1, 2, 32), 0x88, dtype=np.uint8)
    s = np.full((1, 2, 2), 0x3C00, dtype=np.uint16)  # 2^-7
    q[0, 1, 20] = 0xF0  # k=40 -> 0 (low), k=41 -> 15 (high)
    s[0, 1, 1] = 0x3F00  # 0.5 for k in [32, 64)
    assert oracle.weight(q, s, 0, 1, 40) == -8 * 0.5
    assert oracle.weight(q, s, 0, 1, 41) == 7 * 0.5
    assert oracle.weight(q, s, 0, 1, 39) == 0.0
    assert oracle.weight(q, s, 0, 0, 41) == 0.0


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------
def _build_case(c):
    E, H, I, M, k = c["E"], c["H"], c["I"], c["M"], c["top_k"]
    rng = np.random.default_rng(7)
    q13 = np.full((E, 2 * I, H // 2), 0x88, dtype=np.uint8)
    q2 = np.full((E, H, I // 2), 0x88, dtype=np.uint8)
    s13 = np.full((E, 2 * I, H // 32), 0x3C00, dtype=np.uint16)
    s2 = np.full((E, H, I // 32), 0x3C00, dtype=np.uint16)
    routed = {e for row in c["topk_ids"] for e in row}
    for e in range(E):  # experts nobody routes to: random junk
        if e not in routed:
            q13[e] = rng.integers(0, 256, q13[e].shape, dtype=np.uint8)
            q2[e] = rng.integers(0, 256, q2[e].shape, dtype=np.uint8)
    for e_str, spec in c.get("experts", {}).items():
        e = int(e_str)
        nib = lambda v: np.uint8(v | (v << 4))
        q13[e, :I] = nib(spec["gate_q"])
        q13[e, I:] = nib(spec["up_q"])
        q2[e] = nib(spec["down_q"])
        s13[e] = int(spec["s13"], 16)
        s2[e] = int(spec["s2"], 16)
    for mat, q, s in (("w13", q13, s13), ("w2", q2, s2)):
        for ent in c.get("sparse", {}).get(mat, []):
            r, col, v = ent["row"], ent["col"], ent["q"]
            b = q[0, r, col // 2]
            b = (b & 0xF0) | v if col % 2 == 0 else (b & 0x0F) | (v << 4)
            q[0, r, col // 2] = b
            s[0, r, col // 32] = int(ent["scale"], 16)
    xs = c["x"]
    if "fill" in xs:
        x = np.full((M, H), xs["fill"], dtype=np.float32)
    else:
        x = np.zeros((M, H), dtype=np.float32)
        x[:, xs["one_hot"]] = xs["value"]
    w = {"q13": q13, "s13": s13, "q2": q2, "s2": s2}
    t = {"x": inputs.bf16_bits_from_f32(x),
         "topk_ids": np.array(c["topk_ids"], dtype=np.int32),
         "topk_weights": np.array(c["topk_weights"], dtype=np.float32)}
    return w, t


@pytest.mark.parametrize("name", ["uniform_sigmoid", "two_slot_combine", "one_hot_index"])
def test_closed_form(name):
    cases = {c["name"]: c for c in json.load(open(GOLDEN))["cases"]}
    c = cases[name]
    w, t = _build_case(c)
    out, dropped = run_oracle(w, t)
    assert dropped == 0
    if "expected_all" in c:
        np.testing.assert_allclose(out, c["expected_all"], rtol=1e-13, atol=0)
    else:
        exp = np.zeros_like(out)
        for h, v in c["expected_sparse"].items():
            exp[0, int(h)] = v
        np.testing.assert_allclose(out, exp, rtol=1e-13, atol=1e-300)


# ----------------------------------------------------------------------------
# library routine / brute force
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_dense_all_expert_numpy(seed):
    w, t = tiny_case(seed)
    out, _ = run_oracle(w, t)
    ref = np_dense_moe(t["x"], w, t["topk_ids"], t["topk_weights"])
    assert rel(out, ref) < 1e-12


def test_odd_shapes_and_k():
    cfg = inputs.MoEConfig("t", 5, 3, 96, 64, (7,), "uniform", 0, 55)
    w = inputs.make_weights(5, 96, 64, 55)
    t = inputs.make_tokens(cfg, 7)
    out, _ = run_oracle(w, t)
    ref = np_dense_moe(t["x"], w, t["topk_ids"], t["topk_weights"])
    assert rel(out, ref) < 1e-12


def test_top1_weight1_is_dense_mlp():
    w, t = tiny_case(3, M=12)
    ids = t["topk_ids"][:, :1].copy()
    tw = np.ones((12, 1), dtype=np.float32)
    out, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], ids, tw)
    W13 = np_dequant(w["q13"], w["s13"])
    W2 = np_dequant(w["q2"], w["s2"])
    x = inputs.f32_from_bf16_bits(t["x"]).astype(np.float64)
    I = W13.shape[1] // 2
    for m in range(12):
        e = ids[m, 0]
        gu = W13[e] @ x[m]
        a = gu[:I] / (1 + np.exp(-gu[:I])) * gu[I:]
        y = W2[e] @ a
        assert rel(out[m], y) < 1e-12


def test_linearity_in_routing_weights():
    w, t = tiny_case(4)
    base, _ = run_oracle(w, t)
    t2 = dict(t, topk_weights=(t["topk_weights"] * 4).astype(np.float32))
    out2, _ = run_oracle(w, t2)
    np.testing.assert_array_equal(out2, 4 * base)  # power-of-two scale is exact
    rng = np.random.default_rng(9)
    wa = rng.uniform(-1, 1, t["topk_weights"].shape).astype(np.float32)
    wb = rng.uniform(-1, 1, t["topk_weights"].shape).astype(np.float32)
    oa, _ = run_oracle(w, dict(t, topk_weights=wa))
    ob, _ = run_oracle(w, dict(t, topk_weights=wb))
    oab, _ = run_oracle(w, dict(t, topk_weights=(wa.astype(np.float64) + wb).astype(np.float32)))
    # wa+wb is rounded to fp32 once; compare against the same rounded weights
    assert rel(oab, oa + ob) < 1e-6
    exact = (wa.astype(np.float64) + wb) == (wa + wb).astype(np.float64)
    assert exact.mean() > 0.3


def test_unrouted_experts_do_not_matter():
    w, t = tiny_case(5)
    used = set(np.unique(t["topk_ids"]).tolist())
    base, _ = run_oracle(w, t)
    rng = np.random.default_rng(11)
    w2 = {k: v.copy() for k, v in w.items()}
    for e in range(w["q13"].shape[0]):
        if e not in used:
            for key in w2:
                w2[key][e] = rng.integers(0, 2 ** (8 if key[0] == "q" else 16),
                                          w2[key][e].shape).astype(w2[key].dtype)
    out, _ = run_oracle(w2, t)
    np.testing.assert_array_equal(out, base)


def test_slot_permutation_invariance():
    w, t = tiny_case(6)
    base, _ = run_oracle(w, t)
    perm = [1, 0]
    t2 = dict(t, topk_ids=t["topk_ids"][:, perm].copy(),
              topk_weights=t["topk_weights"][:, perm].copy())
    out, _ = run_oracle(w, t2)
    assert rel(out, base) < 1e-12


def test_zero_cases():
    w, t = tiny_case(7)
    zx = dict(t, x=np.zeros_like(t["x"]))
    out, _ = run_oracle(w, zx)
    assert not out.any()
    w8 = dict(w, q13=np.full_like(w["q13"], 0x88))
    out, _ = run_oracle(w8, t)
    assert not out.any()
    # a zero scale group equals zeroing that slice of x (w13 groups are along H)
    g = 3
    wz = dict(w, s13=w["s13"].copy())
    wz["s13"][:, :, g] = 0
    xz = t["x"].copy()
    xz[:, 32 * g: 32 * g + 32] = 0
    a, _ = run_oracle(wz, t)
    b, _ = run_oracle(w, dict(t, x=xz))
    np.testing.assert_array_equal(a, b)


def test_invalid_ids_dropped_and_counted():
    w, t = tiny_case(8)
    ids = t["topk_ids"].copy()
    ids[3, 1] = 8
    ids[5, 0] = -1
    out, dropped = run_oracle(w, dict(t, topk_ids=ids))
    assert dropped == 2
    ref = np_dense_moe(t["x"], w, ids, t["topk_weights"])
    assert rel(out, ref) < 1e-12


def test_intermediate_matches_numpy():
    w, t = tiny_case(9)
    pairs = np.arange(t["topk_ids"].size)
    a = oracle.moe_intermediate(t["x"], w["q13"], w["s13"], t["topk_ids"], pairs)
    W13 = np_dequant(w["q13"], w["s13"])
    x = inputs.f32_from_bf16_bits(t["x"]).astype(np.float64)
    I = W13.shape[1] // 2
    k = t["topk_ids"].shape[1]
    for p in pairs:
        e = t["topk_ids"].reshape(-1)[p]
        gu = W13[e] @ x[p // k]
        ref = gu[:I] / (1 + np.exp(-gu[:I])) * gu[I:]
        assert rel(a[p], ref) < 1e-12


def test_token_subset_equals_full():
    w, t = tiny_case(10)
    full, _ = run_oracle(w, t)
    sub, _ = run_oracle(w, t, tokens=np.array([15, 0, 7]))
    np.testing.assert_array_equal(sub, full[[15, 0, 7]])


# ----------------------------------------------------------------------------
# align
# ----------------------------------------------------------------------------
def brute_align(ids, E, B):
    flat = list(np.asarray(ids).reshape(-1))
    P = len(flat)
    valid = sorted((int(e), i) for i, e in enumerate(flat) if 0 <= e < E)
    sorted_ids, expert_ids = [], []
    for e in range(E):
        bucket = [i for (ee, i) in valid if ee == e]
        if not bucket:
            continue
        n = math.ceil(len(bucket) / B) * B
        sorted_ids += bucket + [P] * (n - len(bucket))
        expert_ids += [e] * (n // B)
    return sorted_ids, expert_ids, P - len(valid)


@pytest.mark.parametrize("M,k,E,B,seed", [
    (16, 2, 8, 16, 0), (1, 8, 384, 16, 1), (90, 8, 384, 16, 2), (33, 6, 64, 64, 3),
    (200, 8, 384, 128, 4), (5, 3, 7, 1, 5), (0, 8, 384, 16, 6), (64, 4, 3, 48, 7)])
def test_align_matches_brute_force(M, k, E, B, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-1, E + 1, (M, k)).astype(np.int32)  # includes invalid ids
    s, e, n, dropped = oracle.align(ids, E, B)
    bs, be, bd = brute_align(ids, E, B)
    assert list(s) == bs and list(e) == be and n == len(bs) and dropped == bd
    valid = ids[(ids >= 0) & (ids < E)]
    assert (s < M * k).sum() == valid.size  # every valid pair exactly once
    assert len(set(s[s < M * k].tolist())) == valid.size
    assert n % max(B, 1) == 0


def test_align_all_one_expert():
    ids = np.full((40, 2), 3, dtype=np.int32)
    s, e, n, d = oracle.align(ids, 8, 16)
    assert n == 80 and list(e) == [3] * 5 and list(s) == list(range(80))


# --------------------------------------------------------------- router --
# Router oracle (top-k by logit, renormalised softmax over the chosen k).

def test_route_closed_form_two_experts():
    """Logits 0 and ln 3: softmax weights 1/4 and 3/4 (closed form)."""
    lg = np.array([[0.0, np.log(3.0), -2.0]], dtype=np.float32)
    ids, w = oracle.route(lg, 2)
    assert ids.tolist() == [[1, 0]]
    l1 = float(np.float32(np.log(3.0)))
    expect = np.array([np.exp(l1), 1.0]) / (np.exp(l1) + 1.0)
    np.testing.assert_allclose(w[0], expect, rtol=0, atol=1e-15)
    np.testing.assert_allclose(w[0], [0.75, 0.25], atol=1e-7)


def test_route_distinct_logits_reduce_to_library_sort_and_softmax():
    """With distinct logits the ids are numpy's descending argsort and the
    weights scipy's softmax of the chosen logits."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((40, 96)).astype(np.float32)
    for k in (1, 2, 8, 96):
        ids, w = oracle.route(lg, k)
        order = np.argsort(-lg.astype(np.float64), axis=1, kind="stable")[:, :k]
        np.testing.assert_array_equal(ids, order)
        chosen = np.take_along_axis(lg.astype(np.float64), order, axis=1)
        np.testing.assert_allclose(w, special.softmax(chosen, axis=1), rtol=1e-13, atol=0)


def test_route_invariants():
    rng = np.random.default_rng(6)
    lg = rng.standard_normal((64, 384)).astype(np.float32)
    ids, w = oracle.route(lg, 8)
    # weights sum to one, are positive and descending with the logits
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-14)
    assert (w > 0).all() and (np.diff(w, axis=1) <= 0).all()
    # ids are distinct and every chosen logit is >= every unchosen one
    for t in range(64):
        assert len(set(ids[t].tolist())) == 8
        rest = np.delete(lg[t], ids[t])
        assert lg[t, ids[t]].min() >= rest.max()
    # a shift of every logit by an exactly representable constant changes nothing
    ids2, w2 = oracle.route((lg.astype(np.float64) + 4.0).astype(np.float32), 8)
    np.testing.assert_array_equal(ids2, ids)
    np.testing.assert_allclose(w2, w, rtol=1e-6)
    # top-1: weight exactly one
    _, w1 = oracle.route(lg, 1)
    assert (w1 == 1.0).all()


def test_route_ties_take_the_lower_index_with_equal_weights():
    lg = np.zeros((2, 16), dtype=np.float32)
    lg[0, [3, 7, 11]] = 2.0  # three-way tie at the top
    ids, w = oracle.route(lg, 4)
    assert ids[0].tolist() == [3, 7, 11, 0]
    assert ids[1].tolist() == [0, 1, 2, 3]
    np.testing.assert_allclose(w[1], 0.25, atol=1e-15)
    assert w[0, 0] == w[0, 1] == w[0, 2]


def test_route_agrees_with_the_generator_recipe():
    """The input generator routes by an independent recipe (fp32 softmax over
    all experts, stable top-k of the probabilities, renormalise)."""
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((128, 384)).astype(np.float32)
    gid, gw = inputs.route(lg, 8)
    ids, w = oracle.route(lg, 8)
    np.testing.assert_array_equal(ids, gid)
    np.testing.assert_allclose(w, gw, rtol=2e-6)
