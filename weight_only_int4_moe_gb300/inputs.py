"""Seeded synthetic inputs for the INT4 MoE expert MLP.

This module only draws random inputs and converts them to their storage formats;
it contains none of the layer's arithmetic.  Both the CUDA path's tests/benchmark
and the oracle receive the arrays it returns.

Recipe (numpy ``default_rng``; the pages publish no dataset and no weights, so
every workload is synthetic with the shapes the pages benchmark -- 384 experts,
top-8, hidden 7168, intermediate 2048 in "The Throughput Lever", section
"Building the Benchmark"):

* weights, seed ``[0, weight_seed]`` (the three K2.6-shaped workloads share one
  weight set), drawn in the order q13, s13, q2, s2:
    - q: uniform random bytes, i.e. two nibbles per byte, each U{0..15};
      canonical storage [E][N][K/2], element k of a row in byte k/2, low nibble
      for even k;
    - s: U(0.005, 0.02) in fp32, rounded to bf16 (round to nearest even); the
      bf16 value is the scale.  One scale per 32 consecutive k.
* tokens, seed ``[0, config, M]``, drawn in the order x, logits (then, for the
  skewed routing, the hot-set permutation):
    - x: N(0, 1) fp32 rounded to bf16;
    - logits: N(0, 1) fp32 [M, E]; probabilities = softmax over all E; the top-k
      experts by probability (ties to the lower expert id); routing weights are
      the top-k probabilities renormalised to sum to 1 (fp32);
    - skewed routing: a hot set of ceil(0.2 E) experts (the first ids of a seeded
      permutation) gets a logit bias b found by bisection so that the hot share
      of all routing assignments is 0.50 +- 0.01.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GROUP = 32


@dataclass(frozen=True)
class MoEConfig:
    name: str
    E: int
    top_k: int
    H: int
    I: int
    Ms: tuple
    routing: str = "uniform"
    weight_seed: int = 0
    seed_id: int = 0  # stream id of the token and routing draws
    extra: dict = field(default_factory=dict)


# The five workloads, by name: tiny, K2.6-shaped decode, K2.6-shaped verify batch
# (skewed routing), K2.6-shaped prefill chunk, mid-size MoE.
WORKLOADS = {c.name: c for c in (
    MoEConfig("tiny", 8, 2, 256, 128, (16,), "uniform", 0, 0),
    MoEConfig("k26_decode", 384, 8, 7168, 2048, (1, 9, 90), "uniform", 1, 1),
    MoEConfig("k26_verify", 384, 8, 7168, 2048, (256, 512, 1024), "skewed", 1, 2),
    MoEConfig("k26_prefill", 384, 8, 7168, 2048, (8192,), "uniform", 1, 3),
    MoEConfig("mid", 64, 6, 4096, 1408, (1, 32, 128, 2048, 8192), "uniform", 4, 4),
)}


def bf16_bits_from_f32(a) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def f32_from_bf16_bits(b) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _random_nibble_bytes(rng, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return np.frombuffer(rng.bytes(n), dtype=np.uint8).reshape(shape).copy()


def _random_scales(rng, shape) -> np.ndarray:
    return bf16_bits_from_f32(rng.uniform(0.005, 0.02, size=shape).astype(np.float32))


def make_weights(E: int, H: int, I: int, seed: int) -> dict:
    """Canonical INT4 weights and bf16 scales for w13 [E, 2I, H] and w2 [E, H, I]."""
    assert H % GROUP == 0 and I % GROUP == 0
    rng = np.random.default_rng([0, seed])
    q13 = _random_nibble_bytes(rng, (E, 2 * I, H // 2))
    s13 = _random_scales(rng, (E, 2 * I, H // GROUP))
    q2 = _random_nibble_bytes(rng, (E, H, I // 2))
    s2 = _random_scales(rng, (E, H, I // GROUP))
    return {"q13": q13, "s13": s13, "q2": q2, "s2": s2}


# MXFP4 weights: E8M0 scale codes are drawn from [119, 123] (2^-8 .. 2^-4), so
# weights e2m1(q) * scale span about the same range as the INT4 ones.
MXFP4_SCALE_CODES = (119, 123)


def make_weights_mxfp4(E: int, H: int, I: int, seed: int) -> dict:
    """Canonical MXFP4 weights for w13 [E, 2I, H] and w2 [E, H, I]: E2M1 codes
    in the INT4 nibble order (uniform over the 16 codes) and E8M0 scale bytes."""
    assert H % GROUP == 0 and I % GROUP == 0
    rng = np.random.default_rng([1, seed])
    lo, hi = MXFP4_SCALE_CODES

    def scales(shape):
        return rng.integers(lo, hi + 1, size=shape, dtype=np.uint8)

    q13 = _random_nibble_bytes(rng, (E, 2 * I, H // 2))
    s13 = scales((E, 2 * I, H // GROUP))
    q2 = _random_nibble_bytes(rng, (E, H, I // 2))
    s2 = scales((E, H, I // GROUP))
    return {"q13": q13, "s13": s13, "q2": q2, "s2": s2}


def _softmax(logits: np.ndarray) -> np.ndarray:
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    return (p / p.sum(axis=1, keepdims=True)).astype(np.float32)


def _topk(p: np.ndarray, k: int):
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    top = np.take_along_axis(p, order, axis=1)
    w = (top / top.sum(axis=1, keepdims=True)).astype(np.float32)
    return order.astype(np.int32), w


def route(logits: np.ndarray, k: int):
    """Softmax over all experts, top-k, renormalised weights."""
    return _topk(_softmax(logits.astype(np.float32)), k)


def route_skewed(logits: np.ndarray, k: int, hot: np.ndarray, share=0.5, tol=0.01):
    """Bias the hot experts' logits so that they take `share` of assignments."""
    mask = np.zeros(logits.shape[1], dtype=np.float32)
    mask[hot] = 1.0

    def hot_share(b):
        ids, _ = route(logits + np.float32(b) * mask, k)
        return float(np.isin(ids, hot).mean())

    lo, hi = 0.0, 16.0
    best = (abs(hot_share(0.0) - share), 0.0)
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        s = hot_share(mid)
        best = min(best, (abs(s - share), mid))
        if abs(s - share) <= tol * 0.5:
            break
        if s < share:
            lo = mid
        else:
            hi = mid
    b = best[1]
    ids, w = route(logits + np.float32(b) * mask, k)
    return ids, w, b, hot_share(b)


def make_tokens(cfg: MoEConfig, M: int) -> dict:
    """x (bf16 bits [M, H]), topk_ids int32 [M, k], topk_weights fp32 [M, k]."""
    rng = np.random.default_rng([0, cfg.seed_id, M])
    x = bf16_bits_from_f32(rng.standard_normal((M, cfg.H), dtype=np.float32))
    logits = rng.standard_normal((M, cfg.E), dtype=np.float32)
    out = {"x": x}
    if cfg.routing == "skewed":
        perm = rng.permutation(cfg.E)
        hot = np.sort(perm[: math.ceil(0.2 * cfg.E)])
        ids, w, b, s = route_skewed(logits, cfg.top_k, hot)
        out.update(topk_ids=ids, topk_weights=w, hot=hot, bias=b, hot_share=s)
    else:
        ids, w = route(logits, cfg.top_k)
        out.update(topk_ids=ids, topk_weights=w)
    return out


def touched_experts(topk_ids, E: int) -> np.ndarray:
    ids = np.asarray(topk_ids).reshape(-1)
    ids = ids[(ids >= 0) & (ids < E)]
    return np.unique(ids)


def routing_pool(cfg: MoEConfig, M: int, n: int, base_seed: int = 1000):
    """n further independent routings of M tokens (same recipe, other seeds);
    used to rotate the touched expert set between timed calls."""
    pool = []
    for r in range(n):
        rng = np.random.default_rng([0, cfg.seed_id, M, base_seed + r])
        logits = rng.standard_normal((M, cfg.E), dtype=np.float32)
        if cfg.routing == "skewed":
            perm = rng.permutation(cfg.E)
            hot = np.sort(perm[: math.ceil(0.2 * cfg.E)])
            ids, w, _, _ = route_skewed(logits, cfg.top_k, hot)
        else:
            ids, w = route(logits, cfg.top_k)
        pool.append((ids, w))
    return pool


def router_logits_pool(cfg: MoEConfig, M: int, n: int, base_seed: int = 1000):
    """Router logits (fp32 [M, E]) behind make_tokens(cfg, M) followed by the n
    routings of routing_pool(cfg, M, n): the same draws, with the hot-expert
    bias of the skewed recipe added, so that routing them gives those routings."""
    out = []
    rng = np.random.default_rng([0, cfg.seed_id, M])
    rng.standard_normal((M, cfg.H), dtype=np.float32)  # x
    seeds = [None] + [base_seed + r for r in range(n)]
    for sd in seeds:
        if sd is not None:
            rng = np.random.default_rng([0, cfg.seed_id, M, sd])
        logits = rng.standard_normal((M, cfg.E), dtype=np.float32)
        if cfg.routing == "skewed":
            perm = rng.permutation(cfg.E)
            hot = np.sort(perm[: math.ceil(0.2 * cfg.E)])
            _, _, b, _ = route_skewed(logits, cfg.top_k, hot)
            mask = np.zeros(cfg.E, dtype=np.float32)
            mask[hot] = 1.0
            logits = logits + np.float32(b) * mask
        out.append(logits)
    return out

