"""moe_int4_forward on the GPU against the oracle, element by element, at sizes
the oracle finishes in seconds (several tiles, ragged tails, every block-height
regime), plus the invariants and edge cases of the layer."""
import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import inputs
from helpers import assert_parity, gpu_forward, parity, to_device_tokens

pytestmark = pytest.mark.gpu


def _ops():
    from weight_only_int4_moe_gb300 import ops
    return ops


_cache = {}


def setup(E, k, H, I, M, seed, routing="uniform"):
    key = (E, H, I, seed)
    ops = _ops()
    if key not in _cache:
        w = inputs.make_weights(E, H, I, 500 + seed)
        _cache[key] = (w, ops.PackedWeights(w, E, H, I, k))
    w, pw = _cache[key]
    pw.shape.top_k = k
    cfg = inputs.MoEConfig("t", E, k, H, I, (M,), routing, 0, 700 + seed)
    t = inputs.make_tokens(cfg, M)
    return w, pw, t


def oracle_out(w, t, tokens=None):
    out, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], t["topk_ids"],
                                t["topk_weights"], tokens=tokens)
    return out


SMALL = [
    # E, k, H, I, M, seed  (block heights 16..192, single- and multi-block align)
    (8, 2, 256, 128, 16, 0),      # the tiny workload's shape
    (8, 2, 256, 128, 1, 1),
    (16, 4, 384, 256, 37, 2),     # ragged M, 2 gate/up tiles, 3 down tiles
    (4, 1, 256, 128, 300, 3),     # ~75 tokens per expert
    (8, 2, 512, 256, 1000, 4),    # ~250 tokens per expert -> block 192, 2 blocks
    (64, 6, 512, 256, 700, 5),    # P = 4200 -> multi-block align
    (32, 8, 1024, 384, 5, 6),     # many k stages per tile, stream-K splits
    (4, 2, 1024, 384, 300, 7),    # ~150 tokens per expert -> wide block 192, odd down k tail
    (8, 2, 256, 128, 500, 8),     # ~125 tokens per expert -> wide block 192
    (4, 2, 384, 256, 300, 11),    # wide block 192, three down row tiles
    # narrow block heights 48..112: each tensor-memory plan, scalar and float4 combines
    (16, 4, 384, 256, 64, 12),    # block 48
    (16, 4, 384, 256, 96, 13),    # block 64 (scalar combine)
    (8, 2, 256, 128, 128, 14),    # block 80
    (8, 2, 256, 128, 160, 15),    # block 96 (scalar combine)
    (8, 2, 512, 256, 192, 16),    # block 112 (scalar combine)
]


def with_flags(pw, flags):
    """The same packed weights with other forward flags (a shallow copy)."""
    import copy
    ops = _ops()
    b = copy.copy(pw)
    sh = pw.shape
    b.shape = ops.Shape.of(sh.E, sh.top_k, sh.hidden, sh.inter, sh.out_dtype, sh.weight_format,
                           flags)
    return b


@pytest.mark.parametrize("plan", ["default", "tensor", "unfused"])
@pytest.mark.parametrize("E,k,H,I,M,seed", SMALL)
def test_forward_matches_oracle(E, k, H, I, M, seed, plan):
    """Every shape through the default launch plan (the small-batch kernels or
    the fused decode kernel where they apply), the tensor-core kernels only
    (MOE_FLAG_NO_GEMV) and the separate kernels."""
    ops = _ops()
    w, pw, t = setup(E, k, H, I, M, seed)
    if plan == "tensor":
        pw = with_flags(pw, ops.MOE_FLAG_NO_GEMV)
        assert not ops.moe_int4_gemv(M, pw.shape)
    if plan == "unfused":
        pw = with_flags(pw, ops.MOE_FLAG_UNFUSED)
        assert not ops.moe_int4_fused(M, pw.shape) and not ops.moe_int4_gemv(M, pw.shape)
    got = gpu_forward(pw, t)
    ref = oracle_out(w, t)
    m = assert_parity(got, ref, f"E{E} k{k} H{H} I{I} M{M} {plan}")
    print(plan, ops.moe_int4_gemv(M, pw.shape), ops.moe_int4_fused(M, pw.shape), m)


# the small-batch kernels: ragged row-tile groups (I / 128 and H / 128 not
# multiples of 4), one to many k splits, top-1 to top-8, up to the 64-pair limit
GEMV = [
    (16, 4, 384, 256, 3, 40),     # 2 gate/up row tiles, 3 down row tiles
    (32, 8, 1280, 384, 1, 41),    # 3 gate/up tiles, 10 down tiles (ragged groups)
    (64, 8, 512, 256, 8, 42),     # 64 pairs: the limit
    (8, 1, 2048, 512, 7, 43),     # top-1
    (48, 8, 2048, 1024, 2, 44),   # 16 pairs over 170 MB of experts: the re-read rule
    (8, 2, 256, 128, 128, 46),    # 256 pairs on 8 experts (L2-resident): the pair limit
    (512, 8, 512, 256, 12, 47),   # 96 pairs over 113 MB of experts (1.09 per touched)
]


@pytest.mark.parametrize("E,k,H,I,M,seed", GEMV)
def test_small_batch_kernels_match_oracle(E, k, H, I, M, seed):
    ops = _ops()
    w, pw, t = setup(E, k, H, I, M, seed)
    assert ops.moe_int4_gemv(M, pw.shape)
    got = gpu_forward(pw, t)
    ref = oracle_out(w, t)
    print(assert_parity(got, ref, f"gemv E{E} k{k} H{H} I{I} M{M}"))


# the separate plan's per-block down step: blocks of 16 rows with about two real
# rows each, odd down row-tile counts, and skewed routing whose fullest blocks
# need two passes of eight rows
BLOCK_DOWN = [
    (384, 8, 256, 128, 90, 50, "uniform"),
    (384, 8, 384, 256, 80, 51, "uniform"),   # three down row tiles: a half CTA tile
    (384, 8, 512, 256, 120, 52, "skewed"),  # up to 12 rows on one expert
]


@pytest.mark.parametrize("E,k,H,I,M,seed,routing", BLOCK_DOWN)
def test_block_down_matches_oracle_and_tensor_path(E, k, H, I, M, seed, routing):
    ops = _ops()
    w, pw, t = setup(E, k, H, I, M, seed, routing)
    assert ops.moe_int4_block_down(M, pw.shape) and ops.moe_int4_block_m(M, pw.shape) == 16
    got = gpu_forward(pw, t)
    ref = oracle_out(w, t)
    print(assert_parity(got, ref, f"block down E{E} H{H} I{I} M{M} {routing}"))
    if routing == "skewed":  # some block holds more than eight real rows
        assert np.bincount(t["topk_ids"].ravel(), minlength=E).max() > 8
    b = gpu_forward(with_flags(pw, ops.MOE_FLAG_NO_GEMV), t)
    assert not ops.moe_int4_block_down(M, with_flags(pw, ops.MOE_FLAG_NO_GEMV).shape)
    rms = float(np.sqrt(np.mean(b.astype(np.float64) ** 2)))
    assert np.abs(got.astype(np.float64) - b).max() <= 1e-3 * rms


def test_small_batch_kernels_match_the_tensor_path_closely():
    """Both paths form the same fp16 weights and intermediates and sum exact
    products in fp32, so they differ only by summation order: far below the
    oracle bound."""
    ops = _ops()
    w, pw, t = setup(32, 8, 1024, 384, 4, 45)
    a = gpu_forward(pw, t)
    b = gpu_forward(with_flags(pw, ops.MOE_FLAG_NO_GEMV), t)
    rms = float(np.sqrt(np.mean(b.astype(np.float64) ** 2)))
    assert np.abs(a.astype(np.float64) - b).max() <= 1e-3 * rms


def test_tiny_workload_seed():
    cfg = inputs.WORKLOADS["tiny"]
    w = inputs.make_weights(cfg.E, cfg.H, cfg.I, cfg.weight_seed)
    pw = _ops().PackedWeights(w, cfg.E, cfg.H, cfg.I, cfg.top_k)
    t = inputs.make_tokens(cfg, 16)
    assert_parity(gpu_forward(pw, t), oracle_out(w, t), "tiny")


def test_skewed_routing_small():
    w, pw, t = setup(64, 8, 512, 256, 256, 7, routing="skewed")
    assert_parity(gpu_forward(pw, t), oracle_out(w, t), "skewed")


def test_all_tokens_one_expert():
    w, pw, t = setup(8, 2, 256, 128, 200, 8)
    t = dict(t)
    t["topk_ids"] = np.tile(np.array([[3, 5]], dtype=np.int32), (200, 1))
    assert_parity(gpu_forward(pw, t), oracle_out(w, t), "one expert")


def test_duplicate_expert_in_slots():
    w, pw, t = setup(8, 2, 256, 128, 16, 9)
    t = dict(t)
    ids = t["topk_ids"].copy()
    ids[:, 1] = ids[:, 0]
    t["topk_ids"] = ids
    assert_parity(gpu_forward(pw, t), oracle_out(w, t), "duplicates")


def test_top1_weight1():
    w, pw, t = setup(8, 1, 256, 128, 33, 10)
    t = dict(t, topk_weights=np.ones((33, 1), dtype=np.float32))
    assert_parity(gpu_forward(pw, t), oracle_out(w, t), "top1")


def test_invalid_ids_dropped_and_reported():
    import torch
    ops = _ops()
    w, pw, t = setup(8, 2, 256, 128, 16, 11)
    t = dict(t)
    ids = t["topk_ids"].copy()
    ids[2, 0] = 8
    ids[7, 1] = -3
    t["topk_ids"] = ids
    ws = ops.alloc_workspace(16, pw.shape)
    got = gpu_forward(pw, t, workspace=ws)
    assert_parity(got, oracle_out(w, t), "invalid ids")
    flags, count = ops.moe_int4_get_errors(ws)
    assert flags == ops.MOE_DEVERR_BAD_EXPERT_ID and count == 2
    # the report accumulates: a clean call keeps it, a second bad call adds to it
    t2 = dict(t, topk_ids=np.abs(t["topk_ids"]) % 8)
    gpu_forward(pw, t2, workspace=ws)
    assert ops.moe_int4_get_errors(ws) == (ops.MOE_DEVERR_BAD_EXPERT_ID, 2)
    gpu_forward(pw, t, workspace=ws)
    assert ops.moe_int4_get_errors(ws) == (ops.MOE_DEVERR_BAD_EXPERT_ID, 4)
    # until it is cleared
    ops.moe_int4_clear_errors(ws)
    gpu_forward(pw, t2, workspace=ws)
    assert ops.moe_int4_get_errors(ws) == (0, 0)


@pytest.mark.parametrize("plan", ["default", "tensor"])
def test_unrouted_experts_cannot_change_output(plan):
    """Random bytes in the weights and scales of the experts no pair routes to
    leave the output as it was.  The default plan here is the small-batch one,
    whose down kernel adds top_k x (k splits) fp32 partial sums per output
    element in a run-dependent order, so only the one-ulp bound applies to it;
    the tensor-core plan adds top_k terms per element and must also match
    nearly everywhere bit for bit."""
    import torch
    ops = _ops()
    E, k, H, I, M = 16, 2, 256, 128, 24
    w, pw, t = setup(E, k, H, I, M, 12)
    flags = ops.MOE_FLAG_NO_GEMV if plan == "tensor" else 0
    pw = with_flags(pw, flags)
    assert ops.moe_int4_gemv(M, pw.shape) == (plan == "default")
    base = gpu_forward(pw, t)
    used = set(np.unique(t["topk_ids"]).tolist())
    rng = np.random.default_rng(3)
    w2 = {kk: v.copy() for kk, v in w.items()}
    for e in range(E):
        if e not in used:
            for kk in w2:
                w2[kk][e] = rng.integers(0, 1 << (8 if kk[0] == "q" else 16), w2[kk][e].shape)
    pw2 = with_flags(ops.PackedWeights(w2, E, H, I, k), flags)
    again = gpu_forward(pw2, t)
    # identical up to the order of fp32 atomic additions (at most one bf16 ulp)
    ulp = np.abs(base) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(again - base) <= ulp)
    if plan == "tensor":
        assert np.mean(again == base) > 0.99


def test_zero_input_gives_zero():
    w, pw, t = setup(8, 2, 256, 128, 16, 13)
    t = dict(t, x=np.zeros_like(t["x"]))
    assert not gpu_forward(pw, t).any()


def test_m_zero_is_noop():
    import torch
    ops = _ops()
    w, pw, t = setup(8, 2, 256, 128, 16, 14)
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((0, 2), dtype=torch.int32, device="cuda")
    tw = torch.zeros((0, 2), dtype=torch.float32, device="cuda")
    out = torch.full((1, 256), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    lib = ops.load_library()
    import ctypes
    rc = lib.moe_int4_forward(x.data_ptr(), pw.w13.data_ptr(), pw.w13_scales.data_ptr(),
                              pw.w2.data_ptr(), pw.w2_scales.data_ptr(), ids.data_ptr(),
                              tw.data_ptr(), out.data_ptr(), 0, ctypes.byref(pw.shape),
                              ws.data_ptr(), 256, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert (out.float() == 7.0).all()


def test_repeated_calls_and_workspace_reuse():
    ops = _ops()
    w, pw, t = setup(16, 4, 384, 256, 37, 15)
    ws = ops.alloc_workspace(37, pw.shape)
    ref = oracle_out(w, t)
    for _ in range(3):
        assert_parity(gpu_forward(pw, t, workspace=ws), ref, "reuse")


def test_forward_host_buffers():
    import torch
    ops = _ops()
    w, pw, t = setup(16, 4, 384, 256, 37, 16)
    ws = ops.alloc_workspace(37, pw.shape, flags=ops.MOE_WS_HOST_IO)
    x = torch.from_numpy(t["x"].view(np.int16)).pin_memory()
    ids = torch.from_numpy(t["topk_ids"]).pin_memory()
    tw = torch.from_numpy(t["topk_weights"]).pin_memory()
    out = torch.empty((37, 384), dtype=torch.float32).pin_memory()
    ops.moe_int4_forward_host(x, pw.w13, pw.w13_scales, pw.w2, pw.w2_scales, ids, tw, out,
                              pw.shape, ws)
    got = out.numpy()
    assert_parity(got, oracle_out(w, t), "host io")


def test_no_timeout_flag_on_normal_runs():
    ops = _ops()
    w, pw, t = setup(32, 8, 1024, 384, 5, 6)
    ws = ops.alloc_workspace(5, pw.shape)
    gpu_forward(pw, t, workspace=ws)
    flags, _ = ops.moe_int4_get_errors(ws)
    assert not (flags & ops.MOE_DEVERR_TIMEOUT)


@pytest.mark.parametrize("E,k,H,I,M,seed", [(16, 4, 384, 256, 37, 2), (64, 6, 512, 256, 700, 5),
                                            (8, 2, 512, 256, 1000, 4)])
def test_internal_align_and_intermediate(E, k, H, I, M, seed):
    """The forward's own align buffers are bit-exact, and the gate/up GEMM's
    SwiGLU output matches the oracle's intermediate before the down GEMM."""
    import torch
    ops = _ops()
    w, pw, t = setup(E, k, H, I, M, seed)
    pw = with_flags(pw, ops.MOE_FLAG_NO_GEMV)  # the tensor-core plans' buffers
    ws = ops.alloc_workspace(M, pw.shape)
    gpu_forward(pw, t, workspace=ws)
    lay = ops.moe_int4_workspace_layout(M, pw.shape)
    BM = ops.moe_int4_block_m(M, pw.shape)
    raw = ws.cpu().numpy()
    npp = int(raw[lay["num_post_pad"]:lay["num_post_pad"] + 4].view(np.int32)[0])
    rs, re_, rn, _ = oracle.align(t["topk_ids"], E, BM)
    assert npp == rn
    got_sorted = raw[lay["sorted_ids"]:lay["sorted_ids"] + 4 * npp].view(np.int32)
    np.testing.assert_array_equal(got_sorted, rs)
    got_exp = raw[lay["expert_ids"]:lay["expert_ids"] + 4 * (npp // BM)].view(np.int32)
    np.testing.assert_array_equal(got_exp, re_)
    a = raw[lay["intermediate"]:lay["intermediate"] + 2 * npp * I].view(np.float16)
    a = a.astype(np.float32).reshape(npp, I)
    real = np.nonzero(rs < M * k)[0]
    pick = real[:: max(1, len(real) // 64)]
    ref = oracle.moe_intermediate(t["x"], w["q13"], w["s13"], t["topk_ids"], rs[pick])
    assert_parity(a[pick], ref, "intermediate")


def test_bf16_output_is_rounded_fp32_output():
    """The bf16 output is the fp32 combine rounded to nearest even (up to the
    order of fp32 atomic additions)."""
    import torch
    ops = _ops()
    w, pw, t = setup(16, 4, 384, 256, 37, 17)
    f32 = gpu_forward(pw, t)
    pw_b = ops.PackedWeights(w, 16, 384, 256, 4, out_dtype=ops.MOE_OUT_BF16)
    x, ids, tw = to_device_tokens(t)
    ws = ops.alloc_workspace(37, pw_b.shape)
    ob = pw_b.forward(x, ids, tw, workspace=ws)
    torch.cuda.synchronize()
    assert ob.dtype == torch.bfloat16
    got = ob.float().cpu().numpy()
    want = inputs.f32_from_bf16_bits(inputs.bf16_bits_from_f32(f32))
    ulp = np.abs(want) * 2.0 ** -7
    assert np.all(np.abs(got - want) <= ulp)
    assert np.mean(got == want) > 0.98
    # the bf16 output itself meets the acceptance bound
    assert_parity(got, oracle_out(w, t), "bf16 output")


@pytest.mark.parametrize("E,k,H,I,M,seed,n_tok", [
    # ~13 tokens per expert, block 32: gate/up 4 x ~130 tiles (one round-robin
    # wave, then the split part), down 8 x ~130 (several waves); every token
    (128, 8, 1024, 512, 200, 9, None),
    # ~170 tokens per expert, wide blocks of 192: ~67 blocks, down 8 row tiles
    # (two round-robin waves, then the split part); sampled tokens
    (64, 8, 1024, 512, 1360, 10, 48),
])
def test_round_robin_waves_then_split(E, k, H, I, M, seed, n_tok):
    """With at least two waves of tiles, whole waves go round-robin and the
    remainder is split by stages; both parts must give the oracle's result."""
    w, pw, t = setup(E, k, H, I, M, seed)
    BM = _ops().moe_int4_block_m(M, pw.shape)
    blocks = sum(-(-int(c) // BM) for c in np.bincount(t["topk_ids"].ravel(), minlength=E) if c)
    assert blocks * (H // 128) >= 2 * 152  # the down GEMM has round-robin waves on GB300
    got = gpu_forward(pw, t)
    toks = None
    if n_tok is not None:
        toks = np.sort(np.random.default_rng(seed).choice(M, size=n_tok, replace=False))
    ref = oracle_out(w, t, tokens=toks)
    m = assert_parity(got if toks is None else got[toks], ref, f"E{E} M{M}")
    print(BM, blocks, m)
