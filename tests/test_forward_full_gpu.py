"""Full-size parity: the five workloads at their real sizes, in the launch
configuration the benchmark times (moe_int4_forward with its own plan), checked
against the oracle on sampled tokens (the oracle computes each token's output
one by one), plus checks that hold for every output at any size."""
import copy

import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import inputs
from helpers import assert_parity, gpu_forward

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLES = 6


def _ops():
    from weight_only_int4_moe_gb300 import ops
    return ops


@pytest.fixture(scope="module")
def k26():
    cfg = inputs.WORKLOADS["k26_decode"]
    w = inputs.make_weights(cfg.E, cfg.H, cfg.I, cfg.weight_seed)
    pw = _ops().PackedWeights(w, cfg.E, cfg.H, cfg.I, cfg.top_k)
    yield w, pw
    del pw


@pytest.fixture(scope="module")
def mid():
    cfg = inputs.WORKLOADS["mid"]
    w = inputs.make_weights(cfg.E, cfg.H, cfg.I, cfg.weight_seed)
    pw = _ops().PackedWeights(w, cfg.E, cfg.H, cfg.I, cfg.top_k)
    yield w, pw
    del pw


def _check(w, pw, cfg, M, n_samples=SAMPLES):
    t = inputs.make_tokens(cfg, M)
    got = gpu_forward(pw, t).astype(np.float64)
    assert np.all(np.isfinite(got))
    # tokens whose every slot went to experts... all tokens have k valid slots here,
    # so no output row may be identically zero
    assert np.all(np.abs(got).max(axis=1) > 0)
    rng = np.random.default_rng([M, 99])
    toks = np.sort(rng.choice(M, size=min(n_samples, M), replace=False))
    ref, _ = oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], t["topk_ids"],
                                t["topk_weights"], tokens=toks)
    return assert_parity(got[toks], ref, f"{cfg.name} M={M}")


@pytest.mark.parametrize("workload,M", [("k26_decode", 1), ("k26_decode", 9), ("k26_decode", 90),
                                        ("k26_verify", 256), ("k26_verify", 512),
                                        ("k26_verify", 1024), ("k26_prefill", 8192)])
def test_k26_workloads(k26, workload, M):
    w, pw = k26
    print(_check(w, pw, inputs.WORKLOADS[workload], M))


@pytest.mark.parametrize("M", [1, 32, 128, 2048, 8192])
def test_mid_workload(mid, M):
    w, pw = mid
    print(_check(w, pw, inputs.WORKLOADS["mid"], M, n_samples=M if M <= 32 else SAMPLES))


def _bf16_view(pw):
    """The same packed weights with bf16 output (the fp32 combine rounded to
    nearest even by the finalize kernel)."""
    ops = _ops()
    b = copy.copy(pw)
    sh = pw.shape
    b.shape = ops.Shape.of(sh.E, sh.top_k, sh.hidden, sh.inter, ops.MOE_OUT_BF16, sh.weight_format,
                           sh.flags)
    return b


@pytest.mark.parametrize("workload,M", [("k26_decode", 1), ("k26_decode", 90),
                                        ("k26_verify", 1024), ("k26_prefill", 8192)])
def test_k26_bf16_output(k26, workload, M):
    """bf16 output at full size, held to the same bound as fp32 output."""
    w, pw = k26
    print(_check(w, _bf16_view(pw), inputs.WORKLOADS[workload], M))


@pytest.mark.parametrize("M", [128, 2048])
def test_mid_bf16_output(mid, M):
    w, pw = mid
    print(_check(w, _bf16_view(pw), inputs.WORKLOADS["mid"], M))


@pytest.mark.parametrize("workload,M", [("k26_decode", 1), ("k26_decode", 9)])
def test_k26_separate_kernels(k26, workload, M):
    """The same decode calls through the separate gather / gate/up / down
    kernels (where the default plan runs the small-batch or the fused decode
    kernels)."""
    ops = _ops()
    w, pw = k26
    b = copy.copy(pw)
    sh = pw.shape
    b.shape = ops.Shape.of(sh.E, sh.top_k, sh.hidden, sh.inter, sh.out_dtype, sh.weight_format,
                           ops.MOE_FLAG_UNFUSED)
    assert ops.moe_int4_fused(M, pw.shape) or ops.moe_int4_gemv(M, pw.shape)
    assert not ops.moe_int4_fused(M, b.shape) and not ops.moe_int4_gemv(M, b.shape)
    print(_check(w, b, inputs.WORKLOADS[workload], M))


@pytest.mark.parametrize("M", [9, 64])
def test_k26_fused_decode_kernel(k26, M):
    """The fused decode kernel at the full K2.6 size (MOE_FLAG_NO_GEMV: at these
    sizes the default plan runs the small-batch kernels or the separate plan
    with the per-block down kernel)."""
    ops = _ops()
    w, pw = k26
    b = copy.copy(pw)
    sh = pw.shape
    b.shape = ops.Shape.of(sh.E, sh.top_k, sh.hidden, sh.inter, sh.out_dtype, sh.weight_format,
                           ops.MOE_FLAG_NO_GEMV)
    assert not ops.moe_int4_fused(M, pw.shape) and ops.moe_int4_fused(M, b.shape)
    print(_check(w, b, inputs.WORKLOADS["k26_decode"], M))
