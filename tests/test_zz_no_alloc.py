"""moe_align_noalloc: the align entry point for callers that cannot allocate
device memory (a plugin given only its input and output buffers, or a
latency-critical path where cudaMalloc/cudaFree may block).  Its scratch table
is a fixed 1 MiB array inside the library.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.  The GPU tests call the entry point
through the C ABI twice in a row and require the same bit-exact result as
moe_align with caller-provided scratch and as the oracle's align (index work:
no tolerance)."""
import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import ops

LIMIT = 1 << 20


def _ids(M, k, E, seed, bad=0.0):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, (M, k)).astype(np.int32)
    if bad and M:
        mask = rng.random((M, k)) < bad
        ids[mask] = rng.choice([-1, E, E + 3], mask.sum())
    return ids


def test_limit_rejected_on_host():
    """Sizes whose chunk table exceeds 1 MiB are refused before any CUDA call."""
    lib = ops.load_library()
    # E = 384, top_k = 8: 87,296 tokens = 682 chunks fit (1,047,552 B), 87,424 do not
    assert lib.moe_align_scratch_bytes(87296, 8, 384) <= LIMIT
    assert lib.moe_align_scratch_bytes(87424, 8, 384) > LIMIT
    null = None
    rc = lib.moe_align_noalloc(null, 87424, 8, 384, 16, null, null, null, null, null)
    assert rc == -7  # MOE_ERR_NOALLOC_LIMIT
    assert b"1 MiB" in lib.moe_int4_strerror(rc)
    assert lib.moe_align_noalloc(null, 4, 0, 384, 16, null, null, null, null, null) == -2


def _compare(ids, E, B, first, second):
    import torch
    s_ref, e_ref, n_ref, err_ref = ops.moe_align(torch.from_numpy(ids).cuda(), E, B)
    torch.cuda.synchronize()
    n = int(n_ref.item())
    rs, re_, rn, rd = oracle.align(ids, E, B)
    assert n == rn
    for s, e, npp, err in (first, second):
        assert int(npp.item()) == n
        assert torch.equal(s[:n], s_ref[:n])
        assert torch.equal(e[: n // B], e_ref[: n // B])
        assert torch.equal(err, err_ref)
        # and directly against the oracle's align
        np.testing.assert_array_equal(s[:n].cpu().numpy(), rs)
        np.testing.assert_array_equal(e[: n // B].cpu().numpy(), re_)
        assert err.cpu().numpy().tolist() == [1 if rd else 0, rd]


@pytest.mark.gpu
@pytest.mark.parametrize("M,k,E,B,seed,bad", [
    (1024, 8, 384, 32, 21, 0.0),     # 8 chunks of the multi-block align
    (8192, 8, 384, 128, 22, 0.01),   # 64 chunks, dropped invalid ids
    (87296, 8, 384, 128, 23, 0.0),   # the largest E = 384 routing that fits
    (90, 8, 384, 16, 24, 0.0),       # single-block align (no scratch used)
])
def test_two_calls_in_a_row_match_moe_align(M, k, E, B, seed, bad):
    import torch
    ids = torch.from_numpy(_ids(M, k, E, seed, bad)).cuda()
    first = [t.clone() for t in ops.moe_align_noalloc(ids, E, B)]
    second = ops.moe_align_noalloc(ids, E, B)
    torch.cuda.synchronize()
    _compare(ids.cpu().numpy(), E, B, first, second)


@pytest.mark.gpu
def test_shared_table_left_by_a_larger_call_is_harmless():
    """A call after a larger one (different E and chunk count) sees the array
    full of the previous call's entries and must still be exact."""
    import torch
    big = torch.from_numpy(_ids(60000, 6, 64, 31)).cuda()
    ops.moe_align_noalloc(big, 64, 64)
    ids = _ids(2000, 8, 1024, 32, 0.02)
    d = torch.from_numpy(ids).cuda()
    first = [t.clone() for t in ops.moe_align_noalloc(d, 1024, 48)]
    second = ops.moe_align_noalloc(d, 1024, 48)
    torch.cuda.synchronize()
    _compare(ids, 1024, 48, first, second)
