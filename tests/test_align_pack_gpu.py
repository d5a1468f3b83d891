"""Align and pack on the GPU: bit-exact against the oracle / the layout spec."""
import numpy as np
import pytest

import oracle
from weight_only_int4_moe_gb300 import inputs

pytestmark = pytest.mark.gpu


def _ops():
    from weight_only_int4_moe_gb300 import ops
    return ops


ALIGN_CASES = [
    # M, k, E, block_m, seed, invalid fraction
    (16, 2, 8, 16, 0, 0.0), (1, 8, 384, 16, 1, 0.0), (9, 8, 384, 16, 2, 0.0),
    (90, 8, 384, 16, 3, 0.0), (256, 8, 384, 32, 4, 0.0), (512, 8, 384, 48, 5, 0.05),
    (1024, 8, 384, 48, 6, 0.0), (8192, 8, 384, 192, 7, 0.0), (8192, 6, 64, 192, 8, 0.01),
    (1, 1, 1, 1, 9, 0.0), (37, 3, 5, 7, 10, 0.1), (600, 8, 1024, 64, 11, 0.0),
    (700, 7, 13, 256, 12, 0.0), (0, 8, 384, 16, 13, 0.0),
]


@pytest.mark.parametrize("M,k,E,B,seed,bad", ALIGN_CASES)
def test_align_bit_exact(M, k, E, B, seed, bad):
    import torch
    ops = _ops()
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, (M, k)).astype(np.int32)
    if bad and M:
        mask = rng.random((M, k)) < bad
        ids[mask] = rng.choice([-1, E, E + 7, -100], mask.sum())
    s, e, npp, err = ops.moe_align(torch.from_numpy(ids).cuda(), E, B)
    torch.cuda.synchronize()
    n = int(npp.item())
    rs, re_, rn, rd = oracle.align(ids, E, B)
    assert n == rn
    np.testing.assert_array_equal(s[:n].cpu().numpy(), rs)
    np.testing.assert_array_equal(e[: n // B].cpu().numpy(), re_)
    flags, count = err.cpu().numpy().tolist()
    assert count == rd
    assert flags == (1 if rd else 0)


def test_align_all_tokens_one_expert():
    import torch
    ops = _ops()
    ids = np.full((3000, 2), 5, dtype=np.int32)
    s, e, npp, _ = ops.moe_align(torch.from_numpy(ids).cuda(), 8, 64)
    n = int(npp.item())
    assert n == 6016
    np.testing.assert_array_equal(s[:6000].cpu().numpy(), np.arange(6000))
    assert (s[6000:n].cpu().numpy() == 6000).all()
    assert (e[: n // 64].cpu().numpy() == 5).all()


def np_pack_reference(q, s, is_w13):
    """The packed layout written out from its definition in include/moe_int4.h."""
    E, N, K2 = q.shape
    K = 2 * K2
    nib = np.empty((E, N, K), dtype=np.uint32)
    nib[..., 0::2] = q & 0xF
    nib[..., 1::2] = q >> 4
    if is_w13:
        I = N // 2
        RT, KS = I // 128, K // 64
        rows0 = lambda r: slice(128 * r, 128 * r + 128)
        rows1 = lambda r: slice(I + 128 * r, I + 128 * r + 128)
        ks0 = lambda kk: slice(64 * kk, 64 * kk + 64)
        ks1 = ks0
    else:
        RT, KS = N // 128, K // 128
        rows0 = rows1 = lambda r: slice(128 * r, 128 * r + 128)
        ks0 = lambda kk: slice(128 * kk, 128 * kk + 64)
        ks1 = lambda kk: slice(128 * kk + 64, 128 * kk + 128)
    # scales are stored as fp16 (saturated to +-65504), two per 32-bit word
    sf = np.clip(s.astype(np.uint32).__lshift__(16).view(np.float32), -65504, 65504)
    sv = sf.astype(np.float16).view(np.uint16).astype(np.uint32)
    out_w, out_s = [], []
    for e in range(E):
        for r in range(RT):
            for kk in range(KS):
                for rows, ks in ((rows0(r), ks0(kk)), (rows1(r), ks1(kk))):
                    blk = nib[e, rows, ks]  # [128, 64]
                    words = np.zeros((128, 8), dtype=np.uint32)
                    for v in range(8):
                        for sft in range(4):
                            words[:, v] |= blk[:, 8 * v + 2 * sft] << (4 * sft)
                            words[:, v] |= blk[:, 8 * v + 2 * sft + 1] << (16 + 4 * sft)
                    slab = np.concatenate([words[:, :4].reshape(-1), words[:, 4:].reshape(-1)])
                    out_w.append(slab)
                for rows, ks in ((rows0(r), ks0(kk)), (rows1(r), ks1(kk))):
                    g0 = ks.start // 32
                    out_s.append(sv[e, rows, g0] | (sv[e, rows, g0 + 1] << 16))
    return (np.concatenate(out_w).astype("<u4").view(np.uint8),
            np.concatenate(out_s).astype("<u4").view(np.uint8))


@pytest.mark.parametrize("is_w13,E,N,K", [(1, 2, 256, 128), (0, 2, 256, 256), (1, 1, 512, 192),
                                          (0, 3, 384, 128)])
def test_pack_matches_layout_spec(is_w13, E, N, K):
    import torch
    ops = _ops()
    rng = np.random.default_rng(E * N + K + is_w13)
    q = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    # finite bf16 scales over a wide range, signs included, plus fp16 edge cases
    mag = np.exp2(rng.uniform(-20, 18, (E, N, K // 32))).astype(np.float32)
    sgn = np.where(rng.random(mag.shape) < 0.5, -1.0, 1.0).astype(np.float32)
    s = inputs.bf16_bits_from_f32(mag * sgn)
    pw, ps = ops.moe_int4_pack(torch.from_numpy(q).cuda(),
                               torch.from_numpy(s.view(np.int16)).cuda(), bool(is_w13))
    torch.cuda.synchronize()
    rw, rs = np_pack_reference(q, s, is_w13)
    np.testing.assert_array_equal(pw.cpu().numpy(), rw)
    np.testing.assert_array_equal(ps.cpu().numpy(), rs)
