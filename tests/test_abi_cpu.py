"""The C-ABI library builds, loads and exports every declared entry point; host
logic that needs no GPU (sizes, policy, argument checks) behaves as declared."""
import ctypes
import os
import re

import pytest

from weight_only_int4_moe_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_int4.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("moe_int4_pack", "moe_align", "moe_int4_forward"):
        assert required in names
    assert set(names) == set(ops.EXPORTED)


def test_header_constants_match_the_binding():
    """The device error flags, output types and weight formats of the header
    are the values the Python binding uses."""
    text = open(HEADER).read()
    defs = dict(re.findall(r"^#define\s+(MOE_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|\d+)u?\b", text,
                           flags=re.M))
    for name in ("MOE_DEVERR_BAD_EXPERT_ID", "MOE_DEVERR_TIMEOUT", "MOE_DEVERR_BOUNDS",
                 "MOE_DEVERR_RANGE", "MOE_OUT_BF16", "MOE_OUT_F32", "MOE_W_INT4", "MOE_W_MXFP4",
                 "MOE_WS_HOST_IO", "MOE_FLAG_UNFUSED", "MOE_FLAG_NO_GEMV"):
        assert int(defs[name], 0) == getattr(ops, name), name
    flags = [int(v, 0) for k, v in defs.items() if k.startswith("MOE_DEVERR_")]
    assert all(f & (f - 1) == 0 for f in flags) and len(set(flags)) == len(flags)


def test_library_exports_every_declared_symbol():
    lib = ops.load_library()
    assert os.path.exists(ops.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_sizes_and_policy():
    assert ops.moe_int4_packed_bytes(384, 4096, 7168) == 384 * 4096 * 3584
    assert ops.moe_int4_packed_scale_bytes(384, 4096, 7168) == 384 * 4096 * 224 * 2
    # the pages' ~8.5 GB per layer for 384 experts (int4 bytes only)
    gb = (ops.moe_int4_packed_bytes(384, 4096, 7168) + ops.moe_int4_packed_bytes(384, 7168, 2048)) / 1e9
    assert abs(gb - 8.456) < 0.01
    assert ops.moe_align_capacity(1, 8, 384, 16) == 8 + 8 * 15
    assert ops.moe_align_capacity(10, 8, 4, 16) == 80 + 4 * 15
    sh = ops.Shape.of(384, 8, 7168, 2048)
    assert ops.moe_int4_block_m(1, sh) == 16
    assert ops.moe_int4_block_m(8192, sh) == 192  # ~170 tokens per expert: one wide block
    # 2 x mean + 8: the verify batches' busier experts (skewed routing, ~2.5x the
    # mean) fit one block
    assert [ops.moe_int4_block_m(M, sh) for M in (90, 256, 512, 1024)] == [16, 32, 32, 64]
    mid = ops.Shape.of(64, 6, 4096, 1408)
    # ~192 tokens per expert: two blocks per expert whether 128 or 192 rows high,
    # so the 128-row kernel; ~768: five wide blocks instead of seven
    assert ops.moe_int4_block_m(2048, mid) == 128
    assert ops.moe_int4_block_m(8192, mid) == 192
    for M in range(1, 20000, 37):  # a wide block only where it saves a pass
        bm = ops.moe_int4_block_m(M, mid)
        if bm > 128:
            n = M * 6 / 64 * 1.05
            assert -(-n // 192) < -(-n // 128)
    for M in (1, 9, 90, 256, 1024, 8192):
        bm = ops.moe_int4_block_m(M, sh)
        assert 16 <= bm <= 192 and bm % 16 == 0
        assert ops.moe_int4_workspace_bytes(M, sh, 0) > M * 7168 * 4
        assert ops.moe_int4_workspace_bytes(M, sh, ops.MOE_WS_HOST_IO) > ops.moe_int4_workspace_bytes(M, sh, 0)
    assert ops.moe_align_scratch_bytes(512, 8, 384) == 0
    assert ops.moe_align_scratch_bytes(8192, 8, 384) == 64 * 384 * 4


def test_bad_out_dtype_rejected():
    lib = ops.load_library()
    sh = ops.Shape(8, 2, 256, 128, 32, 7)
    assert lib.moe_int4_workspace_bytes(4, ctypes.byref(sh), 0) == 0


def test_fp32_output_needs_no_accumulator_workspace():
    f = ops.moe_int4_workspace_bytes(4096, ops.Shape.of(64, 6, 4096, 1408, ops.MOE_OUT_F32))
    b = ops.moe_int4_workspace_bytes(4096, ops.Shape.of(64, 6, 4096, 1408, ops.MOE_OUT_BF16))
    assert b - f >= 4096 * 4096 * 4


@pytest.mark.parametrize("E,k,H,I,grp", [(0, 1, 128, 128, 32), (8, 9, 128, 128, 32),
                                         (8, 2, 192, 128, 32), (8, 2, 128, 64, 32),
                                         (8, 2, 128, 128, 64), (2000, 2, 128, 128, 32)])
def test_bad_shapes_rejected_on_host(E, k, H, I, grp):
    lib = ops.load_library()
    sh = ops.Shape(E, k, H, I, grp, 0)
    assert lib.moe_int4_workspace_bytes(4, ctypes.byref(sh), 0) == 0
    one = ctypes.c_void_p(16)
    rc = lib.moe_int4_forward(one, one, one, one, one, one, one, one, 4, ctypes.byref(sh), one,
                              1 << 30, None)
    assert rc == -2  # MOE_ERR_SHAPE


def test_null_and_alignment_rejected_on_host():
    lib = ops.load_library()
    sh = ops.Shape.of(8, 2, 256, 128)
    good = ctypes.c_void_p(1 << 20)
    rc = lib.moe_int4_forward(None, good, good, good, good, good, good, good, 4, ctypes.byref(sh),
                              good, 1 << 30, None)
    assert rc == -1
    bad = ctypes.c_void_p((1 << 20) + 4)
    rc = lib.moe_int4_forward(good, good, good, good, good, good, good, bad, 4, ctypes.byref(sh),
                              good, 1 << 30, None)
    assert rc == -3
    rc = lib.moe_int4_forward(good, good, good, good, good, good, good, good, 4, ctypes.byref(sh),
                              good, 16, None)
    assert rc == -4
    # M == 0 is a no-op that touches nothing
    rc = lib.moe_int4_forward(None, None, None, None, None, None, None, None, 0, ctypes.byref(sh),
                              None, 0, None)
    assert rc == 0
    assert lib.moe_int4_pack(None, good, 1, 256, 64, 1, good, good, None, None) == -1
    assert lib.moe_int4_pack(good, good, 1, 128, 64, 1, good, good, None, None) == -2
    assert lib.moe_int4_pack(good, good, 1, 128, 64, 0, good, good, None, None) == -2
    assert ops.moe_int4_strerror(-4) == "workspace too small"


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe_int4.h"

int main(void) {
    moe_int4_shape sh;
    memset(&sh, 0, sizeof sh);
    sh.E = 384; sh.top_k = 8; sh.hidden = 7168; sh.inter = 2048; sh.group = 32;
    sh.out_dtype = MOE_OUT_F32;
    printf("%zu\n", moe_int4_packed_bytes(384, 4096, 7168));
    printf("%zu\n", moe_int4_workspace_bytes(90, &sh, 0));
    printf("%d\n", moe_int4_block_m(90, &sh));
    printf("%zu\n", moe_align_capacity(90, 8, 384, 16));
    printf("%d\n", moe_int4_forward(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, &sh,
                                    NULL, 0, NULL));
    sh.hidden = 7200;
    printf("%zu\n", moe_int4_workspace_bytes(90, &sh, 0));
    printf("%s\n", moe_int4_strerror(MOE_ERR_SHAPE));
    return 0;
}
"""


def test_header_is_plain_c_and_the_library_links_from_c(tmp_path):
    """The boundary is a C ABI: a C11 program (pedantic, warnings as errors)
    includes the header, links the library and calls its host-side entry points,
    which agree with the Python binding."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    ops.load_library()
    lib = ops.library_path()
    src = tmp_path / "use_abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_abi"
    r = subprocess.run([gcc, "-std=c11", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-I", os.path.join(ROOT, "include"), str(src), lib,
                        "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    sh = ops.Shape.of(384, 8, 7168, 2048)
    assert int(out[0]) == ops.moe_int4_packed_bytes(384, 4096, 7168)
    assert int(out[1]) == ops.moe_int4_workspace_bytes(90, sh)
    assert int(out[2]) == ops.moe_int4_block_m(90, sh) == 16
    assert int(out[3]) == ops.moe_align_capacity(90, 8, 384, 16) == 720 + 384 * 15
    assert int(out[4]) == 0          # M == 0: a no-op
    assert int(out[5]) == 0          # a rejected shape needs no workspace
    assert out[6] == ops.moe_int4_strerror(-2)


def test_ep_row_kernels_check_arguments_on_the_host():
    """moe_ep_gather / moe_ep_combine reject bad arguments before any launch
    (no GPU needed) and treat n = 0 as a no-op."""
    lib = ops.load_library()
    s = None
    err_null, err_shape, err_align = -1, -2, -3  # MOE_ERR_NULL, _SHAPE, _ALIGN
    assert lib.moe_ep_gather(None, 4, None, 0, 64, None, None, s) == ops.MOE_OK
    assert lib.moe_ep_combine(None, None, 0, 64, None, 4, None, s) == ops.MOE_OK
    fake = ctypes.c_void_p(16)  # never dereferenced: the checks fail first
    assert lib.moe_ep_gather(None, 4, fake, 3, 64, fake, None, s) == err_null
    assert lib.moe_ep_gather(fake, 4, fake, 3, 60, fake, None, s) == err_shape
    assert lib.moe_ep_gather(fake, 4, fake, -1, 64, fake, None, s) == err_shape
    assert lib.moe_ep_gather(ctypes.c_void_p(24), 4, fake, 3, 64, fake, None, s) == err_align
    assert lib.moe_ep_combine(fake, None, 3, 64, fake, 4, None, s) == err_null
    assert lib.moe_ep_combine(fake, fake, 3, 66, fake, 4, None, s) == err_shape
    assert lib.moe_ep_combine(fake, fake, 3, 64, ctypes.c_void_p(40), 4, None, s) == err_align


def test_launch_plans():
    """Which forwards run which plan (host logic; the measured crossovers): the
    small-batch kernels up to 128 pairs and 1.2 pairs per expected touched
    expert, or up to 256 pairs when all experts fit in half the L2; the fused
    decode kernel up to 512 pairs in blocks of up to 128 rows; the separate
    kernels beyond."""
    k26 = ops.Shape.of(384, 8, 7168, 2048)
    Ms = (1, 8, 9, 16, 17, 64, 65, 90, 1024)
    # 8 of 384 experts per token: 128 pairs touch about 109.7 experts (1.17 per)
    assert [ops.moe_int4_gemv(M, k26) for M in Ms] == [True] * 4 + [False] * 5
    # the fused decode kernel gives way to the separate plan with the per-block
    # down kernel where blocks hold at most 2.5 rows per expected touched expert
    assert not any(ops.moe_int4_fused(M, k26) for M in Ms)
    assert [ops.moe_int4_block_down(M, k26) for M in Ms] == [False] * 4 + [True] * 4 + [False]
    mid = ops.Shape.of(64, 6, 4096, 1408)
    # M = 4: 24 pairs on about 20.8 experts (1.15); M = 5: 30 on 24.9 (1.20+)
    assert [ops.moe_int4_gemv(M, mid) for M in (1, 4, 5, 32)] == [True, True, False, False]
    assert [ops.moe_int4_fused(M, mid) for M in (1, 32, 128, 2048, 8192)] == [False, True, False,
                                                                              False, False]
    # mid-size M = 16: 96 pairs on about 50.8 experts (1.89); M = 32: 3.13
    assert [ops.moe_int4_block_down(M, mid) for M in (5, 16, 32)] == [True, True, False]
    no_gemv = ops.Shape.of(64, 6, 4096, 1408, flags=ops.MOE_FLAG_NO_GEMV)
    assert ops.moe_int4_fused(1, no_gemv) and not ops.moe_int4_gemv(1, no_gemv)
    tiny = ops.Shape.of(8, 2, 256, 128)  # 8 experts of 55 KB: L2-resident
    assert ops.moe_int4_gemv(128, tiny) and not ops.moe_int4_gemv(129, tiny)  # 256 pairs
    assert ops.moe_int4_fused(129, tiny)
    assert ops.moe_int4_fused(64, ops.Shape.of(64, 8, 256, 128))  # 512 pairs, block 32
    assert not ops.moe_int4_fused(512, ops.Shape.of(3, 1, 256, 128))  # 512 pairs, block 192
    unfused = ops.Shape.of(384, 8, 7168, 2048, flags=ops.MOE_FLAG_UNFUSED)
    assert not ops.moe_int4_fused(1, unfused) and not ops.moe_int4_gemv(1, unfused)
    # the per-block down kernel at 16-row blocks only, and never under either flag
    assert not ops.moe_int4_block_down(256, k26)
    assert not ops.moe_int4_block_down(90, unfused)
    k26_tc = ops.Shape.of(384, 8, 7168, 2048, flags=ops.MOE_FLAG_NO_GEMV)
    assert not ops.moe_int4_block_down(90, k26_tc)
    assert [ops.moe_int4_fused(M, k26_tc) for M in (1, 9, 64, 65)] == [True, True, True, False]
