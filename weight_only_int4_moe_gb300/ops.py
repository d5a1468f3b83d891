"""Thin Python binding of the C ABI in ``include/moe_int4.h``.

Argument marshalling only: every step of the layer runs in the CUDA library.
PyTorch provides device memory and the current CUDA stream.  If the library is
missing and cannot be built, or the device is not an sm_103 GPU, calls raise --
there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build

MOE_OK = 0
MOE_WS_HOST_IO = 0x1
MOE_OUT_BF16 = 0
MOE_OUT_F32 = 1
MOE_DEVERR_BAD_EXPERT_ID = 0x1
MOE_DEVERR_TIMEOUT = 0x2
MOE_DEVERR_BOUNDS = 0x4  # debug-bounds builds only
MOE_DEVERR_RANGE = 0x8
MOE_W_INT4 = 0
MOE_W_MXFP4 = 1
MOE_FLAG_UNFUSED = 0x1
MOE_FLAG_NO_GEMV = 0x2

EXPORTED = [
    "moe_int4_packed_bytes", "moe_int4_packed_scale_bytes", "moe_int4_pack", "moe_mxfp4_pack",
    "moe_align_capacity", "moe_align_scratch_bytes", "moe_align",
    "moe_int4_workspace_bytes", "moe_int4_block_m", "moe_int4_fused", "moe_int4_gemv",
    "moe_int4_block_down",
    "moe_int4_workspace_layout",
    "moe_int4_forward",
    "moe_int4_forward_host", "moe_int4_get_errors", "moe_int4_clear_errors",
    "moe_int4_strerror", "moe_int4_profile_enable", "moe_int4_profile_read",
    "moe_int4_last_launch_count", "moe_align_noalloc", "moe_route", "moe_int4_forward_routed",
    "moe_ep_gather", "moe_ep_combine",
]


class Shape(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("top_k", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("group", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("weight_format", ctypes.c_int32),
                ("flags", ctypes.c_int32)]

    @classmethod
    def of(cls, E, top_k, hidden, inter, out_dtype=MOE_OUT_F32, weight_format=0, flags=0):
        return cls(E, top_k, hidden, inter, 32, out_dtype, weight_format, flags)

    @property
    def torch_out_dtype(self):
        return torch.float32 if self.out_dtype == MOE_OUT_F32 else torch.bfloat16


_lib = None
_lock = threading.Lock()


def debug_bounds() -> bool:
    """MOE_INT4_DEBUG_BOUNDS=1 selects the debug-bounds build of the library
    (index checks on routing buffers, MOE_DEVERR_BOUNDS); read once, when the
    library is first loaded."""
    return os.environ.get("MOE_INT4_DEBUG_BOUNDS", "0") == "1"


def library_path() -> str:
    return _build.DEBUG_LIB if debug_bounds() else _build.LIB


def load_library(build_if_missing: bool = True):
    """Load (building first if needed) the CUDA library and declare signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        dbg = debug_bounds()
        path = _build.build(debug_bounds=dbg) if build_if_missing else library_path()
        lib = ctypes.CDLL(path)
        p, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sp = ctypes.POINTER(Shape)
        sig = {
            "moe_int4_packed_bytes": ([i, i, i], sz),
            "moe_int4_packed_scale_bytes": ([i, i, i], sz),
            "moe_int4_pack": ([p, p, i, i, i, i, p, p, p, p], i),
            "moe_mxfp4_pack": ([p, p, i, i, i, i, p, p, p, p], i),
            "moe_align_capacity": ([i, i, i, i], sz),
            "moe_align_scratch_bytes": ([i, i, i], sz),
            "moe_align": ([p, i, i, i, i, p, p, p, p, p, sz, p], i),
            "moe_int4_workspace_bytes": ([i, sp, i], sz),
            "moe_int4_fused": ([i, sp], i),
            "moe_int4_gemv": ([i, sp], i),
            "moe_int4_block_down": ([i, sp], i),
            "moe_int4_block_m": ([i, sp], i),
            "moe_int4_workspace_layout": ([i, sp, p], i),
            "moe_int4_forward": ([p] * 8 + [i, sp, p, sz, p], i),
            "moe_int4_forward_host": ([p] * 8 + [i, sp, p, sz, p], i),
            "moe_int4_get_errors": ([p, p, p, p], i),
            "moe_int4_clear_errors": ([p, p], i),
            "moe_int4_strerror": ([i], ctypes.c_char_p),
            "moe_int4_profile_enable": ([i], i),
            "moe_int4_profile_read": ([p], i),
            "moe_int4_last_launch_count": ([], i),
            "moe_align_noalloc": ([p, i, i, i, i, p, p, p, p, p], i),
            "moe_route": ([p, i, i, i, p, p, p], i),
            "moe_int4_forward_routed": ([p] * 9 + [i, sp, p, sz, p], i),
            "moe_ep_gather": ([p, i, p, i, i, p, p, p], i),
            "moe_ep_combine": ([p, p, i, i, p, i, p, p], i),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != MOE_OK:
        msg = load_library().moe_int4_strerror(rc).decode()
        raise RuntimeError(f"{what} failed ({rc}): {msg}")


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dptr(t: torch.Tensor) -> int:
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _on(*tensors):
    """Context in which a library call runs: the device that holds the call's
    device tensors, made current (the library launches on the current device
    and the current stream belongs to it).  All of them must be on one device."""
    devs = {t.device for t in tensors if isinstance(t, torch.Tensor) and t.is_cuda}
    if len(devs) != 1:
        raise ValueError(f"expected the tensors on one CUDA device, got {sorted(map(str, devs))}")
    return torch.cuda.device(devs.pop())


def _u16(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensors are passed by bit pattern."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype in (torch.int16, torch.uint16):
        return t
    raise TypeError(f"expected bf16 (or its int16 bits), got {t.dtype}")


# ----------------------------------------------------------------- packing --
def moe_int4_packed_bytes(E: int, N: int, K: int) -> int:
    return load_library().moe_int4_packed_bytes(E, N, K)


def moe_int4_packed_scale_bytes(E: int, N: int, K: int) -> int:
    return load_library().moe_int4_packed_scale_bytes(E, N, K)


def moe_int4_pack(q: torch.Tensor, scales: torch.Tensor, is_w13: bool, stream=None,
                  inexact: torch.Tensor | None = None):
    """Canonical INT4 (uint8 [E, N, K/2]) + bf16 scales [E, N, K/32] -> packed
    (uint8) and packed scales (uint8) device tensors.  ``inexact`` (optional
    device int32 [1]) counts the scales whose dequantised weights are not exact
    in fp16 (non-zero magnitudes outside [2^-14, 8188])."""
    lib = load_library()
    E, N, K2 = q.shape
    K = 2 * K2
    packed = torch.empty(lib.moe_int4_packed_bytes(E, N, K), dtype=torch.uint8, device=q.device)
    pscales = torch.empty(lib.moe_int4_packed_scale_bytes(E, N, K), dtype=torch.uint8,
                          device=q.device)
    with _on(q, scales, packed, pscales, inexact):
        rc = lib.moe_int4_pack(_dptr(q), _dptr(_u16(scales)), E, N, K, int(bool(is_w13)),
                               _dptr(packed), _dptr(pscales),
                               None if inexact is None else _dptr(inexact), _stream(stream))
    _check(rc, "moe_int4_pack")
    return packed, pscales


def moe_mxfp4_pack(q: torch.Tensor, scales: torch.Tensor, is_w13: bool, stream=None):
    """Canonical MXFP4 (E2M1 codes, uint8 [E, N, K/2]) + E8M0 scales (uint8
    [E, N, K/32]) -> packed (uint8) and packed scales (uint8) device tensors,
    plus the device count of scales clamped to the supported range (int32 [1])."""
    lib = load_library()
    E, N, K2 = q.shape
    K = 2 * K2
    packed = torch.empty(lib.moe_int4_packed_bytes(E, N, K), dtype=torch.uint8, device=q.device)
    pscales = torch.empty(lib.moe_int4_packed_scale_bytes(E, N, K), dtype=torch.uint8,
                          device=q.device)
    bad = torch.zeros(1, dtype=torch.int32, device=q.device)
    with _on(q, scales, packed, pscales, bad):
        rc = lib.moe_mxfp4_pack(_dptr(q), _dptr(scales.contiguous()), E, N, K,
                                int(bool(is_w13)), _dptr(packed), _dptr(pscales), _dptr(bad),
                                _stream(stream))
    _check(rc, "moe_mxfp4_pack")
    return packed, pscales, bad


# ------------------------------------------------------------------- align --
def moe_align_capacity(M: int, top_k: int, E: int, block_m: int) -> int:
    return load_library().moe_align_capacity(M, top_k, E, block_m)


def moe_align_scratch_bytes(M: int, top_k: int, E: int) -> int:
    return load_library().moe_align_scratch_bytes(M, top_k, E)


def moe_align(topk_ids: torch.Tensor, E: int, block_m: int, stream=None):
    """Returns (sorted_ids, expert_ids, num_post_pad, err) device tensors; only
    the first num_post_pad entries of sorted_ids are defined."""
    lib = load_library()
    M, k = topk_ids.shape
    cap = max(lib.moe_align_capacity(M, k, E, block_m), 1)
    dev = topk_ids.device
    sorted_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    expert_ids = torch.empty(cap // block_m + 1, dtype=torch.int32, device=dev)
    npp = torch.zeros(1, dtype=torch.int32, device=dev)
    err = torch.zeros(2, dtype=torch.int32, device=dev)
    scratch_bytes = lib.moe_align_scratch_bytes(M, k, E)
    scratch = torch.empty(max(scratch_bytes, 16), dtype=torch.uint8, device=dev)
    with _on(topk_ids, sorted_ids, expert_ids, npp, err, scratch):
        rc = lib.moe_align(_dptr(topk_ids), M, k, E, block_m, _dptr(sorted_ids),
                           _dptr(expert_ids), _dptr(npp), _dptr(err), _dptr(scratch),
                           scratch_bytes, _stream(stream))
    _check(rc, "moe_align")
    return sorted_ids, expert_ids, npp, err


def moe_align_noalloc(topk_ids: torch.Tensor, E: int, block_m: int, out=None, stream=None):
    """moe_align without caller scratch: the library's fixed device table is
    used instead (limit: moe_align_scratch_bytes <= 1 MiB).  ``out`` may give
    preallocated (sorted_ids, expert_ids, num_post_pad, err) buffers, so that
    the call itself allocates nothing; otherwise they are created here."""
    lib = load_library()
    M, k = topk_ids.shape
    if out is None:
        cap = max(lib.moe_align_capacity(M, k, E, block_m), 1)
        dev = topk_ids.device
        out = (torch.empty(cap, dtype=torch.int32, device=dev),
               torch.empty(cap // block_m + 1, dtype=torch.int32, device=dev),
               torch.zeros(1, dtype=torch.int32, device=dev),
               torch.zeros(2, dtype=torch.int32, device=dev))
    sorted_ids, expert_ids, npp, err = out
    # the library looks up its table on the current device: make it the ids'
    with _on(topk_ids, sorted_ids, expert_ids, npp, err):
        rc = lib.moe_align_noalloc(_dptr(topk_ids), M, k, E, block_m, _dptr(sorted_ids),
                                   _dptr(expert_ids), _dptr(npp), _dptr(err), _stream(stream))
    _check(rc, "moe_align_noalloc")
    return sorted_ids, expert_ids, npp, err


# ----------------------------------------------------------------- forward --
def moe_int4_workspace_bytes(M: int, shape: Shape, flags: int = 0) -> int:
    return load_library().moe_int4_workspace_bytes(M, ctypes.byref(shape), flags)


def moe_int4_fused(M: int, shape: Shape) -> bool:
    """Whether a forward of M tokens runs the fused decode kernel (the gather
    and both GEMMs in one launch)."""
    return load_library().moe_int4_fused(M, ctypes.byref(shape)) == 1


def moe_int4_block_down(M: int, shape: Shape) -> bool:
    """Whether a forward of M tokens runs the separate plan's down step as
    per-block matrix-vector work."""
    return load_library().moe_int4_block_down(M, ctypes.byref(shape)) == 1


def moe_int4_gemv(M: int, shape: Shape) -> bool:
    """Whether a forward of M tokens runs the small-batch matrix-vector kernels
    (a few tokens: the expert MLP on the CUDA cores, no align)."""
    return load_library().moe_int4_gemv(M, ctypes.byref(shape)) == 1


def moe_int4_block_m(M: int, shape: Shape) -> int:
    return load_library().moe_int4_block_m(M, ctypes.byref(shape))


def moe_int4_workspace_layout(M: int, shape: Shape) -> dict:
    off = (ctypes.c_size_t * 6)()
    _check(load_library().moe_int4_workspace_layout(M, ctypes.byref(shape), off),
           "moe_int4_workspace_layout")
    keys = ["err", "num_post_pad", "sorted_ids", "expert_ids", "intermediate", "acc"]
    return dict(zip(keys, list(off)))


def alloc_workspace(M: int, shape: Shape, flags: int = 0, device="cuda") -> torch.Tensor:
    """A workspace for forwards of up to M tokens, its error words cleared
    (they accumulate over calls until moe_int4_clear_errors)."""
    n = moe_int4_workspace_bytes(M, shape, flags)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def moe_int4_forward(x, w13_packed, w13_scales, w2_packed, w2_scales, topk_ids, topk_weights,
                     shape: Shape, out=None, workspace=None, stream=None):
    """out [M, H] (fp32 or bf16 per shape.out_dtype) = the MoE expert MLP."""
    lib = load_library()
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, shape.hidden), dtype=shape.torch_out_dtype, device=x.device)
    if out.dtype != shape.torch_out_dtype:
        raise TypeError(f"out must be {shape.torch_out_dtype}")
    if workspace is None:
        workspace = alloc_workspace(M, shape, device=x.device)
    with _on(x, w13_packed, w13_scales, w2_packed, w2_scales, topk_ids, topk_weights, out,
             workspace):
        rc = lib.moe_int4_forward(
            _dptr(_u16(x)), _dptr(w13_packed), _dptr(w13_scales), _dptr(w2_packed),
            _dptr(w2_scales), _dptr(topk_ids), _dptr(topk_weights), _dptr(out), M,
            ctypes.byref(shape), _dptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "moe_int4_forward")
    return out


def moe_route(router_logits: torch.Tensor, top_k: int, stream=None):
    """(topk_ids int32 [M, k], topk_weights fp32 [M, k]) from fp32 logits [M, E]."""
    M, E = router_logits.shape
    dev = router_logits.device
    ids = torch.empty((M, top_k), dtype=torch.int32, device=dev)
    w = torch.empty((M, top_k), dtype=torch.float32, device=dev)
    with _on(router_logits, ids, w):
        _check(load_library().moe_route(_dptr(router_logits), M, E, top_k, _dptr(ids), _dptr(w),
                                        _stream(stream)), "moe_route")
    return ids, w


def moe_ep_gather(src: torch.Tensor, rows: torch.Tensor, out=None, bad=None, stream=None):
    """out[i] = src[rows[i]] for a 2-byte [R, H] tensor and int32 row indices
    (expert-parallel dispatch).  bad: optional device uint32 word, bit 0 set for
    an index outside [0, R) (that row of out is zeroed)."""
    if src.element_size() != 2 or src.dim() != 2:
        raise ValueError("moe_ep_gather: expected a 2-D tensor of 2-byte elements")
    src = src.contiguous()
    rows = rows.to(torch.int32).contiguous()
    n, H = rows.numel(), src.shape[1]
    if out is None:
        out = torch.empty((n, H), dtype=src.dtype, device=src.device)
    with _on(src, rows, out):
        _check(load_library().moe_ep_gather(_dptr(src), src.shape[0], _dptr(rows) if n else None,
                                            n, H, _dptr(out) if n else None,
                                            _dptr(bad) if bad is not None else None,
                                            _stream(stream)), "moe_ep_gather")
    return out


def moe_ep_combine(src: torch.Tensor, rows: torch.Tensor, out: torch.Tensor, bad=None,
                   stream=None):
    """out[rows[i]] += src[i] for fp32 [n, H] rows (expert-parallel combine);
    rows may repeat.  bad: optional device uint32 word, bit 0 set for an index
    outside [0, out rows) (that row is dropped)."""
    if src.dtype != torch.float32 or out.dtype != torch.float32:
        raise ValueError("moe_ep_combine: expected fp32 rows")
    src = src.contiguous()
    rows = rows.to(torch.int32).contiguous()
    n, H = rows.numel(), out.shape[1]
    if n and tuple(src.shape) != (n, H):
        raise ValueError("moe_ep_combine: src must be [len(rows), H]")
    if not out.is_contiguous():
        raise ValueError("moe_ep_combine: out must be contiguous")
    with _on(src, rows, out):
        _check(load_library().moe_ep_combine(_dptr(src) if n else None,
                                             _dptr(rows) if n else None, n, H, _dptr(out),
                                             out.shape[0],
                                             _dptr(bad) if bad is not None else None,
                                             _stream(stream)), "moe_ep_combine")
    return out


def moe_int4_forward_routed(x, w13, w13_scales, w2, w2_scales, router_logits, shape: Shape,
                            out=None, topk_ids=None, topk_weights=None, workspace=None,
                            stream=None):
    """moe_int4_forward with the routing computed from fp32 router logits [M, E].
    Returns (out, topk_ids, topk_weights)."""
    M = x.shape[0]
    dev = x.device
    if out is None:
        out = torch.empty((M, shape.hidden), dtype=shape.torch_out_dtype, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((M, shape.top_k), dtype=torch.int32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((M, shape.top_k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(M, shape, device=dev)
    with _on(x, w13, w13_scales, w2, w2_scales, router_logits, topk_ids, topk_weights, out,
             workspace):
        rc = load_library().moe_int4_forward_routed(
            _dptr(x), _dptr(w13), _dptr(w13_scales), _dptr(w2), _dptr(w2_scales),
            _dptr(router_logits), _dptr(topk_ids), _dptr(topk_weights), _dptr(out), M,
            ctypes.byref(shape), _dptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "moe_int4_forward_routed")
    return out, topk_ids, topk_weights


def moe_int4_forward_host(x_host, w13_packed, w13_scales, w2_packed, w2_scales, ids_host,
                          weights_host, out_host, shape: Shape, workspace, stream=None):
    """Host-buffer variant: x/ids/weights/out are CPU tensors (pinned for async
    copies); the call returns once out_host holds the result."""
    lib = load_library()
    for t in (x_host, ids_host, weights_host, out_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors")
    M = x_host.shape[0]
    with _on(w13_packed, w13_scales, w2_packed, w2_scales, workspace):
        rc = lib.moe_int4_forward_host(
            _u16(x_host).data_ptr(), _dptr(w13_packed), _dptr(w13_scales), _dptr(w2_packed),
            _dptr(w2_scales), ids_host.data_ptr(), weights_host.data_ptr(),
            out_host.data_ptr(), M, ctypes.byref(shape), _dptr(workspace), workspace.numel(),
            _stream(stream))
    _check(rc, "moe_int4_forward_host")
    return out_host


def moe_int4_get_errors(workspace, stream=None):
    lib = load_library()
    flags = ctypes.c_uint32(0)
    count = ctypes.c_uint32(0)
    with _on(workspace):
        rc = lib.moe_int4_get_errors(_dptr(workspace), ctypes.byref(flags), ctypes.byref(count),
                                     _stream(stream))
    _check(rc, "moe_int4_get_errors")
    return flags.value, count.value


def moe_int4_clear_errors(workspace, stream=None):
    with _on(workspace):
        _check(load_library().moe_int4_clear_errors(_dptr(workspace), _stream(stream)),
               "moe_int4_clear_errors")


def moe_int4_strerror(code: int) -> str:
    return load_library().moe_int4_strerror(code).decode()


def moe_int4_profile_enable(on: bool):
    _check(load_library().moe_int4_profile_enable(int(bool(on))), "moe_int4_profile_enable")


def moe_int4_profile_read():
    ms = (ctypes.c_float * 4)()
    _check(load_library().moe_int4_profile_read(ms), "moe_int4_profile_read")
    return list(ms)


def moe_int4_last_launch_count() -> int:
    return load_library().moe_int4_last_launch_count()


# --------------------------------------------------------------- helpers --
class PackedWeights:
    """Device copies of one weight set in the kernels' packed layout.  fmt "int4":
    w holds q13/q2 nibble bytes and bf16 scales s13/s2; "mxfp4": E2M1 codes and
    E8M0 scale bytes (the weights' canonical forms in inputs.make_weights*).
    An MXFP4 set with a scale outside the supported range raises."""

    def __init__(self, w: dict, E: int, H: int, I: int, top_k: int, device="cuda",
                 keep_canonical: bool = False, out_dtype: int = MOE_OUT_F32, fmt: str = "int4"):
        if fmt not in ("int4", "mxfp4"):
            raise ValueError(f"unknown weight format {fmt!r}")
        mx = fmt == "mxfp4"
        self.shape = Shape.of(E, top_k, H, I, out_dtype, MOE_W_MXFP4 if mx else MOE_W_INT4)
        bad = []

        def pack(q_np, s_np, is_w13):
            q = torch.from_numpy(np.ascontiguousarray(q_np)).to(device)
            if mx:
                sc = torch.from_numpy(np.ascontiguousarray(s_np, dtype=np.uint8)).to(device)
                packed, pscales, nbad = moe_mxfp4_pack(q, sc, is_w13)
                bad.append(nbad)
                return packed, pscales
            sc = torch.from_numpy(np.ascontiguousarray(s_np).view(np.int16)).to(device)
            cnt = torch.zeros(1, dtype=torch.int32, device=device)
            bad.append(cnt)
            return moe_int4_pack(q, sc, is_w13, inexact=cnt)

        self.w13, self.w13_scales = pack(w["q13"], w["s13"], True)
        self.w2, self.w2_scales = pack(w["q2"], w["s2"], False)
        torch.cuda.synchronize()
        n_bad = sum(int(t.item()) for t in bad)
        # INT4: scales whose dequantised weights are not exact in fp16 (the
        # forward still runs; see moe_int4_pack)
        self.inexact_scales = 0 if mx else n_bad
        if mx and n_bad:
            raise ValueError(f"{n_bad} E8M0 scales outside the supported range [103, 140]")

    def forward(self, x, topk_ids, topk_weights, out=None, workspace=None, stream=None):
        return moe_int4_forward(x, self.w13, self.w13_scales, self.w2, self.w2_scales, topk_ids,
                                topk_weights, self.shape, out=out, workspace=workspace,
                                stream=stream)
