"""Oracle for the weight-only INT4 MoE expert MLP (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The product
path (the CUDA library and its Python binding) never does, and it shares no code
with it.

The arithmetic lives in ``moe_oracle.c`` (plain fp64 C loops, compiled with gcc,
``-ffp-contract=off`` so x86 and Arm give identical bits).  This module only
marshals numpy arrays into it and splits token lists over threads (ctypes drops
the GIL during the call, so threads run the C loops in parallel).

Functions and the passages they follow:

* :func:`moe_forward` -- the routed SwiGLU expert MLP with INT4 group-32 weights
  and the top-k weighted combine ("The Throughput Lever", sections "Building the
  Benchmark" and "Phase 3: The INT4 Marlin MoE Throughput Lever").
* :func:`moe_intermediate` -- the SwiGLU intermediate of single routing pairs.
* :func:`align` -- the bucket-by-expert, pad-to-block index buffers.
* :func:`route` -- top-k routing from router logits (softmax over the experts,
  the top_k largest, renormalised over them): each token activates top_k of the
  experts ("The Throughput Lever", section "The Result: Two Regimes").
* :func:`bf16_to_double`, :func:`nibble`, :func:`weight` -- one INT4 weight
  (q - 8) * scale, exactly.
* :func:`e2m1`, :func:`e8m0`, :func:`weight_fmt` and the ``fmt="mxfp4"``
  argument -- MXFP4 experts, FP4 E2M1 codes with an E8M0 scale per 32 (OCP
  Microscaling v1.0; "From 1,060 to 4,016 tok/s on one B300", MXFP4 experts).

Every function is pinned by CPU tests against closed forms, library routines,
cited tables and brute force (``tests/test_oracle.py``,
``tests/test_oracle_mxfp4.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no GPU).  Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_nibble.argtypes = [p, i64]
        lib.oracle_nibble.restype = ctypes.c_int
        lib.oracle_weight.argtypes = [p, p, i64, i64, i64, i64, i64]
        lib.oracle_weight.restype = ctypes.c_double
        lib.oracle_moe_forward_tokens.argtypes = [p] * 7 + [i64] * 5 + [p, i64, p, p]
        lib.oracle_moe_forward_tokens.restype = i64
        lib.oracle_moe_forward_tokens_fmt.argtypes = ([ctypes.c_int] + [p] * 7 + [i64] * 5
                                                      + [p, i64, p, p])
        lib.oracle_moe_forward_tokens_fmt.restype = i64
        lib.oracle_e2m1.argtypes = [ctypes.c_int]
        lib.oracle_e2m1.restype = ctypes.c_double
        lib.oracle_e8m0.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0.restype = ctypes.c_double
        lib.oracle_weight_fmt.argtypes = [ctypes.c_int, p, p, i64, i64, i64, i64, i64]
        lib.oracle_weight_fmt.restype = ctypes.c_double
        lib.oracle_moe_intermediate_pairs.argtypes = [p] * 4 + [i64] * 5 + [p, i64, p]
        lib.oracle_moe_intermediate_pairs.restype = None
        lib.oracle_moe_intermediate_pairs_fmt.argtypes = ([ctypes.c_int] + [p] * 4 + [i64] * 5
                                                          + [p, i64, p])
        lib.oracle_moe_intermediate_pairs_fmt.restype = None
        lib.oracle_align.argtypes = [p, i64, i64, i64, i64, p, i64, p, i64, p]
        lib.oracle_route.argtypes = [p, i64, i64, i64, p, p]
        lib.oracle_route.restype = None
        lib.oracle_align.restype = i64
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def bf16_to_double(bits: int) -> float:
    """Exact value of one bf16 bit pattern."""
    return _load().oracle_bf16_to_double(int(bits))


def nibble(row: np.ndarray, k: int) -> int:
    """Canonical nibble k of a packed byte row."""
    row = _c(row, np.uint8)
    return _load().oracle_nibble(_ptr(row), int(k))


def weight(q: np.ndarray, s: np.ndarray, e: int, n: int, k: int) -> float:
    """Dequantised weight W[e, n, k] = (q - 8) * scale of a [E, N, K] matrix."""
    q = _c(q, np.uint8)
    s = _c(s, np.uint16)
    E, N, K2 = q.shape
    return _load().oracle_weight(_ptr(q), _ptr(s), N, 2 * K2, e, n, k)


# Weight formats: INT4 (q - 8) * bf16 scale; MXFP4 e2m1(q) * 2^(e8m0 - 127).
FORMATS = {"int4": (0, np.uint16), "mxfp4": (1, np.uint8)}


def e2m1(code: int) -> float:
    """Value of one FP4 E2M1 code (OCP Microscaling v1.0 element type)."""
    return _load().oracle_e2m1(int(code))


def e8m0(bits: int) -> float:
    """Value of one E8M0 scale: 2^(bits - 127); 255 is NaN."""
    return _load().oracle_e8m0(int(bits))


def weight_fmt(fmt: str, q: np.ndarray, s: np.ndarray, e: int, n: int, k: int) -> float:
    """Dequantised weight W[e, n, k] of a [E, N, K] matrix in format fmt."""
    code, sdt = FORMATS[fmt]
    q = _c(q, np.uint8)
    s = _c(s, sdt)
    E, N, K2 = q.shape
    return _load().oracle_weight_fmt(code, _ptr(q), _ptr(s), N, 2 * K2, e, n, k)


def _default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def moe_forward(x, q13, s13, q2, s2, topk_ids, topk_weights, tokens=None,
                threads: int | None = None, fmt: str = "int4"):
    """Layer output in fp64 for the given tokens (all tokens by default).

    x: uint16 bf16 bits [M, H]; q13 uint8 [E, 2I, H/2]; s13 [E, 2I, H/32];
    q2 uint8 [E, H, I/2]; s2 [E, H, I/32]; topk_ids int32 [M, k];
    topk_weights float32 [M, k].  Scales: uint16 bf16 bits (fmt "int4") or
    uint8 E8M0 (fmt "mxfp4").  Returns (out float64 [n, H], n_dropped).
    """
    lib = _load()
    fcode, sdt = FORMATS[fmt]
    x = _c(x, np.uint16)
    q13 = _c(q13, np.uint8)
    s13 = _c(s13, sdt)
    q2 = _c(q2, np.uint8)
    s2 = _c(s2, sdt)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_weights, np.float32)
    M, H = x.shape
    E, twoI, _ = q13.shape
    I = twoI // 2
    k = ids.shape[1] if ids.ndim == 2 else 1
    assert q13.shape == (E, 2 * I, H // 2) and s13.shape == (E, 2 * I, H // 32)
    assert q2.shape == (E, H, I // 2) and s2.shape == (E, H, I // 32)
    assert ids.size == M * k and w.size == M * k
    toks = np.arange(M, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    out = np.zeros((len(toks), H), dtype=np.float64)
    nthreads = max(1, min(threads or _default_threads(), len(toks)))
    chunks = [c for c in np.array_split(np.arange(len(toks)), nthreads) if len(c)]

    def run(idx):
        sub = _c(toks[idx], np.int64)
        o = np.zeros((len(sub), H), dtype=np.float64)
        scratch = np.zeros(I + H, dtype=np.float64)
        d = lib.oracle_moe_forward_tokens_fmt(
            fcode, _ptr(x), _ptr(q13), _ptr(s13), _ptr(q2), _ptr(s2), _ptr(ids), _ptr(w),
            M, E, k, H, I, _ptr(sub), len(sub), _ptr(scratch), _ptr(o))
        out[idx] = o
        return d

    if len(chunks) == 1:
        dropped = run(chunks[0]) if len(toks) else 0
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            dropped = sum(ex.map(run, chunks))
    return out, int(dropped)


def moe_intermediate(x, q13, s13, topk_ids, pairs, threads: int | None = None,
                     fmt: str = "int4"):
    """SwiGLU intermediate a [n, I] (fp64) of routing pairs (flat index t*k+j)."""
    lib = _load()
    fcode, sdt = FORMATS[fmt]
    x = _c(x, np.uint16)
    q13 = _c(q13, np.uint8)
    s13 = _c(s13, sdt)
    ids = _c(topk_ids, np.int32)
    M, H = x.shape
    E, twoI, _ = q13.shape
    I = twoI // 2
    k = ids.shape[1] if ids.ndim == 2 else 1
    pairs = _c(pairs, np.int64)
    out = np.zeros((len(pairs), I), dtype=np.float64)
    nthreads = max(1, min(threads or _default_threads(), len(pairs)))
    chunks = [c for c in np.array_split(np.arange(len(pairs)), nthreads) if len(c)]

    def run(idx):
        sub = _c(pairs[idx], np.int64)
        o = np.zeros((len(sub), I), dtype=np.float64)
        lib.oracle_moe_intermediate_pairs_fmt(fcode, _ptr(x), _ptr(q13), _ptr(s13), _ptr(ids),
                                              M, E, k, H, I, _ptr(sub), len(sub), _ptr(o))
        out[idx] = o

    if len(chunks) == 1:
        if len(pairs):
            run(chunks[0])
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            list(ex.map(run, chunks))
    return out


def align(topk_ids, E: int, block_m: int):
    """Bucketed, padded routing-pair indices.

    Returns (sorted_ids int32 [num_post_pad], expert_ids int32 [num_post_pad /
    block_m], num_post_pad, n_dropped).  Pad entries hold P = M*k.
    """
    lib = _load()
    ids = _c(topk_ids, np.int32).reshape(-1)
    P = ids.size
    cap = P + E * (block_m - 1) + 1
    sorted_ids = np.zeros(cap, dtype=np.int32)
    expert_ids = np.zeros(cap // block_m + 1, dtype=np.int32)
    dropped = np.zeros(1, dtype=np.int64)
    M = P  # treat the flat list as M=P tokens of one slot: same flat indices
    n = lib.oracle_align(_ptr(ids), M, 1, E, block_m, _ptr(sorted_ids), cap,
                         _ptr(expert_ids), len(expert_ids), _ptr(dropped))
    if n < 0:
        raise RuntimeError("oracle align capacity exceeded")
    return sorted_ids[:n].copy(), expert_ids[: n // block_m].copy(), int(n), int(dropped[0])


def route(logits, top_k: int):
    """Top-k experts per token by router logit (ties: lower index first) and their
    renormalised softmax weights.  Returns (ids int32 [M, k], weights fp64 [M, k])."""
    lg = _c(logits, np.float32)
    M, E = lg.shape
    ids = np.empty((M, top_k), dtype=np.int32)
    w = np.empty((M, top_k), dtype=np.float64)
    if M:
        _load().oracle_route(_ptr(lg), M, E, top_k, _ptr(ids), _ptr(w))
    return ids, w

