"""Attention forward ORACLE -- test infrastructure only.

A plain float64 CPU statement of the attention forward (``attention_oracle.c``,
which carries the citations).  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package; the
product library never does, and the two share no code.  Inputs come from the
``seeded_inputs`` module as uint16 bit patterns.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, invariants, library routines (numpy/scipy) and an mpmath brute force;
the merge of results over disjoint key sets is pinned against the attention
forward over their union.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attention_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[str, ctypes.CDLL] = {}

DTYPES = {"fp16": 0, "bf16": 1}


def host_threads() -> int:
    """Host cores this process may run on (sched_getaffinity)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def build(source: str | None = None, tag: str = "") -> str:
    """Compile the oracle (or a variant of its source text) with gcc -O2, no fast-math."""
    text = open(SOURCE).read() if source is None else source
    digest = hashlib.sha1(text.encode()).hexdigest()[:12]
    out = os.path.join(_BUILD, f"liboracle{tag}-{digest}.so")
    if not os.path.exists(out):
        os.makedirs(_BUILD, exist_ok=True)
        src_path = out[:-3] + f".{os.getpid()}.c"
        with open(src_path, "w") as f:
            f.write(text)
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-pthread",
                        "-fno-fast-math", "-ffp-contract=off", "-o", tmp, src_path, "-lm"], check=True)
        os.replace(tmp, out)
        os.remove(src_path)
    return out


def load(source: str | None = None, tag: str = "") -> ctypes.CDLL:
    path = build(source, tag)
    with _lock:
        lib = _libs.get(path)
        if lib is None:
            lib = ctypes.CDLL(path)
            lib.oracle_attention_fwd.restype = ctypes.c_int
            lib.oracle_attention_fwd.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_attention_fwd_ex.restype = ctypes.c_int
            lib.oracle_attention_fwd_ex.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_attention_bwd.restype = ctypes.c_int
            lib.oracle_attention_bwd.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_attention_bwd_ex.restype = ctypes.c_int
            lib.oracle_attention_bwd_ex.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_lse_merge.restype = ctypes.c_int
            lib.oracle_lse_merge.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                             ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_decode.restype = ctypes.c_double
            lib.oracle_decode.argtypes = [ctypes.c_uint16, ctypes.c_int]
            _libs[path] = lib
        return lib


def decode(bits: np.ndarray, dtype: str, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """The oracle's own exact fp16/bf16 -> float64 decoding, element by element."""
    lib = lib or load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    code = DTYPES[dtype]
    return np.fromiter((lib.oracle_decode(int(b), code) for b in flat), dtype=np.float64,
                       count=flat.size).reshape(np.shape(bits))


def attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, dtype: str, scale: float, causal: bool,
                  rows: np.ndarray | None = None, nthreads: int | None = None,
                  lib: ctypes.CDLL | None = None):
    """Attention forward in float64.

    q: (Z, Hq, Nq, D), k/v: (Z, Hkv, Nkv, D) uint16 bit arrays (fp16 or bf16).
    rows: optional flat row ids ``(z*Hq + hq)*Nq + i``; by default every row.
    Returns (o, lse): o is (Z, Hq, Nq, D) / lse (Z, Hq, Nq) for all rows, or
    (R, D) / (R,) for the given rows, all float64.
    """
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    Z, Hq, Nq, D = q.shape
    Zk, Hkv, Nkv, Dk = k.shape
    if v.shape != k.shape or Zk != Z or Dk != D:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    if rows is None:
        nrows = Z * Hq * Nq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
    o = np.empty((nrows, D), dtype=np.float64)
    lse = np.empty(nrows, dtype=np.float64)
    rc = lib.oracle_attention_fwd(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, DTYPES[dtype], Z, Hq, Hkv, Nq, Nkv, D,
        float(scale), int(bool(causal)), None if rows_arr is None else rows_arr.ctypes.data, nrows,
        o.ctypes.data if nrows else None, lse.ctypes.data if nrows else None, nthreads or host_threads())
    if rc == -1:
        raise ValueError("oracle_attention_fwd: invalid arguments")
    if rc != 0:
        raise MemoryError("oracle_attention_fwd: out of memory")
    if rows is None:
        return o.reshape(Z, Hq, Nq, D), lse.reshape(Z, Hq, Nq)
    return o, lse


def lse_merge(o_parts, lse_parts, lib: ctypes.CDLL | None = None):
    """Combine results over disjoint key sets in float64 (``oracle_lse_merge``).

    o_parts: sequence of float64 arrays of one shape (..., D); lse_parts:
    matching arrays of shape (...) in natural-log units.  Returns (o, lse)
    for the union of the key sets.
    """
    lib = lib or load()
    n = len(o_parts)
    if n < 1 or n != len(lse_parts):
        raise ValueError("need at least one part and one lse per part")
    shape = np.shape(o_parts[0])
    D = shape[-1]
    rows = int(np.prod(shape[:-1], dtype=np.int64))
    op = np.ascontiguousarray(np.stack([np.asarray(x, dtype=np.float64).reshape(rows, D) for x in o_parts]))
    lp = np.ascontiguousarray(np.stack([np.asarray(x, dtype=np.float64).reshape(rows) for x in lse_parts]))
    o = np.empty((rows, D), dtype=np.float64)
    lse = np.empty(rows, dtype=np.float64)
    rc = lib.oracle_lse_merge(n, op.ctypes.data, lp.ctypes.data, rows, D, o.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_lse_merge: invalid arguments")
    return o.reshape(shape), lse.reshape(shape[:-1])


def attention_fwd_ex(q: np.ndarray, k: np.ndarray, v: np.ndarray, dtype: str, scale: float, causal: bool,
                     window=(-1, -1), alibi=None, cu_q=None, cu_k=None, rows=None, nthreads: int | None = None,
                     lib: ctypes.CDLL | None = None):
    """Attention forward with the variants (``oracle_attention_fwd_ex``), float64.

    window: (left, right), -1 for an open side; alibi: Hq slopes or None.
    Without cu_q/cu_k: q (Z, Hq, Nq, D), k/v (Z, Hkv, Nkv, D) bits as for
    attention_fwd.  With them (int arrays of Z + 1 offsets): q (1, Hq, total_q, D),
    k/v (1, Hkv, total_k, D); rows are flat ids hq * total_q + packed row, and
    rows outside every sequence come back NaN.
    Returns (o, lse) shaped like q without D (all rows) or (R, D) / (R,).
    """
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    Zq, Hq, Nq, D = q.shape
    Zk, Hkv, Nkv, Dk = k.shape
    if v.shape != k.shape or Zk != Zq or Dk != D:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    varlen = cu_q is not None
    if varlen:
        cq = np.ascontiguousarray(cu_q, dtype=np.int32)
        ck = np.ascontiguousarray(cu_k, dtype=np.int32)
        if Zq != 1 or cq.shape != ck.shape:
            raise ValueError("varlen takes (1, H, total, D) tensors and matching offset arrays")
        Z = cq.size - 1
    else:
        cq = ck = None
        Z = Zq
    sl = None if alibi is None else np.ascontiguousarray(alibi, dtype=np.float64)
    total = Hq * Nq * (1 if varlen else Z)
    if rows is None:
        nrows, rows_arr = total, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
    o = np.empty((nrows, D), dtype=np.float64)
    lse = np.empty(nrows, dtype=np.float64)
    rc = lib.oracle_attention_fwd_ex(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, DTYPES[dtype], Z, Hq, Hkv, Nq, Nkv, D, float(scale),
        int(bool(causal)), int(window[0]), int(window[1]), None if sl is None else sl.ctypes.data,
        None if cq is None else cq.ctypes.data, None if ck is None else ck.ctypes.data,
        None if rows_arr is None else rows_arr.ctypes.data, nrows, o.ctypes.data if nrows else None,
        lse.ctypes.data if nrows else None, nthreads or host_threads())
    if rc == -1:
        raise ValueError("oracle_attention_fwd_ex: invalid arguments")
    if rc != 0:
        raise MemoryError("oracle_attention_fwd_ex: out of memory")
    if rows is None:
        return o.reshape(q.shape), lse.reshape(q.shape[:3])
    return o, lse


def attention_bwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray, dtype: str, scale: float, causal: bool,
                  nthreads: int | None = None, lib: ctypes.CDLL | None = None):
    """Gradients (dq, dk, dv) of the attention forward for upstream gradient do, float64.

    q, do: (Z, Hq, Nq, D); k, v: (Z, Hkv, Nkv, D) uint16 bit arrays of dtype.
    """
    lib = lib or load()
    q, k, v, do = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v, do))
    Z, Hq, Nq, D = q.shape
    Zk, Hkv, Nkv, Dk = k.shape
    if v.shape != k.shape or do.shape != q.shape or Zk != Z or Dk != D:
        raise ValueError("shape mismatch")
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(k.shape, dtype=np.float64)
    rc = lib.oracle_attention_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, do.ctypes.data, DTYPES[dtype], Z, Hq,
                                  Hkv, Nq, Nkv, D, float(scale), int(bool(causal)), dq.ctypes.data, dk.ctypes.data,
                                  dv.ctypes.data, nthreads or host_threads())
    if rc == -1:
        raise ValueError("oracle_attention_bwd: invalid arguments")
    if rc != 0:
        raise MemoryError("oracle_attention_bwd: out of memory")
    return dq, dk, dv


def attention_bwd_ex(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray, dtype: str, scale: float,
                     causal: bool, window=(-1, -1), alibi=None, cu_q=None, cu_k=None, nthreads: int | None = None,
                     lib: ctypes.CDLL | None = None):
    """Gradients (dq, dk, dv) of attention_fwd_ex's forward, float64.

    window: (left, right), -1 for an open side; alibi: Hq slopes or None.
    Without cu_q/cu_k: q, do (Z, Hq, Nq, D); k, v (Z, Hkv, Nkv, D) uint16 bit
    arrays of dtype.  With them (int arrays of Z + 1 offsets, as for
    attention_fwd_ex): q, do (1, Hq, total_q, D), k, v (1, Hkv, total_k, D);
    a sequence attends only to its own keys, so its gradients are those of
    the dense backward on its own rows (a sequence without keys: dq = 0), and
    rows outside every sequence get 0.
    """
    lib = lib or load()
    if cu_q is not None or cu_k is not None:
        if cu_q is None or cu_k is None or q.shape[0] != 1:
            raise ValueError("varlen takes (1, H, total, D) tensors and both offset arrays")
        cq, ck = np.asarray(cu_q, dtype=np.int64), np.asarray(cu_k, dtype=np.int64)
        dq = np.zeros(q.shape, dtype=np.float64)
        dk = np.zeros(k.shape, dtype=np.float64)
        dv = np.zeros(k.shape, dtype=np.float64)
        for z in range(len(cq) - 1):
            a, b, c, e = int(cq[z]), int(cq[z + 1]), int(ck[z]), int(ck[z + 1])
            if b == a or e == c:
                continue
            g = attention_bwd_ex(q[:, :, a:b], k[:, :, c:e], v[:, :, c:e], do[:, :, a:b], dtype, scale, causal,
                                 window=window, alibi=alibi, nthreads=nthreads, lib=lib)
            dq[:, :, a:b], dk[:, :, c:e], dv[:, :, c:e] = g
        return dq, dk, dv
    q, k, v, do = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v, do))
    Z, Hq, Nq, D = q.shape
    Zk, Hkv, Nkv, Dk = k.shape
    if v.shape != k.shape or do.shape != q.shape or Zk != Z or Dk != D:
        raise ValueError("shape mismatch")
    slopes = None if alibi is None else np.ascontiguousarray(alibi, dtype=np.float64)
    if slopes is not None and slopes.shape != (Hq,):
        raise ValueError("alibi takes one slope per query head")
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(k.shape, dtype=np.float64)
    rc = lib.oracle_attention_bwd_ex(q.ctypes.data, k.ctypes.data, v.ctypes.data, do.ctypes.data, DTYPES[dtype], Z,
                                     Hq, Hkv, Nq, Nkv, D, float(scale), int(bool(causal)), int(window[0]),
                                     int(window[1]), None if slopes is None else slopes.ctypes.data, dq.ctypes.data,
                                     dk.ctypes.data, dv.ctypes.data, nthreads or host_threads())
    if rc == -1:
        raise ValueError("oracle_attention_bwd_ex: invalid arguments")
    if rc != 0:
        raise MemoryError("oracle_attention_bwd_ex: out of memory")
    return dq, dk, dv
