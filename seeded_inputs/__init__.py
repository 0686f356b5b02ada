"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds no attention arithmetic.  It draws iid N(0, 1) samples from a
counter-based splitmix64 stream through Box-Muller (both in ``normal_gen.c``)
and rounds them, in float64, to IEEE binary16 or bfloat16 (round to nearest
even).  Arrays come back as ``uint16`` bit patterns in BNSD order
``(Z, H, N, D)``, contiguous; callers view them as fp16/bf16 tensors.

Q, K and V for one problem are one stream: Q takes normals ``[0, nQ)``, K
``[nQ, nQ + nK)`` and V ``[nQ + nK, nQ + 2 nK)`` of the stream ``seed``.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "normal_gen.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"fp16": 0, "bf16": 1, "f64": 2}


def _host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux
        return max(1, os.cpu_count() or 1)


def build() -> str:
    """Compile ``normal_gen.c`` into ``_build/libseeded_inputs-<hash>.so`` (gcc, -O2)."""
    with open(_SRC, "rb") as f:
        tag = hashlib.sha1(f.read()).hexdigest()[:12]
    out = os.path.join(_BUILD, f"libseeded_inputs-{tag}.so")
    if not os.path.exists(out):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-pthread",
                        "-fno-fast-math", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, out)
    return out


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.si_fill_normal.restype = ctypes.c_int
            lib.si_fill_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_int]
            lib.si_normal_at.restype = ctypes.c_double
            lib.si_normal_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.si_splitmix64_at.restype = ctypes.c_uint64
            lib.si_splitmix64_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.si_round_f16.restype = ctypes.c_uint16
            lib.si_round_f16.argtypes = [ctypes.c_double]
            lib.si_round_bf16.restype = ctypes.c_uint16
            lib.si_round_bf16.argtypes = [ctypes.c_double]
            _lib = lib
        return _lib


def normals(seed: int, offset: int, n: int, dtype: str = "f64", nthreads: int | None = None) -> np.ndarray:
    """Normals ``offset .. offset+n-1`` of stream ``seed``: float64, or uint16 bits for fp16/bf16."""
    lib = _load()
    out = np.empty(n, dtype=np.float64 if dtype == "f64" else np.uint16)
    rc = lib.si_fill_normal(seed, offset, n, DTYPE_CODES[dtype], out.ctypes.data if n else None,
                            nthreads or _host_threads())
    if rc != 0:
        raise ValueError("si_fill_normal rejected its arguments")
    return out


def round_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to fp16/bf16 bit patterns (nearest even) with the generator's own rounding."""
    lib = _load()
    fn = lib.si_round_f16 if dtype == "fp16" else lib.si_round_bf16
    flat = np.asarray(x, dtype=np.float64).ravel()
    return np.fromiter((fn(float(v)) for v in flat), dtype=np.uint16, count=flat.size).reshape(np.shape(x))


def qkv(seed: int, Z: int, Hq: int, Hkv: int, Nq: int, Nkv: int, D: int, dtype: str):
    """Q (Z,Hq,Nq,D), K and V (Z,Hkv,Nkv,D) as uint16 bit arrays, drawn in that order from one stream."""
    nq = Z * Hq * Nq * D
    nk = Z * Hkv * Nkv * D
    q = normals(seed, 0, nq, dtype).reshape(Z, Hq, Nq, D)
    k = normals(seed, nq, nk, dtype).reshape(Z, Hkv, Nkv, D)
    v = normals(seed, nq + nk, nk, dtype).reshape(Z, Hkv, Nkv, D)
    return q, k, v


def as_torch(bits: np.ndarray, dtype: str):
    """View uint16 bits as a CPU torch fp16/bf16 tensor (no copy of values, no rounding)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == "fp16" else torch.bfloat16)
