"""ctypes binding of libfa: argument marshalling only.

Every step of the attention forward runs inside libfa's CUDA kernels; this
module turns torch tensors into pointers, sizes and element strides and
forwards them to the C ABI declared in include/fa.h, under the same names.
If libfa.so has not been built it raises, it never computes anything itself.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import build as _build

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_ALIGNMENT = 3
FA_ERR_CUDA = 4
FA_ERR_DEVICE_TIMEOUT = 5
FA_DTYPE_F16 = 0
FA_DTYPE_BF16 = 1

# every symbol include/fa.h declares, with its ctypes signature
_SIGNATURES = {
    "fa_fwd": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 6 +
               [ctypes.c_void_p] * 4 + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "fa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fa_device_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]),
    "fa_fwd_plan": (ctypes.c_int, [ctypes.c_int] * 8 + [ctypes.POINTER(ctypes.c_int64)] * 2 +
                    [ctypes.POINTER(ctypes.c_int)] * 3),
    "fa_debug_set_wait_limit_ms": (None, [ctypes.c_double]),
    "fa_debug_inject_stall": (None, [ctypes.c_int]),
}

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


class fa_strides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("n", ctypes.c_int64), ("d", ctypes.c_int64)]


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libfa.so (built by exact_attention_44_gb300.build); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise ImportError(f"libfa.so is not built ({path}); run `python -m exact_attention_44_gb300.build`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def status_string(code: int) -> str:
    try:
        return load().fa_status_string(int(code)).decode()
    except ImportError:
        return f"status {code}"


fa_status_string = status_string


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float16:
        return FA_DTYPE_F16
    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    raise TypeError(f"fa_fwd takes float16 or bfloat16 tensors, got {t.dtype}")


def _strides(t) -> fa_strides:
    b, h, n, d = t.stride()
    return fa_strides(b, h, n, d)


def fa_fwd(q, k, v, o=None, lse=None, *, scale: float | None = None, causal: bool = False, stream=None,
           want_lse: bool = True):
    """Attention forward through libfa.

    q: (Z, Hq, Nq, D); k, v: (Z, Hkv, Nkv, D) CUDA tensors of one dtype (fp16
    or bf16), any strides with d-stride 1.  o (optional) receives the output
    in the same dtype; lse (optional) is a contiguous (Z, Hq, Nq) fp32 tensor.
    scale defaults to 1/sqrt(D).  Launches on `stream` (a torch.cuda.Stream)
    or the current stream and returns (o, lse) without synchronising.
    """
    import torch

    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D (Z, H, N, D)")
    Z, Hq, Nq, D = q.shape
    Zk, Hkv, Nkv, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Zk != Z or Dk != D:
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if o is None:
        o = torch.empty_like(q, memory_format=torch.contiguous_format)
    if tuple(o.shape) != tuple(q.shape) or o.dtype != q.dtype:
        raise ValueError("o must match q's shape and dtype")
    if lse is None and want_lse:
        lse = torch.empty((Z, Hq, Nq), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (Z, Hq, Nq) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 (Z, Hq, Nq) tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sq, sk, sv, so = _strides(q), _strides(k), _strides(v), _strides(o)
    with torch.cuda.device(q.device):
        rc = load().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr() if lse is not None else None, Z, Hq, Hkv, Nq, Nkv, D,
                           ctypes.byref(sq), ctypes.byref(sk), ctypes.byref(sv), ctypes.byref(so),
                           float(scale), int(bool(causal)), dt, ctypes.c_void_p(stream.cuda_stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return o, lse


def fa_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None, Z: int, Hq: int, Hkv: int,
               Nq: int, Nkv: int, D: int, sq, sk, sv, so, scale: float, causal: bool, dtype: int,
               stream_handle: int = 0) -> int:
    """The C entry point with raw pointers and (b, h, n, d) stride tuples; returns the status code."""
    st = [fa_strides(*s) if s is not None else None for s in (sq, sk, sv, so)]
    refs = [ctypes.byref(s) if s is not None else None for s in st]
    return load().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, Z, Hq, Hkv, Nq, Nkv, D, *refs, float(scale),
                         int(causal), int(dtype), ctypes.c_void_p(stream_handle))


def fa_device_status(stream=None) -> tuple[int, int]:
    """Synchronise the stream, read and clear the device status word: (code, raw word)."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    word = ctypes.c_uint32(0)
    rc = load().fa_device_status(ctypes.c_void_p(stream.cuda_stream), ctypes.byref(word))
    return rc, word.value


def fa_fwd_plan(Z: int, Hq: int, Hkv: int, Nq: int, Nkv: int, D: int, causal: bool, num_sms: int = 0) -> dict:
    """Host-only work description (no CUDA call): tiles, kv_blocks, block_n, grid, smem_bytes."""
    tiles, pairs = ctypes.c_int64(), ctypes.c_int64()
    bn, grid, smem = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = load().fa_fwd_plan(Z, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), num_sms, ctypes.byref(tiles),
                            ctypes.byref(pairs), ctypes.byref(bn), ctypes.byref(grid), ctypes.byref(smem))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_plan")
    return {"tiles": tiles.value, "kv_blocks": pairs.value, "block_n": bn.value, "grid": grid.value,
            "smem_bytes": smem.value}


def fa_debug_set_wait_limit_ms(ms: float) -> None:
    load().fa_debug_set_wait_limit_ms(float(ms))


def fa_debug_inject_stall(enable: bool) -> None:
    load().fa_debug_inject_stall(int(bool(enable)))
