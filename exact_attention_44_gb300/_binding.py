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
FA_ERR_WORKSPACE = 6
FA_ERR_DEVICE_CHECK = 7
FA_MERGE_MAX_PARTS = 16
FA_DTYPE_F16 = 0
FA_DTYPE_BF16 = 1

# every symbol include/fa.h declares, with its ctypes signature
_SIGNATURES = {
    "fa_fwd": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 6 +
               [ctypes.c_void_p] * 4 + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "fa_fwd_splitkv": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 6 +
                       [ctypes.c_void_p] * 4 + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                                 ctypes.c_size_t, ctypes.c_void_p]),
    "fa_fwd_splitkv_workspace_size": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "fa_fwd_splitkv_workspace_size_for": (ctypes.c_int, [ctypes.c_int, ctypes.c_int,
                                                         ctypes.POINTER(ctypes.c_size_t)]),
    "fa_bwd": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 6 + [ctypes.c_void_p] * 8 +
               [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "fa_bwd_workspace_size": (ctypes.c_int, [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_size_t)]),
    "fa_bwd_ex": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 6 + [ctypes.c_void_p] * 8 +
                  [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                   ctypes.c_void_p]),
    "fa_fwd_ex": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 6 +
                  [ctypes.c_void_p] * 4 + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                            ctypes.c_void_p]),
    "fa_fwd_splitkv_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 6 +
                               [ctypes.c_void_p] * 4 + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "fa_lse_merge": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p)] +
                     [ctypes.c_int] * 4 + [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_void_p]),
    "fa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fa_device_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]),
    "fa_fwd_plan": (ctypes.c_int, [ctypes.c_int] * 8 + [ctypes.POINTER(ctypes.c_int64)] * 2 +
                    [ctypes.POINTER(ctypes.c_int)] * 3),
    "fa_fwd_schedule": (ctypes.c_int, [ctypes.c_int] * 9 + [ctypes.c_int64, ctypes.c_void_p]),
    "fa_debug_set_wait_limit_ms": (None, [ctypes.c_double]),
    "fa_debug_inject_stall": (None, [ctypes.c_int]),
    "fa_debug_force_split": (None, [ctypes.c_int]),
    "fa_debug_force_chains": (None, [ctypes.c_int]),
    "fa_debug_force_pair": (None, [ctypes.c_int]),
    "fa_debug_exp2": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
}

_lock = threading.Lock()
_lib = None
_path = None  # another build of libfa to load instead of the default one (use_library)


class FaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


class fa_strides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("n", ctypes.c_int64), ("d", ctypes.c_int64)]


class fa_fwd_options(ctypes.Structure):
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int), ("alibi_slopes", ctypes.c_void_p),
                ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p), ("max_seqlen_q", ctypes.c_int),
                ("max_seqlen_k", ctypes.c_int)]


class fa_fwd_schedule_info(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int), ("split", ctypes.c_int), ("gqa_packed", ctypes.c_int),
                ("head_group", ctypes.c_int), ("alternate", ctypes.c_int), ("tiles", ctypes.c_int64),
                ("kv_blocks", ctypes.c_int64), ("busiest_blocks", ctypes.c_int64), ("softmax_chains", ctypes.c_int),
                ("cta_pairs", ctypes.c_int)]


def library_path() -> str:
    return _build.LIB


def use_library(path: str | None) -> str | None:
    """Make later calls go to the libfa.so at `path` (None: the default build), e.g. the
    debug-check build; returns the path used before.  Not for concurrent use."""
    global _lib, _path
    with _lock:
        before = _path
        _path = path
        _lib = None
    return before


def load() -> ctypes.CDLL:
    """Load libfa.so (built by exact_attention_44_gb300.build); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = _path or library_path()
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


def _prepare(q, k, v, o, lse, scale, want_lse, stream):
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
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr() if lse is not None else None,
            Z, Hq, Hkv, Nq, Nkv, D]
    strides = [_strides(q), _strides(k), _strides(v), _strides(o)]
    return o, lse, dt, float(scale), stream, args, strides


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

    o, lse, dt, scale, stream, args, st = _prepare(q, k, v, o, lse, scale, want_lse, stream)
    with torch.cuda.device(q.device):
        rc = load().fa_fwd(*args, *[ctypes.byref(x) for x in st], scale, int(bool(causal)), dt,
                           ctypes.c_void_p(stream.cuda_stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return o, lse


def _packed(t):
    """(total, H, D) packed rows -> the (1, H, total, D) view the C ABI takes; 4-D passes through."""
    return t.unsqueeze(0).permute(0, 2, 1, 3) if t.dim() == 3 else t


def fa_fwd_ex(q, k, v, o=None, lse=None, *, scale: float | None = None, causal: bool = False, window=(-1, -1),
              alibi_slopes=None, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q: int | None = None,
              stream=None, want_lse: bool = True):
    """fa_fwd with a sliding window, ALiBi slopes and/or packed variable-length sequences (libfa's fa_fwd_ex).

    window: (left, right), -1 for an open side.  alibi_slopes: CUDA fp32 (Hq,).
    With cu_seqlens_q / cu_seqlens_k (CUDA int32, Z + 1 offsets), q, k, v
    (and o) hold packed rows, either (total, H, D) or (1, H, total, D), and o
    comes back in q's form; lse is then (Hq, total_q); max_seqlen_q defaults
    to the longest query sequence (read back from the device once).
    """
    import torch

    varlen = cu_seqlens_q is not None or cu_seqlens_k is not None
    o_user = o
    if varlen:
        if cu_seqlens_q is None or cu_seqlens_k is None:
            raise ValueError("pass both cu_seqlens_q and cu_seqlens_k")
        if o is None and q.dim() == 3:
            o_user = torch.empty_like(q, memory_format=torch.contiguous_format)
        q, k, v = _packed(q), _packed(k), _packed(v)
        if o_user is not None:
            o = _packed(o_user)
        if max_seqlen_q is None:
            cq = cu_seqlens_q.cpu()
            max_seqlen_q = int((cq[1:] - cq[:-1]).max().item()) if cq.numel() > 1 else 0
    if o is None:
        o = torch.empty_like(q, memory_format=torch.contiguous_format)
    _, Hq, Nq, D = q.shape
    if varlen and lse is None and want_lse:
        lse = torch.empty((Hq, Nq), dtype=torch.float32, device=q.device)
    lse_arg = lse
    if varlen and lse is not None:
        if lse.dtype != torch.float32 or tuple(lse.shape) != (Hq, Nq) or not lse.is_contiguous():
            raise ValueError("lse must be a contiguous float32 (Hq, total_q) tensor")
        lse_arg = lse.view(1, Hq, Nq)
    o, lse_arg, dt, scale, stream, args, st = _prepare(q, k, v, o, lse_arg, scale, want_lse and not varlen, stream)
    if varlen:
        args[5] = cu_seqlens_q.numel() - 1  # Z: number of sequences
        if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
    if alibi_slopes is not None and (alibi_slopes.dtype != torch.float32 or alibi_slopes.numel() != Hq):
        raise ValueError("alibi_slopes must be float32 with Hq entries")
    opt = fa_fwd_options(int(window[0]), int(window[1]),
                         alibi_slopes.data_ptr() if alibi_slopes is not None else None,
                         cu_seqlens_q.data_ptr() if varlen else None, cu_seqlens_k.data_ptr() if varlen else None,
                         int(max_seqlen_q or 0))
    with torch.cuda.device(q.device):
        rc = load().fa_fwd_ex(*args, *[ctypes.byref(x) for x in st], scale, int(bool(causal)), dt, ctypes.byref(opt),
                              ctypes.c_void_p(stream.cuda_stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_ex")
    return (o_user if o_user is not None else o), (lse if varlen else lse_arg)


def fa_bwd_workspace_size(Z: int, Hq: int, Nq: int, D: int) -> int:
    """Workspace bytes fa_bwd needs (host only)."""
    n = ctypes.c_size_t(0)
    rc = load().fa_bwd_workspace_size(int(Z), int(Hq), int(Nq), int(D), ctypes.byref(n))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_workspace_size")
    return n.value


def fa_bwd(q, k, v, o, lse, do, dq=None, dk=None, dv=None, *, scale: float | None = None, causal: bool = False,
           workspace=None, stream=None):
    """Gradients (dq, dk, dv) of the attention forward through libfa's fa_bwd.

    q, k, v, o, lse: the forward's inputs, output and lse (fa_fwd's layouts);
    do: upstream gradient shaped like o.  Outputs are allocated when omitted;
    workspace (CUDA uint8, >= fa_bwd_workspace_size bytes) likewise.
    """
    return _bwd(q, k, v, o, lse, do, dq, dk, dv, scale, causal, workspace, stream, None)


def fa_bwd_ex(q, k, v, o, lse, do, dq=None, dk=None, dv=None, *, scale: float | None = None, causal: bool = False,
              window=(-1, -1), alibi_slopes=None, cu_seqlens_q=None, cu_seqlens_k=None,
              max_seqlen_q: int | None = None, max_seqlen_k: int | None = None, workspace=None, stream=None):
    """Gradients of fa_fwd_ex's forward (libfa's fa_bwd_ex; every head dim, any option).

    Arguments as for fa_bwd, plus the options the forward took: window (left,
    right), -1 for an open side; alibi_slopes (CUDA fp32 (Hq,) or None); and
    cu_seqlens_q / cu_seqlens_k (CUDA int32, Z + 1 offsets) for packed
    sequences: q, k, v, o, do (and dq, dk, dv) then hold packed rows, either
    (total, H, D) or (1, H, total, D), the gradients come back in q's / k's
    form, lse is the forward's (Hq, total_q), and max_seqlen_q / max_seqlen_k
    default to the longest sequences (read back from the device once).
    """
    import torch

    varlen = cu_seqlens_q is not None or cu_seqlens_k is not None
    Hq = q.shape[1] if q.dim() == 4 else q.shape[-2]
    if alibi_slopes is not None and (alibi_slopes.dtype != torch.float32 or alibi_slopes.numel() != Hq):
        raise ValueError("alibi_slopes must be float32 with Hq entries")
    if not varlen:
        opt = fa_fwd_options(int(window[0]), int(window[1]),
                             alibi_slopes.data_ptr() if alibi_slopes is not None else None, None, None, 0, 0)
        return _bwd(q, k, v, o, lse, do, dq, dk, dv, scale, causal, workspace, stream, opt)
    if cu_seqlens_q is None or cu_seqlens_k is None:
        raise ValueError("pass both cu_seqlens_q and cu_seqlens_k")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must hold the same Z + 1 offsets")

    def longest(cu):
        c = cu.cpu()
        return int((c[1:] - c[:-1]).max().item()) if c.numel() > 1 else 0

    if max_seqlen_q is None:
        max_seqlen_q = longest(cu_seqlens_q)
    if max_seqlen_k is None:
        max_seqlen_k = longest(cu_seqlens_k)
    grads = []
    for g, like in ((dq, q), (dk, k), (dv, v)):
        grads.append(torch.empty_like(like, memory_format=torch.contiguous_format) if g is None else g)
    dq_user, dk_user, dv_user = grads
    opt = fa_fwd_options(int(window[0]), int(window[1]),
                         alibi_slopes.data_ptr() if alibi_slopes is not None else None, cu_seqlens_q.data_ptr(),
                         cu_seqlens_k.data_ptr(), int(max_seqlen_q), int(max_seqlen_k))
    _bwd(_packed(q), _packed(k), _packed(v), _packed(o), lse, _packed(do), _packed(dq_user), _packed(dk_user),
         _packed(dv_user), scale, causal, workspace, stream, opt,
         seqs=(cu_seqlens_q.numel() - 1, int(max_seqlen_q)))
    return dq_user, dk_user, dv_user


def _bwd(q, k, v, o, lse, do, dq, dk, dv, scale, causal, workspace, stream, opt, seqs=None):
    """Marshal one fa_bwd / fa_bwd_ex call.  seqs = (number of sequences,
    longest query sequence) for packed tensors (batch extent one, lse (Hq, total))."""
    import torch

    Z, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    dt = _dtype_code(q)
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do)):
        if t.dtype != q.dtype:
            raise TypeError(f"{name} must have q's dtype")
    if tuple(o.shape) != tuple(q.shape) or tuple(do.shape) != tuple(q.shape) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch")
    lse_shape, ws_rows = (Z, Hq, Nq), Nq
    if seqs is not None:
        if Z != 1:
            raise ValueError("packed sequences take (1, H, total, D) or (total, H, D) tensors")
        Z, ws_rows = seqs
        lse_shape = (Hq, Nq)
    if lse.dtype != torch.float32 or tuple(lse.shape) != lse_shape or not lse.is_contiguous():
        raise ValueError(f"lse must be the forward's contiguous float32 {lse_shape} tensor")
    dq = torch.empty_like(q, memory_format=torch.contiguous_format) if dq is None else dq
    dk = torch.empty_like(k, memory_format=torch.contiguous_format) if dk is None else dk
    dv = torch.empty_like(v, memory_format=torch.contiguous_format) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(max(1, fa_bwd_workspace_size(Z, Hq, ws_rows, D)), dtype=torch.uint8, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = [_strides(x) for x in (q, k, v, o, do, dq, dk, dv)]
    with torch.cuda.device(q.device):
        lib = load()
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
                dk.data_ptr(), dv.data_ptr(), Z, Hq, Hkv, Nq, Nkv, D, *[ctypes.byref(x) for x in st], float(scale),
                int(bool(causal)), dt)
        ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size(), ctypes.c_void_p(stream.cuda_stream))
        if opt is None:
            rc, name = lib.fa_bwd(*args, *ws), "fa_bwd"
        else:
            rc, name = lib.fa_bwd_ex(*args, ctypes.byref(opt), *ws), "fa_bwd_ex"
    if rc != FA_OK:
        raise FaError(rc, name)
    return dq, dk, dv


def fa_fwd_splitkv_workspace_size(D: int, device=None) -> int:
    """Workspace bytes fa_fwd_splitkv needs for head dim D on `device` (default: current)."""
    import torch

    n = ctypes.c_size_t(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        rc = load().fa_fwd_splitkv_workspace_size(int(D), ctypes.byref(n))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv_workspace_size")
    return n.value


def fa_fwd_splitkv_workspace_size_for(D: int, num_sms: int) -> int:
    """Workspace bytes fa_fwd_splitkv needs for head dim D on a device of num_sms SMs (host only)."""
    n = ctypes.c_size_t(0)
    rc = load().fa_fwd_splitkv_workspace_size_for(int(D), int(num_sms), ctypes.byref(n))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv_workspace_size_for")
    return n.value


def workspace_for(D: int, device=None):
    """A uint8 CUDA tensor big enough to serve as fa_fwd_splitkv's workspace for head dim D."""
    import torch

    device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    return torch.empty(fa_fwd_splitkv_workspace_size(D, device), dtype=torch.uint8, device=device)


def fa_fwd_splitkv(q, k, v, o=None, lse=None, *, scale: float | None = None, causal: bool = False,
                   workspace=None, stream=None, want_lse: bool = True):
    """fa_fwd with the key blocks of all query tiles cut into one equal range per SM.

    Same arguments and results as fa_fwd, plus `workspace`: a CUDA uint8
    tensor of at least fa_fwd_splitkv_workspace_size(D) bytes (256-byte
    aligned, as torch allocations are); one is allocated when omitted.
    """
    import torch

    o, lse, dt, scale, stream, args, st = _prepare(q, k, v, o, lse, scale, want_lse, stream)
    if workspace is None:
        workspace = workspace_for(q.shape[3], q.device)
    with torch.cuda.device(q.device):
        rc = load().fa_fwd_splitkv(*args, *[ctypes.byref(x) for x in st], scale, int(bool(causal)), dt,
                                   workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                   ctypes.c_void_p(stream.cuda_stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv")
    return o, lse


def fa_fwd_splitkv_noalloc(q, k, v, o, lse=None, *, scale: float | None = None, causal: bool = False,
                           stream=None):
    """fa_fwd_splitkv working in the library's fixed device array instead of a workspace.

    The C entry point allocates nothing; so that this wrapper does not either,
    the caller passes the output `o` (and optionally `lse`).  Calls whose work
    may overlap on the GPU share the array and must be ordered (one stream).
    """
    import torch

    if o is None:
        raise ValueError("fa_fwd_splitkv_noalloc needs a preallocated output o")
    o, lse, dt, scale, stream, args, st = _prepare(q, k, v, o, lse, scale, False, stream)
    with torch.cuda.device(q.device):
        rc = load().fa_fwd_splitkv_noalloc(*args, *[ctypes.byref(x) for x in st], scale, int(bool(causal)), dt,
                                           ctypes.c_void_p(stream.cuda_stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv_noalloc")
    return o, lse


def fa_lse_merge(o_parts, lse_parts, o=None, lse=None, *, stream=None, want_lse: bool = True):
    """Combine results over disjoint key sets by their log-sum-exps (libfa's fa_lse_merge).

    o_parts: sequence of (Z, H, N, D) fp16/bf16 CUDA tensors sharing one
    layout; lse_parts: matching contiguous (Z, H, N) fp32 tensors.  Returns
    (o, lse) for the union of the key sets, without synchronising.
    """
    import torch

    n = len(o_parts)
    if n != len(lse_parts) or not 1 <= n <= FA_MERGE_MAX_PARTS:
        raise ValueError(f"need 1..{FA_MERGE_MAX_PARTS} matching O and lse parts")
    o0 = o_parts[0]
    Z, H, N, D = o0.shape
    dt = _dtype_code(o0)
    for x, l in zip(o_parts, lse_parts):
        if tuple(x.shape) != (Z, H, N, D) or x.dtype != o0.dtype or x.stride() != o0.stride():
            raise ValueError("O parts must share shape, dtype and strides")
        if l.dtype != torch.float32 or tuple(l.shape) != (Z, H, N) or not l.is_contiguous():
            raise ValueError("lse parts must be contiguous float32 (Z, H, N) tensors")
    if o is None:
        o = torch.empty((Z, H, N, D), dtype=o0.dtype, device=o0.device)
    if lse is None and want_lse:
        lse = torch.empty((Z, H, N), dtype=torch.float32, device=o0.device)
    if stream is None:
        stream = torch.cuda.current_stream(o0.device)
    optr = (ctypes.c_void_p * n)(*[x.data_ptr() for x in o_parts])
    lptr = (ctypes.c_void_p * n)(*[l.data_ptr() for l in lse_parts])
    sp, so = _strides(o0), _strides(o)
    with torch.cuda.device(o0.device):
        rc = load().fa_lse_merge(n, optr, lptr, Z, H, N, D, ctypes.byref(sp), o.data_ptr(),
                                 lse.data_ptr() if lse is not None else None, ctypes.byref(so), dt,
                                 ctypes.c_void_p(stream.cuda_stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_lse_merge")
    return o, lse


def fa_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None, Z: int, Hq: int, Hkv: int,
               Nq: int, Nkv: int, D: int, sq, sk, sv, so, scale: float, causal: bool, dtype: int,
               stream_handle: int = 0) -> int:
    """The C entry point with raw pointers and (b, h, n, d) stride tuples; returns the status code."""
    st = [fa_strides(*s) if s is not None else None for s in (sq, sk, sv, so)]
    refs = [ctypes.byref(s) if s is not None else None for s in st]
    return load().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, Z, Hq, Hkv, Nq, Nkv, D, *refs, float(scale),
                         int(causal), int(dtype), ctypes.c_void_p(stream_handle))


def fa_fwd_splitkv_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None, Z: int, Hq: int,
                       Hkv: int, Nq: int, Nkv: int, D: int, sq, sk, sv, so, scale: float, causal: bool, dtype: int,
                       ws_ptr: int | None, ws_bytes: int, stream_handle: int = 0) -> int:
    """fa_fwd_splitkv with raw pointers and (b, h, n, d) stride tuples; returns the status code."""
    st = [fa_strides(*s) if s is not None else None for s in (sq, sk, sv, so)]
    refs = [ctypes.byref(s) if s is not None else None for s in st]
    return load().fa_fwd_splitkv(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, Z, Hq, Hkv, Nq, Nkv, D, *refs, float(scale),
                                 int(causal), int(dtype), ws_ptr, int(ws_bytes), ctypes.c_void_p(stream_handle))


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


def fa_fwd_schedule(Z: int, Hq: int, Hkv: int, Nq: int, Nkv: int, D: int, causal: bool, *, splitkv: bool = False,
                    num_sms: int, l2_bytes: int) -> dict:
    """Host-only (no CUDA call): the schedule fa_fwd (or fa_fwd_splitkv) picks for contiguous BNSD
    tensors on a device with num_sms SMs and l2_bytes of L2 -- grid, split, gqa_packed, head_group,
    alternate, tiles, kv_blocks, busiest_blocks, softmax_chains, cta_pairs (libfa's fa_fwd_schedule)."""
    info = fa_fwd_schedule_info()
    rc = load().fa_fwd_schedule(Z, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), int(bool(splitkv)), num_sms, l2_bytes,
                                ctypes.byref(info))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_schedule")
    return {name: getattr(info, name) for name, _ in fa_fwd_schedule_info._fields_}


def fa_debug_set_wait_limit_ms(ms: float) -> None:
    load().fa_debug_set_wait_limit_ms(float(ms))


def fa_debug_inject_stall(enable: bool) -> None:
    load().fa_debug_inject_stall(int(bool(enable)))


def fa_debug_exp2(x, y=None, stream=None):
    """The softmax kernels' polynomial exponential on a CUDA float32 tensor (a test hook); returns y."""
    import torch

    if x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    y = torch.empty_like(x) if y is None else y
    stream = torch.cuda.current_stream(x.device) if stream is None else stream
    with torch.cuda.device(x.device):
        rc = load().fa_debug_exp2(x.data_ptr(), y.data_ptr(), x.numel(), ctypes.c_void_p(stream.cuda_stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_debug_exp2")
    return y


def fa_debug_force_chains(mode: int) -> None:
    """Which kernel runs whole tiles of D <= 128: 0 by shape (default), 1 two softmax chains, 2 one."""
    load().fa_debug_force_chains(int(mode))


def fa_debug_force_pair(mode: int) -> None:
    """Whether whole tiles of D = 128 run on CTA pairs: 0 default (no), 1 wherever they apply, 2 never."""
    load().fa_debug_force_pair(int(mode))


def fa_debug_force_split(mode: int) -> None:
    """fa_fwd_splitkv's choice: 0 by shape (default), 1 always cut key ranges, 2 never."""
    load().fa_debug_force_split(int(mode))
