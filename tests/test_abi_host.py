"""libfa on the host: it builds, exports every symbol include/fa.h declares, and
rejects bad arguments before touching CUDA.  No GPU needed (none of these
calls reaches a kernel launch)."""
import ctypes
import json
import math
import os
import re

import pytest

import exact_attention_44_gb300 as fa
from exact_attention_44_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ("fa_fwd", "fa_status_string", "fa_device_status", "fa_fwd_plan"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) == set(_binding._SIGNATURES)


def test_status_strings(lib):
    assert fa.fa_status_string(0) == "FA_OK"
    assert fa.fa_status_string(5) == "FA_ERR_DEVICE_TIMEOUT"
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


# ------------------------------------------------------------- plan (host) ---

def test_causal_tile_count_matches_the_page(lib):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "causal_tile_count.json")))
    n = g["tiles_per_side"] * 128
    nc = fa.fa_fwd_plan(1, 1, 1, n, n, 128, False)
    c = fa.fa_fwd_plan(1, 1, 1, n, n, 128, True)
    assert nc["kv_blocks"] == g["noncausal_tiles"]
    assert c["kv_blocks"] == g["causal_tiles"]
    assert 1 - c["kv_blocks"] / nc["kv_blocks"] == pytest.approx(g["skipped_fraction"])


@pytest.mark.parametrize("T", [1, 2, 3, 8, 16, 256])
def test_causal_block_count_is_triangular(lib, T):
    p = fa.fa_fwd_plan(2, 3, 1, 128 * T, 128 * T, 64, True)
    assert p["kv_blocks"] == 2 * 3 * T * (T + 1) // 2
    assert p["tiles"] == 2 * 3 * T


def test_plan_d256_uses_64_key_blocks(lib):
    p = fa.fa_fwd_plan(1, 1, 1, 256, 256, 256, True)
    assert p["block_n"] == 64
    # q tile 0 covers rows 0..127 -> key blocks 0,1; tile 1 rows 128..255 -> blocks 0..3
    assert p["kv_blocks"] == 2 + 4


def test_plan_ragged_and_cross(lib):
    p = fa.fa_fwd_plan(1, 32, 8, 1000, 8192, 128, False, num_sms=152)
    assert p["tiles"] == 32 * 8 and p["kv_blocks"] == 32 * 8 * 64 and p["grid"] == 152
    # causal, Nq > Nkv: every tile stops at the last key block
    p = fa.fa_fwd_plan(1, 1, 1, 1000, 300, 64, True)
    assert p["kv_blocks"] == sum(min(3, (min(128 * mb + 128, 1000) - 1) // 128 + 1) for mb in range(8))
    assert p["smem_bytes"] <= 227 * 1024


# -------------------------------------------------- argument validation -----

def _call(Z=1, Hq=2, Hkv=1, Nq=64, Nkv=64, D=64, scale=0.125, causal=0, dtype=0, ptr=0x10000, strides=None,
          lse=None):
    if strides is None:
        s = (Hq * Nq * D, Nq * D, D, 1)
        skv = (Hkv * Nkv * D, Nkv * D, D, 1)
        strides = (s, skv, skv, s)
    return fa.fa_fwd_raw(ptr, ptr, ptr, ptr, lse, Z, Hq, Hkv, Nq, Nkv, D, *strides, scale, causal, dtype)


@pytest.mark.parametrize("kw,code", [
    (dict(Z=-1), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=-5), fa.FA_ERR_INVALID_ARG),
    (dict(Hkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), fa.FA_ERR_INVALID_ARG),
    (dict(Nkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-0.1), fa.FA_ERR_INVALID_ARG),
    (dict(D=48), fa.FA_ERR_UNSUPPORTED),
    (dict(D=512), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=2), fa.FA_ERR_UNSUPPORTED),
    (dict(ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(ptr=0x10008), fa.FA_ERR_ALIGNMENT),
    (dict(lse=0x10002), fa.FA_ERR_ALIGNMENT),
])
def test_argument_errors(lib, kw, code):
    assert _call(**kw) == code


def test_stride_errors(lib):
    good = (2 * 64 * 64, 64 * 64, 64, 1)
    kv = (64 * 64, 64 * 64, 64, 1)
    assert _call(strides=((good[0], good[1], good[2], 2), kv, kv, good)) == fa.FA_ERR_ALIGNMENT   # d-stride
    assert _call(strides=(good, (kv[0], kv[1], 60, 1), kv, good)) == fa.FA_ERR_ALIGNMENT          # n-stride % 8
    assert _call(strides=(good, kv, kv, (good[0], -good[1], good[2], 1))) == fa.FA_ERR_ALIGNMENT  # negative
    assert _call(strides=(good, kv, kv, None)) == fa.FA_ERR_INVALID_ARG                          # missing


def test_empty_problem_is_a_noop(lib):
    # nothing to compute: FA_OK without touching any pointer or the device
    assert fa.fa_fwd_raw(0, 0, 0, 0, None, 0, 2, 1, 64, 64, 64, None, None, None, None, 0.1, 0, 0) == fa.FA_OK
    assert fa.fa_fwd_raw(0, 0, 0, 0, None, 1, 2, 1, 0, 64, 64, None, None, None, None, 0.1, 1, 1) == fa.FA_OK
    assert _call(Nq=0, Nkv=0) == fa.FA_OK


def test_no_cpu_fallback_without_a_device(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    # a well-formed call with no GPU fails loudly instead of computing anything
    assert _call() == fa.FA_ERR_CUDA
    with pytest.raises(Exception):
        q = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
        fa.fa_fwd(q, q, q)


def test_binding_never_imports_the_oracle():
    import subprocess
    import sys
    code = ("import sys, exact_attention_44_gb300 as m; m.load(); "
            "bad = [k for k in sys.modules if k == 'oracle' or k.startswith('oracle.')]; "
            "assert not bad, bad")
    subprocess.run([sys.executable, "-c", code], check=True, cwd=ROOT)


# ------------------------------------------------ split-KV and merge (host) ---

def test_splitkv_rejects_missing_or_misaligned_workspace(lib):
    s = (2 * 64 * 64, 64 * 64, 64, 1)
    kv = (64 * 64, 64 * 64, 64, 1)
    args = (0x10000, 0x10000, 0x10000, 0x10000, None, 1, 2, 1, 64, 64, 64, s, kv, kv, s, 0.125, 0, 0)
    assert fa.fa_fwd_splitkv_raw(*args, None, 1 << 30) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_splitkv_raw(*args, 0x10010, 1 << 30) == fa.FA_ERR_WORKSPACE
    # argument errors come first, as in fa_fwd
    bad = list(args)
    bad[10] = 48
    assert fa.fa_fwd_splitkv_raw(*bad, None, 0) == fa.FA_ERR_UNSUPPORTED
    # nothing to compute: no workspace needed
    empty = list(args)
    empty[8] = 0
    assert fa.fa_fwd_splitkv_raw(*empty, None, 0) == fa.FA_OK


def _merge_raw(lib, nparts=2, Z=1, H=2, N=64, D=64, optr=0x10000, lptr=0x20000, out=0x30000, dtype=0):
    s = fa.fa_strides(H * N * D, N * D, D, 1)
    o_arr = (ctypes.c_void_p * max(nparts, 1))(*([optr] * max(nparts, 1)))
    l_arr = (ctypes.c_void_p * max(nparts, 1))(*([lptr] * max(nparts, 1)))
    return lib.fa_lse_merge(nparts, o_arr, l_arr, Z, H, N, D, ctypes.byref(s), out, None, ctypes.byref(s), dtype,
                            None)


@pytest.mark.parametrize("kw,code", [
    (dict(nparts=0), fa.FA_ERR_INVALID_ARG),
    (dict(nparts=17), fa.FA_ERR_INVALID_ARG),
    (dict(N=-1), fa.FA_ERR_INVALID_ARG),
    (dict(D=48), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=2), fa.FA_ERR_UNSUPPORTED),
    (dict(optr=0x10008), fa.FA_ERR_ALIGNMENT),
    (dict(lptr=0x20002), fa.FA_ERR_ALIGNMENT),
    (dict(lptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(out=0), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_OK),
])
def test_merge_argument_errors(lib, kw, code):
    assert _merge_raw(lib, **kw) == code


def test_fwd_ex_option_errors_on_the_host(lib):
    s = fa.fa_strides(2 * 64 * 64, 64 * 64, 64, 1)
    kv = fa.fa_strides(64 * 64, 64 * 64, 64, 1)

    def call(**kw):
        opt = fa.fa_fwd_options(kw.get("wl", -1), kw.get("wr", -1), kw.get("alibi"), kw.get("cq"), kw.get("ck"),
                                kw.get("maxq", 0))
        return lib.fa_fwd_ex(0x10000, 0x10000, 0x10000, 0x10000, None, 1, 2, 1, 64, 64, 64, ctypes.byref(s),
                             ctypes.byref(kv), ctypes.byref(kv), ctypes.byref(s), 0.125, 0, 0, ctypes.byref(opt), None)
    assert call(wl=-2) == fa.FA_ERR_INVALID_ARG
    assert call(wr=-5) == fa.FA_ERR_INVALID_ARG
    assert call(cq=0x1000) == fa.FA_ERR_INVALID_ARG          # only one offset array
    assert call(cq=0x1000, ck=0x2000, maxq=-1) == fa.FA_ERR_INVALID_ARG
    assert call(cq=0x1002, ck=0x2000, maxq=8) == fa.FA_ERR_ALIGNMENT
    assert call(alibi=0x1001) == fa.FA_ERR_ALIGNMENT
