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
    (dict(scale=3.0e38), fa.FA_ERR_INVALID_ARG),   # scale * log2(e) overflows fp32
    (dict(scale=-3.0e38), fa.FA_ERR_INVALID_ARG),
    (dict(D=48), fa.FA_ERR_UNSUPPORTED),
    (dict(D=512), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=2), fa.FA_ERR_UNSUPPORTED),
    (dict(ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(ptr=0x10008), fa.FA_ERR_ALIGNMENT),
    (dict(lse=0x10002), fa.FA_ERR_ALIGNMENT),
])
def test_argument_errors(lib, kw, code):
    assert _call(**kw) == code


@pytest.mark.parametrize("scale", [0.0, -0.0, -0.1, -8.0, 1e-40, -1e-40, 2.0e38, -2.0e38])
def test_every_finite_scale_passes_validation(lib, scale):
    # "1/sqrt(D) or a custom value" ("Write Triton Attention Kernel", Inputs 4):
    # zero, negative and subnormal scales are valid.  An empty problem (Z = 0)
    # returns FA_OK right after validation, before any device call.
    assert _call(Z=0, scale=scale) == fa.FA_OK
    assert _call(Z=0, scale=float("nan")) == fa.FA_ERR_INVALID_ARG


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


def test_bwd_ex_option_errors_on_the_host(lib):
    s = fa.fa_strides(2 * 64 * 64, 64 * 64, 64, 1)
    kv = fa.fa_strides(64 * 64, 64 * 64, 64, 1)

    def call(D=64, **kw):
        opt = fa.fa_fwd_options(kw.get("wl", -1), kw.get("wr", -1), kw.get("alibi"), kw.get("cq"), kw.get("ck"),
                                kw.get("maxq", 0), kw.get("maxk", 0))
        t = 0x10000
        return lib.fa_bwd_ex(t, t, t, t, t, t, t, t, t, 1, 2, 1, 64, 64, D, *[ctypes.byref(x) for x in (s, kv, kv, s, s, s, kv, kv)],
                             0.125, 0, 0, ctypes.byref(opt), t, 1 << 20, None)
    assert call(wl=-2) == fa.FA_ERR_INVALID_ARG
    assert call(cq=0x1000) == fa.FA_ERR_INVALID_ARG          # only one offset array
    assert call(ck=0x1000) == fa.FA_ERR_INVALID_ARG
    assert call(cq=0x1000, ck=0x2000, maxq=-1) == fa.FA_ERR_INVALID_ARG
    assert call(cq=0x1000, ck=0x2000, maxk=-1) == fa.FA_ERR_INVALID_ARG
    assert call(cq=0x1002, ck=0x2000, maxq=8) == fa.FA_ERR_ALIGNMENT
    assert call(cq=0x1000, ck=0x2001, maxq=8) == fa.FA_ERR_ALIGNMENT
    assert call(alibi=0x1001) == fa.FA_ERR_ALIGNMENT


# ---- fa_fwd_schedule: the forward's schedule, host-only -------------------
# An independent statement of the documented whole-tile orders: non-causal
# tiles head-major; causal tiles in groups of head_group heads, each group
# from the last query block to the first with its heads innermost; tile t of
# round r = t // grid goes to CTA t - r * grid, or to grid - 1 - (t - r * grid)
# when the rounds alternate and r is odd.  The busiest CTA's key blocks must
# equal the planner's.

GB300_SMS, GB300_L2 = 152, 126 * 2 ** 20


def _tile_blocks(mb, Nq, Nkv, bn, causal):
    tk = -(-Nkv // bn)
    if not causal:
        return tk
    last_row = min(mb * 128 + 128, Nq) - 1
    return min(tk, last_row // bn + 1)


def _busiest(Z, Hq, Nq, Nkv, bn, causal, grid, head_group, alternate):
    heads, tq = Z * Hq, -(-Nq // 128)
    if causal:
        order = []
        for g0 in range(0, heads, head_group):
            gc = min(head_group, heads - g0)
            for mb in reversed(range(tq)):
                order += [_tile_blocks(mb, Nq, Nkv, bn, True)] * gc
    else:
        order = [_tile_blocks(0, Nq, Nkv, bn, False)] * (heads * tq)
    loads = [0] * grid
    for t, blocks in enumerate(order):
        r, k = divmod(t, grid)
        loads[grid - 1 - k if (alternate and r % 2) else k] += blocks
    return max(loads)


def _pair_units(Z, Hq, Hkv, Nq):
    """CTA-pair kernel: (mode, virtual heads, virtual query blocks); mode 1 pairs the query
    heads 2k, 2k + 1 of a GQA group, mode 2 the query blocks 2m, 2m + 1 of one head."""
    tq = -(-Nq // 128)
    if (Hq // Hkv) % 2 == 0:
        return 1, Z * Hq // 2, tq
    return 2, Z * Hq, -(-tq // 2)


def _pair_busiest(Z, Hq, Hkv, Nq, Nkv, causal, clusters, head_group, alternate):
    mode, vheads, vtq = _pair_units(Z, Hq, Hkv, Nq)
    tq = -(-Nq // 128)

    def blocks(vmb):  # both tiles of a unit visit the key blocks of the later one
        mb = vmb if mode == 1 else min(2 * vmb + 1, tq - 1)
        return _tile_blocks(mb, Nq, Nkv, 128, causal)

    if causal:
        order = []
        for g0 in range(0, vheads, head_group):
            gc = min(head_group, vheads - g0)
            for vmb in reversed(range(vtq)):
                order += [blocks(vmb)] * gc
    else:
        order = [blocks(vmb) for _ in range(vheads) for vmb in range(vtq)]
    loads = [0] * clusters
    for t, b in enumerate(order):
        r, k = divmod(t, clusters)
        loads[clusters - 1 - k if (alternate and r % 2) else k] += b
    return max(loads)


@pytest.mark.parametrize("shape", [
    (4, 16, 16, 1024, 1024, 128, False),   # the bench workload, both masks
    (4, 16, 16, 1024, 1024, 128, True),
    (8, 16, 16, 2048, 2048, 256, True),    # long causal tiles (64-key blocks): alternating rounds
    (128, 8, 8, 1024, 1024, 128, True),    # 1024 heads: several head groups
    (1, 32, 8, 8192, 8192, 128, True),
    (1, 32, 8, 32768, 32768, 128, True),   # GQA: groups of 8 query heads
    (1, 32, 8, 8192, 8192, 128, False),
    (2, 3, 1, 4000, 4000, 128, True),      # CTA pairs of query blocks, odd block count
    (2, 3, 1, 1000, 300, 64, True),        # odd sizes, fewer tiles than SMs
    (3, 5, 5, 130, 4000, 32, False),
])
@pytest.mark.parametrize("pairs", [False, True], ids=["one_sm", "cta_pairs"])
def test_schedule_matches_the_documented_order(shape, pairs):
    import exact_attention_44_gb300 as fa
    Z, Hq, Hkv, Nq, Nkv, D, causal = shape
    fa.fa_debug_force_pair(1 if pairs else 0)
    try:
        s = fa.fa_fwd_schedule(Z, Hq, Hkv, Nq, Nkv, D, causal, num_sms=GB300_SMS, l2_bytes=GB300_L2)
    finally:
        fa.fa_debug_force_pair(0)
    bn = 64 if D == 256 else 128
    heads, tq, tk = Z * Hq, -(-Nq // 128), -(-Nkv // bn)
    assert s["split"] == 0 and s["gqa_packed"] == 0
    long_tiles = s["kv_blocks"] >= 16 * s["tiles"]
    # head dims up to 64 with long tiles (>= 16 key blocks a tile on average)
    # run two softmax chains, the rest one; CTA pairs (D = 128) only when asked
    assert s["cta_pairs"] == int(pairs and D == 128)
    assert s["softmax_chains"] == (2 if (D <= 64 and long_tiles) or s["cta_pairs"] else 1)
    assert s["tiles"] == heads * tq
    if s["cta_pairs"]:
        mode, vheads, vtq = _pair_units(Z, Hq, Hkv, Nq)
        clusters = min(vheads * vtq, GB300_SMS // 2)
        assert s["grid"] == 2 * clusters
        assert s["kv_blocks"] == Z * Hq * sum(_tile_blocks(mb, Nq, Nkv, bn, causal) for mb in range(tq))
        alternate = int(causal and long_tiles)
        assert s["alternate"] == alternate
        assert s["kv_blocks"] == Z * Hq * sum(_tile_blocks(mb, Nq, Nkv, bn, causal) for mb in range(tq))
        if causal:
            per_kv = (Hq // Hkv) // 2 if mode == 1 else Hq // Hkv
            kv_heads = max(1, (GB300_L2 // 3) // (Nkv * D * 4))
            want = min(vheads, max(kv_heads * per_kv, -(-4 * clusters // vtq)))
            assert s["head_group"] == want
        assert s["busiest_blocks"] == _pair_busiest(Z, Hq, Hkv, Nq, Nkv, causal, clusters, s["head_group"],
                                                    alternate)
        return
    assert s["grid"] == min(heads * tq, GB300_SMS)
    assert s["kv_blocks"] == Z * Hq * sum(_tile_blocks(mb, Nq, Nkv, bn, causal) for mb in range(tq))
    if causal:
        # a group's K/V within a third of L2, at least four rounds of tiles, at most every head
        kv_heads = max(1, (GB300_L2 // 3) // (Nkv * D * 4))
        want = min(heads, max(kv_heads * (Hq // Hkv), -(-4 * GB300_SMS // tq)))
        assert s["head_group"] == want
        # rounds alternate only for long tiles (>= 16 key blocks a tile on average)
        assert s["alternate"] == int(s["kv_blocks"] >= 16 * s["tiles"])
    else:
        assert s["alternate"] == 0
    assert s["busiest_blocks"] == _busiest(Z, Hq, Nq, Nkv, bn, causal, s["grid"], s["head_group"], s["alternate"])


def test_schedule_known_values():
    import exact_attention_44_gb300 as fa
    kw = dict(num_sms=GB300_SMS, l2_bytes=GB300_L2)
    # the Z4 H16 N1024 workload: 512 tiles on 152 CTAs, 4 tiles of 8 blocks on the busiest;
    # causal: heaviest first, round-robin, 19 blocks on the busiest (15.2 on average)
    assert fa.fa_fwd_schedule(4, 16, 16, 1024, 1024, 128, False, **kw)["busiest_blocks"] == 32
    c = fa.fa_fwd_schedule(4, 16, 16, 1024, 1024, 128, True, **kw)
    assert (c["head_group"], c["alternate"], c["busiest_blocks"], c["softmax_chains"]) == (64, 0, 19, 1)
    # the two-chain kernel runs the same schedule
    try:
        fa.fa_debug_force_chains(1)
        c = fa.fa_fwd_schedule(4, 16, 16, 1024, 1024, 128, True, **kw)
        assert (c["head_group"], c["alternate"], c["busiest_blocks"], c["softmax_chains"]) == (64, 0, 19, 2)
    finally:
        fa.fa_debug_force_chains(0)
    # head dims up to 64 with long tiles take two chains
    assert fa.fa_fwd_schedule(8, 16, 16, 2048, 2048, 64, False, **kw)["softmax_chains"] == 2
    assert fa.fa_fwd_schedule(8, 16, 16, 2048, 2048, 64, True, **kw)["softmax_chains"] == 1
    # D = 128: one SM per tile unless CTA pairs are asked for; then 1024 units
    # of two tiles on 76 clusters, 14 units of 64 key blocks on the busiest
    c = fa.fa_fwd_schedule(1, 32, 8, 8192, 8192, 128, False, **kw)
    assert (c["cta_pairs"], c["softmax_chains"], c["grid"]) == (0, 1, 152)
    try:
        fa.fa_debug_force_pair(1)
        c = fa.fa_fwd_schedule(1, 32, 8, 8192, 8192, 128, False, **kw)
        assert (c["cta_pairs"], c["softmax_chains"], c["grid"], c["busiest_blocks"]) == (1, 2, 152, 14 * 64)
        # never at other head dims or with cut key ranges
        assert fa.fa_fwd_schedule(1, 32, 8, 8192, 8192, 64, False, **kw)["cta_pairs"] == 0
    finally:
        fa.fa_debug_force_pair(0)
    # alternating rounds: 236 blocks on the busiest CTA instead of 284
    assert fa.fa_fwd_schedule(8, 16, 16, 2048, 2048, 256, True, **kw)["busiest_blocks"] == 236


def test_schedule_split_and_gqa_packing():
    import exact_attention_44_gb300 as fa
    kw = dict(num_sms=GB300_SMS, l2_bytes=GB300_L2)
    # a decode row: the 4 query heads of a group run as one head of 4 rows,
    # and the 8 resulting tiles are cut into one key range per SM
    d = fa.fa_fwd_schedule(1, 32, 8, 1, 32768, 128, False, splitkv=True, **kw)
    assert d["gqa_packed"] == 1 and d["tiles"] == 8 and d["split"] == 1 and d["grid"] == GB300_SMS
    assert d["busiest_blocks"] == -(-8 * 256 // GB300_SMS)
    # fa_fwd never cuts; through fa_fwd_splitkv the bench workload stays whole
    # (32 key blocks on the busiest CTA against 27 for an even cut: under the
    # 2048-key threshold)
    assert fa.fa_fwd_schedule(1, 32, 8, 1, 32768, 128, False, **kw)["split"] == 0
    assert fa.fa_fwd_schedule(4, 16, 16, 1024, 1024, 128, False, splitkv=True, **kw)["split"] == 0
    # and 16 or more tiles per SM are never cut
    assert fa.fa_fwd_schedule(1, 38, 38, 8192, 8192, 128, False, splitkv=True, **kw)["split"] == 0
    # causal rows are never packed (a row's keys depend on its position)
    assert fa.fa_fwd_schedule(1, 32, 8, 64, 4096, 128, True, **kw)["gqa_packed"] == 0
    # the test hook forces either choice
    try:
        fa.fa_debug_force_split(1)
        assert fa.fa_fwd_schedule(4, 16, 16, 1024, 1024, 128, False, splitkv=True, **kw)["split"] == 1
        fa.fa_debug_force_split(2)
        assert fa.fa_fwd_schedule(1, 32, 8, 1, 32768, 128, False, splitkv=True, **kw)["split"] == 0
    finally:
        fa.fa_debug_force_split(0)


def test_schedule_argument_errors():
    import exact_attention_44_gb300 as fa
    for kw in (dict(num_sms=0, l2_bytes=GB300_L2), dict(num_sms=GB300_SMS, l2_bytes=0)):
        with pytest.raises(fa.FaError) as e:
            fa.fa_fwd_schedule(1, 1, 1, 128, 128, 64, False, **kw)
        assert e.value.code == fa.FA_ERR_INVALID_ARG
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_schedule(1, 3, 2, 128, 128, 64, False, num_sms=GB300_SMS, l2_bytes=GB300_L2)
    assert e.value.code != fa.FA_OK


def _noalloc_scratch_bytes():
    # the size the header gives the no-allocation entry point's fixed array
    import re
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa.h")).read()
    m = re.search(r"#define FA_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", text)
    assert m, "FA_NOALLOC_SCRATCH_BYTES not found in include/fa.h"
    return int(m.group(1)) * int(m.group(2)) * int(m.group(3))


def test_noalloc_array_covers_the_documented_sm_count(lib):
    # the header promises two D = 256 partial slots per SM on GPUs of up to
    # 159 SMs (152 on GB300), and that a device needing more is rejected:
    # the array must hold 159 SMs' worth and not 160
    size = _noalloc_scratch_bytes()
    assert fa.fa_fwd_splitkv_workspace_size_for(256, 159) <= size < fa.fa_fwd_splitkv_workspace_size_for(256, 160)
    # smaller head dims need less per slot, so 152 SMs fit at every D
    for D in (16, 32, 64, 128, 256):
        assert fa.fa_fwd_splitkv_workspace_size_for(D, 152) <= size
    # the slot layout: 128 x D fp32 values and 128 log-sum-exps, padded to 256 bytes
    for D in (16, 64, 256):
        slot = ((128 * D + 128) * 4 + 255) // 256 * 256
        assert fa.fa_fwd_splitkv_workspace_size_for(D, 7) == 2 * 7 * slot
    with pytest.raises(fa.FaError):
        fa.fa_fwd_splitkv_workspace_size_for(48, 152)
    with pytest.raises(fa.FaError):
        fa.fa_fwd_splitkv_workspace_size_for(128, 0)


@pytest.mark.parametrize("D", [16, 32, 64, 128, 256])
def test_bwd_workspace_every_head_dim(lib, D):
    # lse2 and Delta per query row, padded to whole 128-row blocks and 256 bytes
    Z, Hq, Nq = 2, 3, 300
    rows = Z * Hq * -(-Nq // 128) * 128 * 4
    assert fa.fa_bwd_workspace_size(Z, Hq, Nq, D) == 2 * (-(-rows // 256) * 256)
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd_workspace_size(Z, Hq, Nq, 96)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED


def test_autograd_layer_imports_without_a_gpu():
    # the autograd functions are defined (torch imported) without any CUDA call
    import exact_attention_44_gb300 as fa
    from exact_attention_44_gb300 import autograd
    assert callable(fa.attention) and callable(fa.attention_varlen)
    assert issubclass(autograd._Attention, __import__("torch").autograd.Function)
    assert autograd._plain((-1, -1), None) and not autograd._plain((8, -1), None)
