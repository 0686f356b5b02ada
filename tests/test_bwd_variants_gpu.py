"""GPU parity of fa_bwd_ex (gradients of the window / ALiBi forward, on dense
(Z, H, N, D) tensors and on packed variable-length sequences) against the fp64
oracle's attention_bwd_ex.

The forward's O and lse come from fa_fwd_ex with the same options (the GPU's
own chain, as for fa_bwd); the oracle differentiates the definition from Q, K,
V and dO.  Tolerance as for fa_bwd (tests/test_bwd_gpu.py): 4 unit roundoffs
of the input type relative to the largest reference gradient.  Cases: each
window side alone and both, with and without the causal rule, ALiBi alone and
with a window, GQA, query and key lengths that differ (rows that keep no key:
dQ = 0), windows so narrow most blocks are skipped, the open window routed to
fa_bwd's kernel, and the head dim the variants do not cover; packed
sequences; and the bench's three variant workloads at full size, whole heads
(or sequences) against the oracle."""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from parity_util import to_device
from test_bwd_gpu import TOL_GRAD

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()


def run_bwd_ex(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype, causal, window, alibi, scale=None):
    import torch
    import exact_attention_44_gb300 as fa
    scale = 1 / math.sqrt(D) if scale is None else scale
    q, k, v = si.qkv(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    do = si.normals(seed + 1000, 0, q.size, dtype).reshape(q.shape)
    qt, kt, vt, dot = (to_device(x, dtype) for x in (q, k, v, do))
    slopes = None if alibi is None else torch.tensor(alibi, dtype=torch.float32, device="cuda")
    o, lse = fa.fa_fwd_ex(qt, kt, vt, scale=scale, causal=causal, window=window, alibi_slopes=slopes)
    dq, dk, dv = fa.fa_bwd_ex(qt, kt, vt, o, lse, dot, scale=scale, causal=causal, window=window, alibi_slopes=slopes)
    torch.cuda.synchronize()
    code, word = fa.fa_device_status()
    assert code == 0, f"device status {word:#x}"
    return (q, k, v, do, scale), (dq, dk, dv)


def check_bwd_ex(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype, causal, window=(-1, -1), alibi=None, scale=None):
    (q, k, v, do, scale), got = run_bwd_ex(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype, causal, window, alibi, scale)
    ref = oracle.attention_bwd_ex(q, k, v, do, dtype, scale, causal, window=window,
                                  alibi=None if alibi is None else np.asarray(alibi, dtype=np.float64))
    worst = {}
    for name, g, want in zip(("dq", "dk", "dv"), got, ref):
        g = g.double().cpu().numpy()
        assert np.all(np.isfinite(g)), f"{name}: non-finite"
        err = float(np.max(np.abs(g - want)))
        mag = float(np.max(np.abs(want)))
        worst[name] = (err, mag)
        assert err <= TOL_GRAD[dtype] * max(mag, 1e-3), f"{name}: max|d| = {err:.3e}, max|ref| = {mag:.3e}"
    return worst, got, ref


@pytest.mark.parametrize("window", [(64, 32), (100, -1), (-1, 50)])
@pytest.mark.parametrize("causal", [False, True])
def test_window_sides(window, causal):
    print(check_bwd_ex(301, 1, 2, 2, 300, 300, 64, "fp16", causal, window)[0])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_alibi(causal, dtype):
    print(check_bwd_ex(302, 2, 4, 2, 400, 400, 128, dtype, causal, alibi=[0.5, 0.25, 0.125, 0.0625])[0])


@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_alibi_with_window_head_dims(D):
    print(check_bwd_ex(303, 1, 4, 1, 333, 333, D, "bf16", True, window=(150, -1), alibi=[1.0, 0.3, 0.05, 0.0])[0])


@pytest.mark.parametrize("window", [(0, 0), (1, 1), (5, -1)])
def test_narrow_windows(window):
    print(check_bwd_ex(304, 1, 2, 1, 600, 600, 32, "fp16", False, window)[0])


def test_rows_that_keep_no_key():
    # causal, left window 10, 300 queries against 100 keys: rows 110.. keep none
    worst, (dq, _, _), _ = check_bwd_ex(305, 1, 2, 2, 300, 100, 64, "bf16", True, window=(10, -1))
    assert float(dq[:, :, 110:].abs().max()) == 0.0


def test_keys_no_row_keeps():
    # right window 0, non-causal, 100 queries against 400 keys: keys 101.. are kept by no row
    worst, (_, dk, dv), _ = check_bwd_ex(306, 1, 2, 2, 100, 400, 64, "fp16", False, window=(-1, 0))
    assert float(dk[:, :, 100:].abs().max()) == 0.0 and float(dv[:, :, 100:].abs().max()) == 0.0


def test_longer_windowed_causal_gqa():
    print(check_bwd_ex(307, 2, 8, 2, 2048, 2048, 128, "bf16", True, window=(512, -1), alibi=[0.02 * (h + 1) for h in range(8)])[0])


def test_open_window_is_the_plain_backward_bit_for_bit():
    import torch
    import exact_attention_44_gb300 as fa
    q, k, v = si.qkv(308, 1, 2, 2, 300, 300, 64, "bf16")
    do = si.normals(1308, 0, q.size, "bf16").reshape(q.shape)
    qt, kt, vt, dot = (to_device(x, "bf16") for x in (q, k, v, do))
    o, lse = fa.fa_fwd(qt, kt, vt, causal=True)
    plain = fa.fa_bwd(qt, kt, vt, o, lse, dot, causal=True)
    ex = fa.fa_bwd_ex(qt, kt, vt, o, lse, dot, causal=True, window=(10000, -1))
    torch.cuda.synchronize()
    for a, b in zip(plain, ex):
        assert torch.equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_256_window(causal):
    # the two-pass D = 256 kernel with window-bounded units, ragged lengths
    check_bwd_ex(440, 1, 4, 2, 300, 333, 256, "bf16", causal, window=(100, 40))


def test_head_dim_256_alibi_with_window():
    check_bwd_ex(441, 2, 4, 4, 257, 257, 256, "fp16", True, window=(150, -1), alibi=[0.5, 0.25, 0.125, 0.0625])


@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_256_varlen(causal):
    # packed sequences at D = 256: a sequence without queries, one without
    # keys, single rows, crossing and ragged blocks, rows past the last
    lens_q = [5, 0, 135, 60, 1, 129]
    lens_k = [7, 23, 0, 300, 1, 200]
    check_bwd_varlen(442, lens_q, lens_k, 4, 2, 256, "bf16", causal, extra_q=9, extra_k=4)


def test_head_dim_256_varlen_window_alibi():
    check_bwd_varlen(443, [200, 17, 260], [200, 300, 260], 4, 2, 256, "fp16", True, window=(50, -1),
                     alibi=[0.5, 0.25, 0.125, 0.0625])


# ---- packed variable-length sequences -------------------------------------
# Sequence z owns query rows cu_q[z] .. cu_q[z+1]-1 and key rows cu_k[z] ..
# cu_k[z+1]-1 and attends only to its own keys; the oracle composes the
# dense backward sequence by sequence.  The gradient buffers start filled
# with a sentinel: packed rows outside every sequence must keep it.

SENTINEL = 7.0


def _varlen_inputs(seed, lens_q, lens_k, Hq, Hkv, D, dtype, extra_q=0, extra_k=0):
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    tq, tk = int(cu_q[-1]) + extra_q, int(cu_k[-1]) + extra_k
    q = si.normals(seed, 0, Hq * tq * D, dtype).reshape(1, Hq, tq, D)
    k = si.normals(seed, q.size, Hkv * tk * D, dtype).reshape(1, Hkv, tk, D)
    v = si.normals(seed, q.size + k.size, Hkv * tk * D, dtype).reshape(1, Hkv, tk, D)
    do = si.normals(seed + 1000, 0, q.size, dtype).reshape(q.shape)
    return cu_q, cu_k, q, k, v, do


def check_bwd_varlen(seed, lens_q, lens_k, Hq, Hkv, D, dtype, causal, window=(-1, -1), alibi=None, thd=False,
                     extra_q=0, extra_k=0, max_seqlen_k=None):
    import torch
    import exact_attention_44_gb300 as fa
    cu_q, cu_k, q, k, v, do = _varlen_inputs(seed, lens_q, lens_k, Hq, Hkv, D, dtype, extra_q, extra_k)
    scale = 1 / math.sqrt(D)
    qt, kt, vt, dot = (to_device(x, dtype) for x in (q, k, v, do))
    if thd:  # (total, H, D) storage
        qt, kt, vt, dot = (x[0].permute(1, 0, 2).contiguous() for x in (qt, kt, vt, dot))
    slopes = None if alibi is None else torch.tensor(alibi, dtype=torch.float32, device="cuda")
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    o, lse = fa.fa_fwd_ex(qt, kt, vt, o=torch.zeros_like(qt), scale=scale, causal=causal, window=window,
                          alibi_slopes=slopes, cu_seqlens_q=cq, cu_seqlens_k=ck)
    dq, dk, dv = (torch.full_like(x, SENTINEL) for x in (qt, kt, vt))
    fa.fa_bwd_ex(qt, kt, vt, o, lse, dot, dq, dk, dv, scale=scale, causal=causal, window=window, alibi_slopes=slopes,
                 cu_seqlens_q=cq, cu_seqlens_k=ck, max_seqlen_k=max_seqlen_k)
    torch.cuda.synchronize()
    code, word = fa.fa_device_status()
    assert code == 0, f"device status {word:#x}"
    ref = oracle.attention_bwd_ex(q, k, v, do, dtype, scale, causal, window=window,
                                  alibi=None if alibi is None else np.asarray(alibi, dtype=np.float64),
                                  cu_q=cu_q, cu_k=cu_k)
    nq, nk = int(cu_q[-1]), int(cu_k[-1])
    got = []
    for name, g, want, n in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, (nq, nk, nk)):
        g = (g.permute(1, 0, 2).unsqueeze(0) if thd else g).double().cpu().numpy()
        assert np.all(g[:, :, n:] == SENTINEL), f"{name}: a packed row outside every sequence was written"
        g = g[:, :, :n]
        assert np.all(np.isfinite(g)), f"{name}: non-finite"
        err = float(np.max(np.abs(g - want[:, :, :n]))) if g.size else 0.0
        mag = float(np.max(np.abs(want[:, :, :n]))) if g.size else 0.0
        assert err <= TOL_GRAD[dtype] * max(mag, 1e-3), f"{name}: max|d| = {err:.3e}, max|ref| = {mag:.3e}"
        got.append(g)
    return cu_q, cu_k, got


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("thd", [False, True])
def test_varlen(causal, thd):
    # a sequence without queries (its keys: dK = dV = 0), one without keys
    # (its rows: dQ = 0), single rows, whole and ragged 128-row blocks, and
    # packed rows past the last sequence
    lens_q = [5, 0, 135, 60, 1, 300, 128, 129]
    lens_k = [7, 23, 0, 300, 1, 290, 128, 500]
    cu_q, cu_k, (dq, dk, dv) = check_bwd_varlen(400, lens_q, lens_k, 4, 2, 128, "bf16", causal, thd=thd,
                                                extra_q=10, extra_k=6)
    assert np.all(dk[:, :, cu_k[1]:cu_k[2]] == 0) and np.all(dv[:, :, cu_k[1]:cu_k[2]] == 0)
    assert np.all(dq[:, :, cu_q[2]:cu_q[3]] == 0)


def test_varlen_with_window_alibi_gqa():
    check_bwd_varlen(401, [200, 17, 260], [200, 300, 260], 8, 2, 64, "fp16", True, window=(50, -1),
                     alibi=[2.0 ** (-(i + 1)) for i in range(8)])


@pytest.mark.parametrize("D", [16, 32, 64])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_varlen_head_dims(D, dtype):
    check_bwd_varlen(402 + D, [33, 129, 256, 70], [40, 100, 300, 1], 2, 1, D, dtype, False, window=(-1, 40))


def test_varlen_window_both_sides_causal_alibi():
    check_bwd_varlen(420, [500, 64, 1, 383], [500, 64, 3, 383], 4, 4, 128, "bf16", True, window=(100, 30),
                     alibi=[0.5, 0.25, 0.125, 0.0625])


def test_varlen_key_bound_defaults_to_the_packed_total():
    # max_seqlen_k = 0: the kernel bounds each sequence's key blocks by the
    # packed total instead of the longest sequence; the gradients are the same
    import torch
    a = check_bwd_varlen(421, [100, 300], [260, 140], 2, 2, 64, "bf16", True)[2]
    b = check_bwd_varlen(421, [100, 300], [260, 140], 2, 2, 64, "bf16", True, max_seqlen_k=0)[2]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_varlen_longer_sequences():
    # a packed batch of 5.4K rows: sequences from 1 to 2000 rows, GQA 4:1
    check_bwd_varlen(422, [2000, 1, 1500, 129, 1800], [2000, 5, 1500, 700, 1800], 4, 1, 128, "bf16", True,
                     extra_q=3)


# ---- the bench's variant workloads at full size, whole heads ----------------
# A head's gradients depend on that head's Q, K, V, dO only (and a packed
# sequence's on its own rows), so the oracle differentiates whole heads (or
# sequences) of the full-size launch one at a time.

def _check_heads(q, k, v, do, got, dtype, scale, causal, heads, **opt):
    for z, h in heads:
        one_q = (slice(z, z + 1), slice(h, h + 1))
        ref = oracle.attention_bwd_ex(q[one_q], k[one_q], v[one_q], do[one_q], dtype, scale, causal, **opt)
        for name, g, want in zip(("dq", "dk", "dv"), got, ref):
            g = g[one_q].double().cpu().numpy()
            err, mag = float(np.max(np.abs(g - want))), float(np.max(np.abs(want)))
            assert err <= TOL_GRAD[dtype] * max(mag, 1e-3), f"head ({z}, {h}) {name}: {err:.3e} vs {mag:.3e}"


def test_full_size_window_whole_heads():
    # Z4 H16 N4096 D128 bf16, causal with a 512-key window
    Z, H, N, D, dtype, window = 4, 16, 4096, 128, "bf16", (512, 0)
    (q, k, v, do, scale), got = run_bwd_ex(430, Z, H, H, N, N, D, dtype, True, window, None)
    _check_heads(q, k, v, do, got, dtype, scale, True, [(0, 0), (1, 7), (3, 15)], window=window)


def test_full_size_alibi_whole_heads():
    # Z4 H16 N2048 D128 bf16, causal with ALiBi slopes 2^(-8(h+1)/H)
    Z, H, N, D, dtype = 4, 16, 2048, 128, "bf16"
    slopes = [2.0 ** (-8.0 * (h + 1) / H) for h in range(H)]
    (q, k, v, do, scale), got = run_bwd_ex(431, Z, H, H, N, N, D, dtype, True, (-1, -1), slopes)
    for z, h in [(0, 0), (2, 9), (3, 15)]:
        _check_heads(q, k, v, do, got, dtype, scale, True, [(z, h)],
                     alibi=np.full(1, slopes[h], dtype=np.float64))


def test_full_size_varlen_whole_sequences():
    # 16 packed causal sequences of 256-4096 rows (seeded), H16 D128 bf16: the
    # oracle differentiates the shortest and the longest sequence, two heads each
    import torch
    import exact_attention_44_gb300 as fa
    H, D, dtype = 16, 128, "bf16"
    lens = np.random.default_rng(0).integers(256, 4097, size=16)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    q = si.normals(432, 0, H * total * D, dtype).reshape(1, H, total, D)
    k = si.normals(432, q.size, H * total * D, dtype).reshape(1, H, total, D)
    v = si.normals(432, 2 * q.size, H * total * D, dtype).reshape(1, H, total, D)
    do = si.normals(1432, 0, q.size, dtype).reshape(q.shape)
    scale = 1 / math.sqrt(D)
    qt, kt, vt, dot = (to_device(x, dtype) for x in (q, k, v, do))
    cu_t = torch.from_numpy(cu).cuda()
    o, lse = fa.fa_fwd_ex(qt, kt, vt, scale=scale, causal=True, cu_seqlens_q=cu_t, cu_seqlens_k=cu_t)
    dq, dk, dv = fa.fa_bwd_ex(qt, kt, vt, o, lse, dot, scale=scale, causal=True, cu_seqlens_q=cu_t,
                              cu_seqlens_k=cu_t)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    for z in (int(np.argmin(lens)), int(np.argmax(lens))):
        rows = slice(int(cu[z]), int(cu[z + 1]))
        for h in (0, H - 1):
            one = (slice(0, 1), slice(h, h + 1), rows)
            ref = oracle.attention_bwd_ex(q[one], k[one], v[one], do[one], dtype, scale, True)
            for name, g, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
                g = g[one].double().cpu().numpy()
                err, mag = float(np.max(np.abs(g - want))), float(np.max(np.abs(want)))
                assert err <= TOL_GRAD[dtype] * max(mag, 1e-3), f"sequence {z} head {h} {name}: {err:.3e} vs {mag:.3e}"
