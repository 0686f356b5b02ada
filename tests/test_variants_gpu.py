"""GPU parity of fa_fwd_ex (sliding window, ALiBi, packed variable-length
batches) against the fp64 oracle's variant forward, element by element, with
rows that keep no key (O = 0, lse = -inf) checked exactly."""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from parity_util import TOL_LSE, TOL_O, relayout, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()


def _compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what):
    empty = np.isneginf(lse_ref)
    assert np.all(np.isneginf(lse_gpu[empty])), f"{what}: rows without keys must have lse = -inf"
    assert np.all(o_gpu[empty] == 0), f"{what}: rows without keys must have O = 0"
    keep = ~empty
    assert np.all(np.isfinite(o_gpu[keep])) and np.all(np.isfinite(lse_gpu[keep])), f"{what}: non-finite"
    do = float(np.max(np.abs(o_gpu[keep] - o_ref[keep]), initial=0.0))
    dl = float(np.max(np.abs(lse_gpu[keep] - lse_ref[keep]), initial=0.0))
    assert do <= TOL_O[dtype], f"{what}: max|dO| = {do:.3e}"
    assert dl <= TOL_LSE, f"{what}: max|dlse| = {dl:.3e}"


def _slopes(Hq):
    # the geometric sequence of slopes 2^(-8 h / Hq), h = 1..Hq
    return np.array([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=np.float32)


def _run_padded(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype, causal, window=(-1, -1), alibi=False, layout="bnsd"):
    import torch
    import exact_attention_44_gb300 as fa
    scale = 1 / math.sqrt(D)
    q, k, v = si.qkv(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    slopes = _slopes(Hq) if alibi else None
    qt, kt, vt = (relayout(to_device(x, dtype), layout) for x in (q, k, v))
    st = torch.from_numpy(slopes).cuda() if alibi else None
    o, lse = fa.fa_fwd_ex(qt, kt, vt, scale=scale, causal=causal, window=window, alibi_slopes=st)
    torch.cuda.synchronize()
    code, word = fa.fa_device_status()
    assert code == 0, f"device status {word:#x}"
    o_ref, l_ref = oracle.attention_fwd_ex(q, k, v, dtype, scale, causal, window=window,
                                           alibi=None if slopes is None else slopes.astype(np.float64))
    _compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, l_ref, dtype,
             f"{(Z, Hq, Hkv, Nq, Nkv, D, dtype, causal, window, alibi)}")


@pytest.mark.parametrize("window", [(0, 0), (64, 64), (200, -1), (-1, 100), (127, 0), (1000, 1000), (5, 300)])
@pytest.mark.parametrize("causal", [False, True])
def test_window(window, causal):
    _run_padded(91, 1, 2, 1, 300, 333, 64, "fp16", causal, window=window)


@pytest.mark.parametrize("D", [16, 32, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_window_head_dims(D, dtype):
    _run_padded(92, 1, 2, 2, 260, 260, D, dtype, True, window=(100, 0))
    _run_padded(93, 1, 2, 2, 260, 300, D, dtype, False, window=(30, 70))


def test_window_rows_without_keys():
    # rows beyond Nkv + left keep no key at all
    _run_padded(94, 1, 2, 1, 400, 100, 64, "bf16", False, window=(10, 10))
    _run_padded(95, 1, 1, 1, 300, 300, 128, "fp16", False, window=(0, 0))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16"), (256, "fp16")])
def test_alibi(causal, D, dtype):
    _run_padded(96, 2, 8, 2, 270, 290, D, dtype, causal, alibi=True)


def test_alibi_with_window_and_layouts():
    _run_padded(97, 1, 4, 4, 333, 333, 128, "bf16", True, window=(96, 0), alibi=True, layout="bsnd")


@pytest.mark.parametrize("window", [(-1, -1), (333 + 444 + 1, -1), (-1, 5000), (10 ** 6, 10 ** 6)])
def test_no_options_is_fa_fwd_bitwise(window):
    # no sequence table, no slopes and open window sides: the call is fa_fwd
    import torch
    import exact_attention_44_gb300 as fa
    for causal in (False, True):
        q, k, v = (to_device(x, "bf16") for x in si.qkv(98, 2, 4, 2, 333, 444, 128, "bf16"))
        a = fa.fa_fwd(q, k, v, causal=causal)
        b = fa.fa_fwd_ex(q, k, v, causal=causal, window=window)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def _varlen_case(seed, lens_q, lens_k, Hq, Hkv, D, dtype, extra_q=0, extra_k=0):
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    tq, tk = int(cu_q[-1]) + extra_q, int(cu_k[-1]) + extra_k
    q = si.normals(seed, 0, Hq * tq * D, dtype).reshape(1, Hq, tq, D)
    k = si.normals(seed, q.size, Hkv * tk * D, dtype).reshape(1, Hkv, tk, D)
    v = si.normals(seed, q.size + k.size, Hkv * tk * D, dtype).reshape(1, Hkv, tk, D)
    return cu_q, cu_k, q, k, v


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("thd", [False, True])
def test_varlen(causal, thd):
    import torch
    import exact_attention_44_gb300 as fa
    dtype, D, Hq, Hkv = "bf16", 128, 4, 2
    lens_q = [5, 0, 135, 60, 1, 300, 128, 129]
    lens_k = [7, 23, 0, 300, 1, 290, 128, 500]
    cu_q, cu_k, q, k, v = _varlen_case(99, lens_q, lens_k, Hq, Hkv, D, dtype, extra_q=10)
    scale = 1 / math.sqrt(D)
    qt, kt, vt = (to_device(x, dtype) for x in (q, k, v))
    if thd:  # (total, H, D) storage
        qt, kt, vt = (x[0].permute(1, 0, 2).contiguous() for x in (qt, kt, vt))
    o = torch.zeros(qt.shape, dtype=qt.dtype, device="cuda")
    o, lse = fa.fa_fwd_ex(qt, kt, vt, o=o, scale=scale, causal=causal,
                          cu_seqlens_q=torch.from_numpy(cu_q).cuda(), cu_seqlens_k=torch.from_numpy(cu_k).cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    og = (o.permute(1, 0, 2).unsqueeze(0) if thd else o).double().cpu().numpy()
    o_ref, l_ref = oracle.attention_fwd_ex(q, k, v, dtype, scale, causal, cu_q=cu_q, cu_k=cu_k)
    n = int(cu_q[-1])
    _compare(og[:, :, :n], lse.double().cpu().numpy()[None, :, :n], o_ref[:, :, :n], l_ref[:, :, :n], dtype,
             f"varlen causal={causal} thd={thd}")
    # packed rows that belong to no sequence are left untouched
    assert np.all(og[:, :, n:] == 0)


def test_varlen_with_window_alibi_gqa():
    import torch
    import exact_attention_44_gb300 as fa
    dtype, D, Hq, Hkv = "fp16", 64, 8, 2
    cu_q, cu_k, q, k, v = _varlen_case(100, [200, 17, 260], [200, 300, 260], Hq, Hkv, D, dtype)
    scale, slopes = 0.125, _slopes(Hq)
    o, lse = fa.fa_fwd_ex(*(to_device(x, dtype) for x in (q, k, v)), scale=scale, causal=True, window=(50, -1),
                          alibi_slopes=torch.from_numpy(slopes).cuda(), cu_seqlens_q=torch.from_numpy(cu_q).cuda(),
                          cu_seqlens_k=torch.from_numpy(cu_k).cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    o_ref, l_ref = oracle.attention_fwd_ex(q, k, v, dtype, scale, True, window=(50, -1),
                                           alibi=slopes.astype(np.float64), cu_q=cu_q, cu_k=cu_k)
    _compare(o.double().cpu().numpy(), lse.double().cpu().numpy()[None], o_ref, l_ref, dtype, "varlen+window+alibi")


def test_full_size_sliding_window_sampled():
    # Z=4 H=16 N=2048 D=128 bf16, causal with a 256-key window: sampled rows
    import torch
    import exact_attention_44_gb300 as fa
    Z, Hq, Hkv, N, D, dtype = 4, 16, 16, 2048, 128, "bf16"
    q, k, v = si.qkv(101, Z, Hq, Hkv, N, N, D, dtype)
    o, lse = fa.fa_fwd_ex(*(to_device(x, dtype) for x in (q, k, v)), causal=True, window=(256, 0))
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    og, lg = o.double().cpu().numpy(), lse.double().cpu().numpy()
    rng = np.random.default_rng(5)
    for z, h in ((0, 0), (Z - 1, Hq - 1), (1, 7)):
        rows = np.array(sorted({0, 127, 128, 255, 256, 257, N - 1} | set(rng.integers(0, N, 40).tolist())))
        o_ref, l_ref = oracle.attention_fwd_ex(q[z:z + 1, h:h + 1], k[z:z + 1, h:h + 1], v[z:z + 1, h:h + 1], dtype,
                                               1 / math.sqrt(D), True, window=(256, 0), rows=rows)
        _compare(og[z, h, rows], lg[z, h, rows], o_ref, l_ref, dtype, f"window z={z} h={h}")


def test_option_errors():
    import torch
    import exact_attention_44_gb300 as fa
    q = torch.zeros(1, 2, 64, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_ex(q, q, q, window=(-2, 0))
    assert e.value.code == fa.FA_ERR_INVALID_ARG
