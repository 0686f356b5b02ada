"""GPU parity of fa_bwd_ex (gradients of the window / ALiBi forward) against
the fp64 oracle's attention_bwd_ex, on dense (Z, H, N, D) tensors.

The forward's O and lse come from fa_fwd_ex with the same options (the GPU's
own chain, as for fa_bwd); the oracle differentiates the definition from Q, K,
V and dO.  Tolerance as for fa_bwd (tests/test_bwd_gpu.py): 4 unit roundoffs
of the input type relative to the largest reference gradient.  Cases: each
window side alone and both, with and without the causal rule, ALiBi alone and
with a window, GQA, query and key lengths that differ (rows that keep no key:
dQ = 0), windows so narrow most blocks are skipped, the open window routed to
fa_bwd's kernel, and the head dim the variants do not cover."""
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


def test_head_dim_256_variants_are_unsupported():
    import torch
    import exact_attention_44_gb300 as fa
    q, k, v = si.qkv(309, 1, 2, 2, 64, 64, 256, "bf16")
    qt, kt, vt = (to_device(x, "bf16") for x in (q, k, v))
    o, lse = fa.fa_fwd(qt, kt, vt, causal=False)
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd_ex(qt, kt, vt, o, lse, torch.zeros_like(qt), window=(8, 8))
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
