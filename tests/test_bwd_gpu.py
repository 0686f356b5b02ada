"""GPU parity of fa_bwd (dQ, dK, dV) against the fp64 oracle's backward.

The GPU backward takes the GPU forward's O and lse (its own chain); the
oracle takes only Q, K, V and dO and differentiates the definition.

Tolerance, relative to the largest reference gradient of each tensor, from
the kernel's roundings (u = unit roundoff of the input type: 2^-11 for fp16,
2^-8 for bf16; fp32 accumulation is far below it):
  * P is rounded to the input type before dV = Pᵀ dO and before dS is formed: 1 u;
  * dS = P (dP − Δ) is rounded to the input type before dQ = dS K, dK = dSᵀ Q: 1 u;
  * Δ = rowsum(dO ∘ O) uses the forward's O, itself rounded to the input type: 1 u;
  * dQ, dK, dV are rounded to the input type when stored: ½ u.
Each gradient element is a sum over keys or queries in which every term
carries at most these relative errors; independent rounding errors add like
the terms themselves, so the error is a small multiple of u times the size
of the gradient: 3.5 u, taken as 4 u (fp16 1.95e-3, bf16 1.56e-2).
"""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from parity_util import relayout, to_device

pytestmark = pytest.mark.gpu

UNIT_ROUNDOFF = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}
TOL_GRAD = {dt: 4 * u for dt, u in UNIT_ROUNDOFF.items()}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()


def check_bwd(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype, causal, scale=None, layout="bnsd"):
    import torch
    import exact_attention_44_gb300 as fa
    scale = 1 / math.sqrt(D) if scale is None else scale
    q, k, v = si.qkv(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    do = si.normals(seed + 1000, 0, q.size, dtype).reshape(q.shape)
    qt, kt, vt, dot = (relayout(to_device(x, dtype), layout) for x in (q, k, v, do))
    o, lse = fa.fa_fwd(qt, kt, vt, scale=scale, causal=causal)
    dq, dk, dv = fa.fa_bwd(qt, kt, vt, o, lse, dot, scale=scale, causal=causal)
    torch.cuda.synchronize()
    code, word = fa.fa_device_status()
    assert code == 0, f"device status {word:#x}"
    ref = oracle.attention_bwd(q, k, v, do, dtype, scale, causal)
    worst = {}
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = got.double().cpu().numpy()
        assert np.all(np.isfinite(g)), f"{name}: non-finite"
        err = float(np.max(np.abs(g - want)))
        mag = float(np.max(np.abs(want)))
        worst[name] = (err, mag)
        assert err <= TOL_GRAD[dtype] * max(mag, 1e-3), f"{name}: max|d| = {err:.3e}, max|ref| = {mag:.3e}"
    return worst


@pytest.mark.parametrize("D", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dims(D, dtype, causal):
    print(check_bwd(201, 1, 2, 2, 300, 300, D, dtype, causal))


# D = 256 runs its own kernel (two passes for dV and dK, 64-row steps): the
# ragged tails of both sequence lengths, a query block that ends inside a
# step, GQA groups, and more units than CTAs so that CTAs take several units
# of both phases.
@pytest.mark.parametrize("Nq,Nkv", [(1, 1), (1, 200), (63, 65), (65, 63), (129, 129), (200, 77), (77, 200),
                                    (256, 640), (640, 256)])
@pytest.mark.parametrize("causal", [False, True])
def test_d256_ragged(Nq, Nkv, causal):
    print(check_bwd(211, 2, 2, 1, Nq, Nkv, 256, "bf16", causal))


@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (8, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_d256_gqa(Hq, Hkv, causal):
    print(check_bwd(212, 1, Hq, Hkv, 330, 330, 256, "fp16", causal))


def test_d256_layouts():
    print(check_bwd(213, 2, 4, 2, 200, 300, 256, "bf16", True, layout="bsnd"))


@pytest.mark.parametrize("causal", [False, True])
def test_d256_many_units_per_cta(causal):
    # 2 x 8 heads x 10 key blocks = 160 dK/dV units and 160 dQ units on
    # at most 152 CTAs
    print(check_bwd(214, 2, 8, 8, 1280, 1280, 256, "bf16", causal))


@pytest.mark.parametrize("scale", [0.0, -1.0])
def test_d256_zero_and_negative_scale(scale):
    print(check_bwd(215, 1, 2, 1, 260, 300, 256, "bf16", True, scale=scale))


@pytest.mark.parametrize("Nq,Nkv", [(1, 1), (1, 200), (129, 129), (200, 77), (77, 200), (256, 640), (640, 256)])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged(Nq, Nkv, causal):
    print(check_bwd(202, 2, 2, 1, Nq, Nkv, 64, "fp16", causal))


@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (8, 2), (8, 8)])
def test_gqa(Hq, Hkv):
    print(check_bwd(203, 1, Hq, Hkv, 260, 260, 128, "bf16", True))


def test_layouts():
    print(check_bwd(204, 2, 4, 2, 200, 300, 64, "bf16", False, layout="bsnd"))


def test_large_scores():
    print(check_bwd(205, 1, 2, 1, 256, 256, 64, "fp16", False, scale=1.0))


@pytest.mark.parametrize("scale", [0.0, -0.125, -1.0])
@pytest.mark.parametrize("causal", [False, True])
def test_zero_and_negative_scale(scale, causal):
    # any finite scale ("Write Triton Attention Kernel", Inputs 4); at scale 0
    # dQ = dK = 0 and dV_j = sum_i dO_i / n_i (the oracle's pinned closed form)
    print(check_bwd(210, 1, 2, 1, 260, 300, 64, "bf16", causal, scale=scale))


def test_workspace_and_argument_errors():
    import torch
    import exact_attention_44_gb300 as fa
    q = torch.zeros(1, 1, 64, 64, dtype=torch.float16, device="cuda")
    lse = torch.zeros(1, 1, 64, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd(q, q, q, q, lse, q, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == fa.FA_ERR_WORKSPACE
    q96 = torch.zeros(1, 1, 64, 96, dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd(q96, q96, q96, q96, lse, q96, workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.code == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("causal", [False, True])
def test_full_size_every_element(causal):
    # Z=4 H=16 N=1024 D=128 bf16: the forward's main workload, every gradient element
    print(check_bwd(206, 4, 16, 16, 1024, 1024, 128, "bf16", causal))


def test_long_gqa_causal_sampled_heads():
    # GQA group of 4 at N=4096: the oracle differentiates one (z, kv head) group
    import torch
    import exact_attention_44_gb300 as fa
    Z, Hq, Hkv, N, D, dtype = 1, 8, 2, 4096, 128, "bf16"
    scale = 1 / math.sqrt(D)
    q, k, v = si.qkv(207, Z, Hq, Hkv, N, N, D, dtype)
    do = si.normals(1207, 0, q.size, dtype).reshape(q.shape)
    qt, kt, vt, dot = (to_device(x, dtype) for x in (q, k, v, do))
    o, lse = fa.fa_fwd(qt, kt, vt, causal=True)
    dq, dk, dv = fa.fa_bwd(qt, kt, vt, o, lse, dot, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    hk = 1
    sl = slice(hk * 4, hk * 4 + 4)
    ref = oracle.attention_bwd(q[:, sl], k[:, hk:hk + 1], v[:, hk:hk + 1], do[:, sl], dtype, scale, True)
    for name, got, want in zip(("dq", "dk", "dv"), (dq[:, sl], dk[:, hk:hk + 1], dv[:, hk:hk + 1]), ref):
        g = got.double().cpu().numpy()
        err, mag = float(np.max(np.abs(g - want))), float(np.max(np.abs(want)))
        assert err <= TOL_GRAD[dtype] * mag, f"{name}: {err:.3e} vs {mag:.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_many_heads_sampled(causal):
    # Z=128 H=8 N=1024 D=64 fp16: 1024 heads, more than one group of the
    # dK/dV and dQ unit orders (a group's Q/dO or K/V fits in a third of L2);
    # the oracle differentiates heads spread over the groups, the last included
    import torch
    import exact_attention_44_gb300 as fa
    Z, H, N, D, dtype = 128, 8, 1024, 64, "fp16"
    scale = 1 / math.sqrt(D)
    q, k, v = si.qkv(209, Z, H, H, N, N, D, dtype)
    do = si.normals(1209, 0, q.size, dtype).reshape(q.shape)
    qt, kt, vt, dot = (to_device(x, dtype) for x in (q, k, v, do))
    o, lse = fa.fa_fwd(qt, kt, vt, causal=causal)
    dq, dk, dv = fa.fa_bwd(qt, kt, vt, o, lse, dot, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    for z, h in [(0, 0), (20, 3), (20, 4), (64, 0), (127, 7)]:
        one = (slice(z, z + 1), slice(h, h + 1))
        ref = oracle.attention_bwd(q[one], k[one], v[one], do[one], dtype, scale, causal)
        for name, got, want in zip(("dq", "dk", "dv"), (dq[one], dk[one], dv[one]), ref):
            g = got.double().cpu().numpy()
            err, mag = float(np.max(np.abs(g - want))), float(np.max(np.abs(want)))
            assert err <= TOL_GRAD[dtype] * mag, f"head ({z}, {h}) {name}: {err:.3e} vs {mag:.3e}"


def test_bitwise_repeatable():
    # no atomics: two runs give identical bits for dQ, dK and dV
    import torch
    import exact_attention_44_gb300 as fa
    q, k, v = (to_device(x, "bf16") for x in si.qkv(208, 2, 8, 2, 700, 900, 128, "bf16"))
    do = to_device(si.normals(1208, 0, 2 * 8 * 700 * 128, "bf16").reshape(2, 8, 700, 128), "bf16")
    for causal in (False, True):
        o, lse = fa.fa_fwd(q, k, v, causal=causal)
        a = fa.fa_bwd(q, k, v, o, lse, do, causal=causal)
        b = fa.fa_bwd(q, k, v, o, lse, do, causal=causal)
        torch.cuda.synchronize()
        assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_headline_size_gradient_invariants():
    # Z1 Hq32 Hkv8 N32768 D128 bf16 causal (the forward's headline workload):
    # too large for the oracle, so two properties that hold at any size are
    # checked per kv head over its GQA group.  Rows of P sum to one, so the
    # keys' dV sum to the queries' dO sum; rows of dS sum to zero (Δ is the
    # row sum of P ∘ dP), so the keys' dK sum to zero.  With these inputs the
    # early key blocks hold most of every causal row's mass: one of them left
    # out or given to the wrong head moves the dV sum far past the tolerance
    # (the last few blocks hold too little mass for this check to see).
    # Sampled rows of dQ are held against the oracle.
    import torch
    import exact_attention_44_gb300 as fa
    Z, Hq, Hkv, N, D = 1, 32, 8, 32768, 128
    g = torch.Generator(device="cuda").manual_seed(2024)
    q, do = (torch.randn(Z, Hq, N, D, generator=g, device="cuda").to(torch.bfloat16) for _ in range(2))
    k, v = (torch.randn(Z, Hkv, N, D, generator=g, device="cuda").to(torch.bfloat16) for _ in range(2))
    o, lse = fa.fa_fwd(q, k, v, causal=True)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    grp = Hq // Hkv
    for hk in range(Hkv):
        want = do[0, hk * grp:(hk + 1) * grp].double().sum(dim=(0, 1))
        got = dv[0, hk].double().sum(dim=0)
        assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
        err = float((got - want).abs().max())
        assert err <= 1e-2 * float(want.abs().max()), f"kv head {hk}: sum dV off by {err:.3e}"
        ksum = dk[0, hk].double().sum(dim=0).abs()
        kabs = dk[0, hk].double().abs().sum(dim=0)
        assert float((ksum / kabs).max()) <= 1e-2, f"kv head {hk}: sum dK not ~0"
    # sampled dQ rows against the oracle: causal row i's dQ is the non-causal
    # dQ of a one-row sequence whose keys are 0 .. i (the oracle's packed
    # sequences), which it differentiates in O(i D)
    def bits(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    scale = 1 / math.sqrt(D)
    for hq, i in [(0, 0), (5, 127), (9, 12345), (31, N - 1)]:
        hk = hq // grp
        one = lambda t, rows: bits(t[0, hq if t.shape[1] == Hq else hk, rows].reshape(1, 1, -1, D))
        ref = oracle.attention_bwd_ex(one(q, slice(i, i + 1)), one(k, slice(0, i + 1)), one(v, slice(0, i + 1)),
                                      one(do, slice(i, i + 1)), "bf16", scale, False,
                                      cu_q=np.array([0, 1], dtype=np.int32), cu_k=np.array([0, i + 1], dtype=np.int32))[0]
        got = dq[0, hq, i].double().cpu().numpy()
        want = ref[0, 0, 0]
        err, mag = float(np.max(np.abs(got - want))), float(np.max(np.abs(want)))
        assert err <= TOL_GRAD["bf16"] * max(mag, 1e-3), f"dQ row ({hq}, {i}): {err:.3e} vs {mag:.3e}"
