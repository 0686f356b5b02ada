"""GPU tests of the autograd layer (exact_attention_44_gb300.attention and
attention_varlen): the autograd path runs the same kernels as the direct
calls, so its outputs and gradients equal fa_fwd / fa_bwd (and their _ex
forms) bit for bit; one case is also held against the fp64 oracle (the
tolerances of tests/test_bwd_gpu.py)."""
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


def _leaves(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype):
    q, k, v = si.qkv(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    do = si.normals(seed + 1000, 0, q.size, dtype).reshape(q.shape)
    qt, kt, vt, dot = (to_device(x, dtype) for x in (q, k, v, do))
    return (q, k, v, do), [t.clone().requires_grad_(True) for t in (qt, kt, vt)], dot


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_attention_matches_the_direct_calls_bitwise(causal, D):
    import torch
    import exact_attention_44_gb300 as fa
    _, (q, k, v), do = _leaves(500 + D, 2, 4, 2, 300, 300, D, "bf16")
    o = fa.attention(q, k, v, causal=causal)
    o.backward(do)
    torch.cuda.synchronize()
    o2, lse2 = fa.fa_fwd(q.detach(), k.detach(), v.detach(), causal=causal)
    dq, dk, dv = fa.fa_bwd(q.detach(), k.detach(), v.detach(), o2, lse2, do, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    assert torch.equal(o.detach(), o2)
    for a, b in zip((q.grad, k.grad, v.grad), (dq, dk, dv)):
        assert torch.equal(a, b)


def test_attention_against_the_oracle():
    import torch
    import exact_attention_44_gb300 as fa
    (qn, kn, vn, don), (q, k, v), do = _leaves(510, 1, 4, 2, 257, 300, 128, "fp16")
    scale = 0.1
    o, lse = fa.attention(q, k, v, scale=scale, causal=True, return_lse=True)
    (o.float() * do.float()).sum().backward()
    torch.cuda.synchronize()
    ref = oracle.attention_bwd(qn, kn, vn, don, "fp16", scale, True)
    for name, g, want in zip(("dq", "dk", "dv"), (q.grad, k.grad, v.grad), ref):
        g = g.double().cpu().numpy()
        err, mag = float(np.max(np.abs(g - want))), float(np.max(np.abs(want)))
        assert err <= TOL_GRAD["fp16"] * mag, f"{name}: {err:.3e} vs {mag:.3e}"
    assert lse.requires_grad is False


def test_attention_window_alibi_matches_fa_bwd_ex_bitwise():
    import torch
    import exact_attention_44_gb300 as fa
    _, (q, k, v), do = _leaves(520, 2, 8, 2, 400, 400, 64, "fp16")
    slopes = torch.tensor([2.0 ** (-(h + 1)) for h in range(8)], dtype=torch.float32, device="cuda")
    o = fa.attention(q, k, v, causal=True, window=(100, -1), alibi_slopes=slopes)
    o.backward(do)
    o2, lse2 = fa.fa_fwd_ex(q.detach(), k.detach(), v.detach(), causal=True, window=(100, -1), alibi_slopes=slopes)
    grads = fa.fa_bwd_ex(q.detach(), k.detach(), v.detach(), o2, lse2, do, causal=True, window=(100, -1),
                         alibi_slopes=slopes)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    assert torch.equal(o.detach(), o2)
    for a, b in zip((q.grad, k.grad, v.grad), grads):
        assert torch.equal(a, b)


def test_attention_varlen_matches_fa_bwd_ex_bitwise():
    # (total, H, D) storage, a sequence without keys among them
    import torch
    import exact_attention_44_gb300 as fa
    lens_q, lens_k = [70, 129, 5, 200], [64, 0, 300, 200]
    H, D, dtype = 4, 128, "bf16"
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device="cuda")
    tq, tk = sum(lens_q), sum(lens_k)
    q = to_device(si.normals(530, 0, tq * H * D, dtype).reshape(tq, H, D), dtype).requires_grad_(True)
    k = to_device(si.normals(531, 0, tk * H * D, dtype).reshape(tk, H, D), dtype).requires_grad_(True)
    v = to_device(si.normals(532, 0, tk * H * D, dtype).reshape(tk, H, D), dtype).requires_grad_(True)
    do = to_device(si.normals(533, 0, tq * H * D, dtype).reshape(tq, H, D), dtype)
    o = fa.attention_varlen(q, k, v, cu_q, cu_k, causal=True)
    o.backward(do)
    o2, lse2 = fa.fa_fwd_ex(q.detach(), k.detach(), v.detach(), causal=True, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
    grads = fa.fa_bwd_ex(q.detach(), k.detach(), v.detach(), o2, lse2, do, causal=True, cu_seqlens_q=cu_q,
                         cu_seqlens_k=cu_k)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    assert o.shape == q.shape and torch.equal(o.detach(), o2)
    for a, b in zip((q.grad, k.grad, v.grad), grads):
        assert a.shape == b.shape and torch.equal(a, b)


def test_attention_with_a_non_contiguous_upstream_gradient():
    # the loss reads O through a transpose: the gradient reaching the
    # backward is not contiguous and is made so before the kernels see it
    import torch
    import exact_attention_44_gb300 as fa
    _, (q, k, v), do = _leaves(540, 1, 2, 2, 256, 256, 64, "bf16")
    o = fa.attention(q, k, v)
    (o.transpose(2, 3) * do.transpose(2, 3)).sum().backward()
    o2, lse2 = fa.fa_fwd(q.detach(), k.detach(), v.detach())
    grads = fa.fa_bwd(q.detach(), k.detach(), v.detach(), o2, lse2, do)
    torch.cuda.synchronize()
    for a, b in zip((q.grad, k.grad, v.grad), grads):
        assert torch.equal(a, b)


@pytest.mark.parametrize("D", [128, 256])
def test_training_step_replays_from_a_cuda_graph(D):
    # forward and backward captured once, replayed: the same bits as eager
    # calls (the kernels are launched as programmatic dependents inside the
    # graph; the backward's workspace comes from the graph's pool)
    import torch
    import exact_attention_44_gb300 as fa
    _, (q, k, v), do = _leaves(550 + D, 2, 8, 2, 512, 512, D, "bf16")

    def step():
        for t in (q, k, v):
            t.grad = None
        o = fa.attention(q, k, v, causal=True)
        o.backward(do)
        return o

    o_ref = step().detach().clone()
    ref = [t.grad.clone() for t in (q, k, v)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):  # warm-up on a side stream, as graph capture wants
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        o = step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    assert torch.equal(o, o_ref)
    for a, b in zip((q.grad, k.grad, v.grad), ref):
        assert torch.equal(a, b)
