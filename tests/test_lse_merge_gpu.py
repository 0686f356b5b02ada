"""GPU parity of fa_lse_merge (results over disjoint key sets combined by
their log-sum-exps) against the oracle's fp64 merge, on seeded synthetic
parts, and end to end: fa_fwd over key shards, merged, against the oracle's
attention over all keys."""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from parity_util import TOL_LSE, TOL_O, compare, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()


def _parts(seed, n, shape, dtype, lse_spread=5.0):
    """n seeded O parts (dtype bits) and fp32-representable lse parts."""
    size = int(np.prod(shape))
    rows = size // shape[-1]
    o_bits = [si.normals(seed, i * size, size, dtype).reshape(shape) for i in range(n)]
    base = n * size
    lse = [(si.normals(seed, base + i * rows, rows, "f64") * lse_spread).astype(np.float32).reshape(shape[:-1])
           for i in range(n)]
    return o_bits, lse


def _merge_gpu(o_bits, lse, dtype):
    import torch
    import exact_attention_44_gb300 as fa
    o_t = [to_device(b, dtype) for b in o_bits]
    l_t = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in lse]
    o, l = fa.fa_lse_merge(o_t, l_t)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), l.double().cpu().numpy()


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("n", [1, 2, 3, 16])
@pytest.mark.parametrize("D", [16, 64, 128, 256])
def test_synthetic_parts(dtype, n, D):
    shape = (2, 3, 77, D)
    o_bits, lse = _parts(50 + n, n, shape, dtype)
    o_ref, l_ref = oracle.lse_merge([si.as_torch(b, dtype).double().numpy() for b in o_bits],
                                    [x.astype(np.float64) for x in lse])
    o_gpu, l_gpu = _merge_gpu(o_bits, lse, dtype)
    compare(o_gpu, l_gpu, o_ref, l_ref, dtype, f"merge n={n} D={D}")


def test_empty_parts():
    dtype = "fp16"
    o_bits, lse = _parts(60, 3, (1, 2, 40, 64), dtype)
    lse[1][:, :, ::3] = -np.inf            # part 1 holds no key for every third row
    for x in lse:
        x[:, 1, 5] = -np.inf               # row (0, 1, 5): no key anywhere
    o_ref, l_ref = oracle.lse_merge([si.as_torch(b, dtype).double().numpy() for b in o_bits],
                                    [x.astype(np.float64) for x in lse])
    o_gpu, l_gpu = _merge_gpu(o_bits, lse, dtype)
    assert np.all(o_gpu[0, 1, 5] == 0) and l_gpu[0, 1, 5] == -np.inf
    keep = np.isfinite(l_ref)
    compare(o_gpu[keep], l_gpu[keep], o_ref[keep], l_ref[keep], dtype, "merge with empty parts")


@pytest.mark.parametrize("cuts", [(0, 1024, 2048), (0, 300, 301, 1500, 2048), (0, 128, 256, 384, 512, 2048)])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_key_shards_end_to_end(cuts, dtype):
    import torch
    import exact_attention_44_gb300 as fa
    Z, Hq, Hkv, Nq, Nkv, D = 1, 4, 2, 200, cuts[-1], 128
    q, k, v = si.qkv(61, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    scale = 1 / math.sqrt(D)
    qt = to_device(q, dtype)
    parts = []
    for a, b in zip(cuts, cuts[1:]):
        kt = to_device(np.ascontiguousarray(k[:, :, a:b]), dtype)
        vt = to_device(np.ascontiguousarray(v[:, :, a:b]), dtype)
        parts.append(fa.fa_fwd(qt, kt, vt, scale=scale))
    o, l = fa.fa_lse_merge([p[0] for p in parts], [p[1] for p in parts])
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    o_ref, l_ref = oracle.attention_fwd(q, k, v, dtype, scale, False)
    compare(o.double().cpu().numpy(), l.double().cpu().numpy(), o_ref, l_ref, dtype, f"shards {cuts}")


def test_strided_parts_and_output():
    import torch
    import exact_attention_44_gb300 as fa
    from parity_util import relayout
    dtype = "bf16"
    o_bits, lse = _parts(62, 2, (2, 4, 50, 64), dtype)
    o_t = [relayout(to_device(b, dtype), "bsnd") for b in o_bits]
    l_t = [torch.from_numpy(x).cuda() for x in lse]
    out = relayout(torch.empty(2, 4, 50, 64, dtype=torch.bfloat16, device="cuda"), "padded")
    o, l = fa.fa_lse_merge(o_t, l_t, o=out)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.lse_merge([si.as_torch(b, dtype).double().numpy() for b in o_bits],
                                    [x.astype(np.float64) for x in lse])
    compare(o.double().cpu().numpy(), l.double().cpu().numpy(), o_ref, l_ref, dtype, "strided merge")
