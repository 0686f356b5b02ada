"""Shared helpers for the GPU-vs-oracle parity tests.

Inputs come from seeded_inputs (the same bits go to the GPU and the oracle);
the CUDA side is called only through the libfa binding; expected values come
only from the oracle.
"""
from __future__ import annotations

import math

import numpy as np

import oracle
import seeded_inputs as si

# max |ΔO| for N(0,1) inputs per dtype and max |Δlse|: the tolerances the
# specification of this path fixes.  They absorb the kernel's fp16/bf16
# rounding of P before P·V and of O at the store (half an ulp of |O| <= 4 is
# 2e-3 in fp16 and 1.6e-2 in bf16) plus fp32 accumulation.
TOL_O = {"fp16": 5e-3, "bf16": 2e-2}
TOL_LSE = 1e-3


def torch_dtype(dtype):
    import torch
    return torch.float16 if dtype == "fp16" else torch.bfloat16


def to_device(bits: np.ndarray, dtype: str, device="cuda"):
    return si.as_torch(bits, dtype).to(device)


def run_gpu(q, k, v, dtype, scale, causal, layout="bnsd", o_layout="bnsd", impl="fwd"):
    """Run libfa on seeded bits; returns (O as float64 numpy (Z,Hq,Nq,D), lse float64 (Z,Hq,Nq)).

    impl: "fwd" (fa_fwd, whole query tiles per CTA) or "splitkv" (fa_fwd_splitkv,
    key blocks cut into one range per SM, parts merged by their lse)."""
    import torch
    from exact_attention_44_gb300 import fa_device_status, fa_fwd, fa_fwd_splitkv

    qt, kt, vt = (relayout(to_device(x, dtype), layout) for x in (q, k, v))
    o = relayout(torch.empty(qt.shape, dtype=qt.dtype, device="cuda"), o_layout)
    if impl == "splitkv":
        o, lse = fa_fwd_splitkv(qt, kt, vt, o=o, scale=scale, causal=causal)
    else:
        o, lse = fa_fwd(qt, kt, vt, o=o, scale=scale, causal=causal)
    code, word = fa_device_status()
    assert code == 0, f"device status {word:#x}: a bounded wait ran out"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def relayout(t, layout):
    """Same values, another memory layout: 'bnsd' (contiguous), 'bsnd' (heads
    inside rows, i.e. (Z, N, H, D) storage), or 'padded' (row pitch D + 8)."""
    import torch
    if layout == "bnsd":
        return t.contiguous()
    Z, H, N, D = t.shape
    if layout == "bsnd":
        store = torch.empty((Z, N, H, D), dtype=t.dtype, device=t.device)
        view = store.permute(0, 2, 1, 3)
    elif layout == "padded":
        store = torch.empty((Z, H, N, D + 8), dtype=t.dtype, device=t.device)
        view = store[..., :D]
    else:
        raise ValueError(layout)
    view.copy_(t)
    return view


def compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    do = float(np.max(np.abs(o_gpu - o_ref))) if o_ref.size else 0.0
    dl = float(np.max(np.abs(lse_gpu - lse_ref))) if lse_ref.size else 0.0
    assert np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu)), f"{what}: non-finite GPU output"
    assert do <= TOL_O[dtype], f"{what}: max|dO| = {do:.3e} > {TOL_O[dtype]}"
    assert dl <= TOL_LSE, f"{what}: max|dlse| = {dl:.3e} > {TOL_LSE}"
    return do, dl


def check_full(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype, causal, scale=None, layout="bnsd", o_layout="bnsd",
               transform=None, impl="fwd"):
    """Every output row against the oracle."""
    scale = 1 / math.sqrt(D) if scale is None else scale
    q, k, v = si.qkv(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    if transform is not None:
        q, k, v = transform(q, k, v)
    o_gpu, lse_gpu = run_gpu(q, k, v, dtype, scale, causal, layout, o_layout, impl)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, dtype, scale, causal)
    return compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype, f"{(Z, Hq, Hkv, Nq, Nkv, D, dtype, causal)}")


def sample_rows(Nq, n_random, rng):
    """Row indices of one head: tile edges (0, 127, 128, ...), the last row, and random rows."""
    rows = {0, Nq - 1}
    for t in range(0, Nq, 128):
        rows.update(r for r in (t, t + 127) if r < Nq)
    rows.update(rng.integers(0, Nq, size=n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def check_sampled(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype, causal, n_groups=2, rows_per_head=48, scale=None,
                  impl="fwd"):
    """Full-size run on the GPU; the oracle checks sampled rows of a few GQA groups.

    For each sampled (z, kv head) the oracle gets just that group's query heads
    and its K/V, and computes the sampled rows one by one."""
    scale = 1 / math.sqrt(D) if scale is None else scale
    q, k, v = si.qkv(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    o_gpu, lse_gpu = run_gpu(q, k, v, dtype, scale, causal, impl=impl)
    g = Hq // Hkv
    rng = np.random.default_rng(seed + 1)
    groups = {(0, 0), (Z - 1, Hkv - 1)}
    while len(groups) < min(n_groups, Z * Hkv):
        groups.add((int(rng.integers(Z)), int(rng.integers(Hkv))))
    worst = (0.0, 0.0)
    for z, hk in sorted(groups):
        qs = q[z:z + 1, hk * g:(hk + 1) * g]
        ks, vs = k[z:z + 1, hk:hk + 1], v[z:z + 1, hk:hk + 1]
        heads = sorted({0, g - 1} | {int(rng.integers(g))})
        rows, flat = [], []
        for h in heads:
            r = sample_rows(Nq, rows_per_head, rng)
            rows.append((h, r))
            flat.append(h * Nq + r)
        o_ref, lse_ref = oracle.attention_fwd(qs, ks, vs, dtype, scale, causal, rows=np.concatenate(flat))
        og = np.concatenate([o_gpu[z, hk * g + h, r] for h, r in rows])
        lg = np.concatenate([lse_gpu[z, hk * g + h, r] for h, r in rows])
        d = compare(og, lg, o_ref, lse_ref, dtype, f"z={z} hk={hk} {(Z, Hq, Hkv, Nq, Nkv, D, dtype, causal)}")
        worst = (max(worst[0], d[0]), max(worst[1], d[1]))
    return worst


def _gpu_tensors(q, k, v, dtype, scale, causal, impl="fwd"):
    """Full-size GPU run on seeded bits; (O, lse) stay on the device."""
    import torch
    from exact_attention_44_gb300 import fa_device_status, fa_fwd, fa_fwd_splitkv

    qt, kt, vt = (to_device(x, dtype) for x in (q, k, v))
    if impl == "splitkv":
        o, lse = fa_fwd_splitkv(qt, kt, vt, scale=scale, causal=causal)
    else:
        o, lse = fa_fwd(qt, kt, vt, scale=scale, causal=causal)
    torch.cuda.synchronize()
    code, word = fa_device_status()
    assert code == 0, f"device status {word:#x}: a bounded wait ran out"
    del qt, kt, vt
    return o, lse


def check_full_chunked(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype, causal, scale=None, impl="fwd",
                       max_rows=1 << 18):
    """Every output row of a full-size run against the oracle.

    The GPU computes the whole problem at once (the launch the benchmark
    times); the oracle then takes it in chunks of whole GQA groups, at most
    about `max_rows` query rows per chunk, so host memory stays bounded.
    Returns the worst (max|dO|, max|dlse|) over all rows."""
    scale = 1 / math.sqrt(D) if scale is None else scale
    q, k, v = si.qkv(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    o_dev, lse_dev = _gpu_tensors(q, k, v, dtype, scale, causal, impl)
    g = Hq // Hkv
    group_rows = g * Nq
    groups_per_chunk = max(1, max_rows // max(group_rows, 1))
    worst = (0.0, 0.0)
    # chunks of (z, kv head) groups in memory order: z outer, kv head inner
    for first in range(0, Z * Hkv, groups_per_chunk):
        last = min(Z * Hkv, first + groups_per_chunk)
        for z in range(first // Hkv, (last - 1) // Hkv + 1):
            h0 = max(first - z * Hkv, 0)
            h1 = min(last - z * Hkv, Hkv)
            qs = q[z:z + 1, h0 * g:h1 * g]
            ks, vs = k[z:z + 1, h0:h1], v[z:z + 1, h0:h1]
            o_ref, lse_ref = oracle.attention_fwd(qs, ks, vs, dtype, scale, causal)
            og = o_dev[z:z + 1, h0 * g:h1 * g].double().cpu().numpy()
            lg = lse_dev[z:z + 1, h0 * g:h1 * g].double().cpu().numpy()
            d = compare(og, lg, o_ref, lse_ref, dtype,
                        f"z={z} kv heads {h0}..{h1 - 1} {(Z, Hq, Hkv, Nq, Nkv, D, dtype, causal)}")
            worst = (max(worst[0], d[0]), max(worst[1], d[1]))
    return worst


def check_heads_full_rest_sampled(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype, causal, full_heads, rows_per_head=512,
                                  scale=None, impl="fwd"):
    """Full-size run; every row of the (z = 0) query heads in `full_heads`, and in
    every other head of z = 0 a seeded sample: rows 0, 127, 128 and Nq - 1, the
    first row of every 128-row tile, and `rows_per_head` random rows.

    For problems whose full comparison would take the oracle far longer
    than a test may (the causal N = 32768 workload is ~8.8 TFLOP in fp64)."""
    scale = 1 / math.sqrt(D) if scale is None else scale
    q, k, v = si.qkv(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    o_dev, lse_dev = _gpu_tensors(q, k, v, dtype, scale, causal, impl)
    g = Hq // Hkv
    rng = np.random.default_rng(seed + 7)
    fixed = {0, 127, 128, Nq - 1} | set(range(0, Nq, 128))
    worst = (0.0, 0.0)
    for hk in range(Hkv):
        rows, flat = [], []
        for h in range(hk * g, (hk + 1) * g):
            if h in full_heads:
                # shuffled: the oracle gives each thread a contiguous slice of
                # the rows, and causal rows cost in proportion to their index
                r = rng.permutation(Nq).astype(np.int64)
            else:
                r = np.array(sorted(x for x in fixed | set(rng.integers(0, Nq, size=rows_per_head).tolist())
                                    if 0 <= x < Nq), dtype=np.int64)
            rows.append((h, r))
            flat.append((h - hk * g) * Nq + r)
        o_ref, lse_ref = oracle.attention_fwd(q[0:1, hk * g:(hk + 1) * g], k[0:1, hk:hk + 1], v[0:1, hk:hk + 1],
                                              dtype, scale, causal, rows=np.concatenate(flat))
        og = np.concatenate([o_dev[0, h][torch_index(r)].double().cpu().numpy() for h, r in rows])
        lg = np.concatenate([lse_dev[0, h][torch_index(r)].double().cpu().numpy() for h, r in rows])
        d = compare(og, lg, o_ref, lse_ref, dtype, f"kv head {hk} {(Z, Hq, Hkv, Nq, Nkv, D, dtype, causal)}")
        worst = (max(worst[0], d[0]), max(worst[1], d[1]))
    return worst


def torch_index(rows):
    import torch
    return torch.from_numpy(np.asarray(rows, dtype=np.int64)).cuda()
