"""The debug-check build of libfa (FA_DEBUG_CHECKS=1): every role of the
forward and backward kernels checks each unit it decodes against the
launch's sizes before touching memory for it, records FA_ERR_DEVICE_CHECK
and stops if one is outside them (no trap, no device assert).

CPU: the variant builds and exports the same C ABI.  GPU: every launch mode
of the forward (whole tiles with one and two softmax chains, causal and not,
the split schedule and its merge, window / ALiBi / packed variable-length
variants, GQA packing) and the backward (the D <= 128 and D = 256 kernels,
causal and not, GQA) runs through the checking kernels with a clean status
and the same results as the oracle -- the checks never fire on valid work.
No test plants a bad index on the GPU: an unchecked bad index is the kind of
fault these GPUs are shared too widely to risk."""
import ctypes
import math
import re

import numpy as np
import pytest

import seeded_inputs as si


def _declared_symbols():
    import os
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa.h")).read()
    return sorted(set(re.findall(r"^(?:fa_status|const char\*|void)\s+(fa_\w+)\s*\(", text, re.M)))


def test_debug_check_variant_builds_with_the_same_abi():
    import exact_attention_44_gb300 as fa
    path = fa.build(debug_checks=True)
    assert path.endswith("checks/libfa.so") and path != fa.library_path()
    lib = ctypes.CDLL(path)
    for name in _declared_symbols():
        assert hasattr(lib, name), name


@pytest.mark.gpu
def test_checking_kernels_run_clean_on_every_launch_mode():
    import torch

    import exact_attention_44_gb300 as fa
    from parity_util import check_full
    path = fa.build(debug_checks=True)
    before = fa.use_library(path)
    try:
        fa.load()
        for chains in (1, 2):
            fa.fa_debug_force_chains(chains)
            check_full(41, 2, 4, 2, 300, 300, 64, "fp16", True)
            check_full(41, 1, 2, 2, 700, 900, 128, "bf16", False)
        fa.fa_debug_force_chains(0)
        check_full(42, 1, 2, 1, 260, 260, 256, "bf16", True)
        # the backward's roles check their dK/dV and dQ units (D <= 128 and D = 256 kernels)
        from test_bwd_gpu import check_bwd
        check_bwd(46, 2, 4, 2, 300, 300, 64, "fp16", True)
        check_bwd(46, 1, 4, 1, 200, 400, 128, "bf16", False)
        check_bwd(46, 1, 2, 2, 260, 260, 256, "bf16", True)
        assert fa.fa_device_status() == (fa.FA_OK, 0)
        check_full(43, 1, 8, 2, 3, 2000, 128, "bf16", False)  # GQA packing
        fa.fa_debug_force_split(1)
        try:
            check_full(44, 1, 4, 2, 150, 1500, 128, "bf16", True, impl="splitkv")
            check_full(44, 1, 4, 4, 130, 1200, 256, "fp16", False, impl="splitkv")
        finally:
            fa.fa_debug_force_split(0)
        # the variant kernel: window, ALiBi, packed sequences
        import oracle
        Hq, D = 2, 64
        lens = [100, 300, 1]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        total = int(cu[-1])
        q = si.normals(45, 0, Hq * total * D, "bf16").reshape(1, Hq, total, D)
        k = si.normals(45, q.size, Hq * total * D, "bf16").reshape(1, Hq, total, D)
        v = si.normals(45, 2 * q.size, Hq * total * D, "bf16").reshape(1, Hq, total, D)
        slopes = np.array([0.5, 0.125])
        qt, kt, vt = (si.as_torch(x, "bf16").cuda() for x in (q, k, v))
        cu_t = torch.from_numpy(cu).cuda()
        o, lse = fa.fa_fwd_ex(qt, kt, vt, scale=1 / 8, causal=True, window=(64, -1),
                              alibi_slopes=torch.tensor(slopes, dtype=torch.float32, device="cuda"),
                              cu_seqlens_q=cu_t, cu_seqlens_k=cu_t, max_seqlen_q=max(lens))
        torch.cuda.synchronize()
        code, word = fa.fa_device_status()
        assert code == fa.FA_OK, hex(word)
        o_ref, lse_ref = oracle.attention_fwd_ex(q, k, v, "bf16", 1 / 8, True, window=(64, -1), alibi=slopes,
                                                 cu_q=cu, cu_k=cu)
        assert np.max(np.abs(o.double().cpu().numpy() - o_ref)) <= 2e-2
        lse_ref = lse_ref.reshape(Hq, total)
        fin = np.isfinite(lse_ref)
        assert np.max(np.abs(lse.double().cpu().numpy()[fin] - lse_ref[fin])) <= 1e-3
    finally:
        fa.fa_debug_force_chains(0)
        fa.use_library(before)
        fa.load()
