"""fa_fwd_splitkv_noalloc against the oracle and against fa_fwd_splitkv.

The no-allocation entry point is for callers that cannot allocate device
memory during a call (a cudaMalloc synchronises the device and can take
milliseconds; some plugin interfaces hand over only inputs and outputs).  It
runs the split-KV forward in a fixed device array inside the library instead
of a caller workspace.  Here it is called through the C ABI twice in a row,
on shapes that cut key ranges (so the array really holds partial results
between the two kernels of each call).  Each call must match the fp64
oracle within the parity tolerances, and must be bitwise equal to
fa_fwd_splitkv on the same inputs, which computes the same thing with a
caller workspace.  The file is collected last so that a failure here stops
a -x run only after every other test has run.
"""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from parity_util import TOL_LSE, TOL_O, compare, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [
    (1, 8, 2, 130, 9000, 128, "bf16", False),
    (1, 4, 4, 200, 3000, 256, "fp16", True),
])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(shape):
    import torch
    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()
    Z, Hq, Hkv, Nq, Nkv, D, dtype, causal = shape
    qb, kb, vb = si.qkv(71, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    q, k, v = (to_device(x, dtype) for x in (qb, kb, vb))
    scale = 1 / math.sqrt(D)
    o_want, lse_want = oracle.attention_fwd(qb, kb, vb, dtype, scale, causal)
    ws = fa.workspace_for(D)
    o_ref = torch.empty_like(q)
    lse_ref = torch.empty((Z, Hq, Nq), dtype=torch.float32, device=q.device)
    fa.fa_debug_force_split(1)  # both entry points cut key ranges on this shape
    try:
        fa.fa_fwd_splitkv(q, k, v, o=o_ref, lse=lse_ref, scale=scale, causal=causal, workspace=ws)
        torch.cuda.synchronize()
        for call in range(2):
            o = torch.full_like(q, float("nan"))
            lse = torch.full((Z, Hq, Nq), float("nan"), dtype=torch.float32, device=q.device)
            fa.fa_fwd_splitkv_noalloc(q, k, v, o, lse, scale=scale, causal=causal)
            torch.cuda.synchronize()
            code, word = fa.fa_device_status()
            assert code == 0, f"call {call}: device status {word:#x}"
            compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_want, lse_want, dtype, f"call {call}")
            assert torch.equal(o, o_ref), f"call {call}: O differs from fa_fwd_splitkv's"
            assert torch.equal(lse, lse_ref), f"call {call}: lse differs from fa_fwd_splitkv's"
    finally:
        fa.fa_debug_force_split(0)
    assert TOL_O[dtype] > 0 and TOL_LSE > 0
