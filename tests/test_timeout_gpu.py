"""Failure detection on the GPU without a fault: every device-side wait is
bounded.  A test hook makes CTA 0 withhold one K copy; its waits run out after
a short limit, the kernel records FA_ERR_DEVICE_TIMEOUT and exits cleanly, and
the context stays usable for the next launch."""
import pytest

import seeded_inputs as si
from parity_util import check_full

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("chains", [1, 2], ids=["two_chains", "one_chain"])
def test_withheld_copy_times_out_and_the_context_recovers(chains):
    import torch

    import exact_attention_44_gb300 as fa
    fa.build()
    fa.fa_debug_force_chains(chains)
    q, k, v = si.qkv(21, 1, 4, 2, 1024, 1024, 64, "bf16")
    qt, kt, vt = (si.as_torch(x, "bf16").cuda() for x in (q, k, v))
    assert fa.fa_device_status()[0] == fa.FA_OK
    fa.fa_debug_set_wait_limit_ms(100)
    fa.fa_debug_inject_stall(True)
    try:
        fa.fa_fwd(qt, kt, vt, causal=False)
        code, word = fa.fa_device_status()
    finally:
        fa.fa_debug_inject_stall(False)
        fa.fa_debug_set_wait_limit_ms(0)
        fa.fa_debug_force_chains(0)
    assert code == fa.FA_ERR_DEVICE_TIMEOUT, hex(word)
    assert word & 0xFF == fa.FA_ERR_DEVICE_TIMEOUT
    assert (word >> 16) == 0          # CTA 0 gave up first
    assert 1 <= (word >> 8) & 0xFF <= 15  # a known wait site
    # the status word was cleared, and the next launch is correct
    assert fa.fa_device_status() == (fa.FA_OK, 0)
    check_full(22, 1, 4, 2, 300, 300, 64, "bf16", True)
    assert fa.fa_device_status() == (fa.FA_OK, 0)
    torch.cuda.synchronize()


def test_withheld_copy_times_out_on_cta_pairs():
    # the CTA-pair kernel (D = 128, long tiles): CTA 0 withholds its first K
    # half; a CTA of cluster 0 records the timeout (the even CTA waiting for
    # that half, or the odd one waiting for the scores that never come), both
    # leave through the cluster barrier, the context stays usable
    import torch

    import exact_attention_44_gb300 as fa
    fa.build()
    fa.fa_debug_force_pair(1)
    q, k, v = si.qkv(23, 1, 4, 2, 1024, 2048, 128, "bf16")
    qt, kt, vt = (si.as_torch(x, "bf16").cuda() for x in (q, k, v))
    assert fa.fa_device_status()[0] == fa.FA_OK
    fa.fa_debug_set_wait_limit_ms(100)
    fa.fa_debug_inject_stall(True)
    try:
        fa.fa_fwd(qt, kt, vt, causal=False)
        code, word = fa.fa_device_status()
    finally:
        fa.fa_debug_inject_stall(False)
        fa.fa_debug_set_wait_limit_ms(0)
    try:
        assert code == fa.FA_ERR_DEVICE_TIMEOUT, hex(word)
        assert (word >> 16) in (0, 1)          # a CTA of cluster 0
        assert 1 <= (word >> 8) & 0xFF <= 19   # a known wait site
        assert fa.fa_device_status() == (fa.FA_OK, 0)
        check_full(24, 1, 4, 2, 300, 2100, 128, "bf16", True)
        assert fa.fa_device_status() == (fa.FA_OK, 0)
    finally:
        fa.fa_debug_force_pair(0)
    torch.cuda.synchronize()


@pytest.mark.parametrize("D", [128, 256])
def test_withheld_copy_times_out_in_the_backward(D):
    # fa_bwd's dK/dV phase (the D <= 128 kernel and the D = 256 kernel): CTA 0
    # withholds its first unit's K (and V); the MMA issuer's wait runs out,
    # every role of that CTA stops (the dQ phase is skipped), in-flight copies
    # land, TMEM is freed, and the next backward is correct
    import torch

    import exact_attention_44_gb300 as fa
    from test_bwd_gpu import check_bwd
    fa.build()
    q, k, v = (si.as_torch(x, "bf16").cuda() for x in si.qkv(25, 1, 4, 4, 512, 512, D, "bf16"))
    do = si.as_torch(si.normals(26, 0, q.numel(), "bf16").reshape(tuple(q.shape)), "bf16").cuda()
    o, lse = fa.fa_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == fa.FA_OK
    fa.fa_debug_set_wait_limit_ms(100)
    fa.fa_debug_inject_stall(True)
    try:
        fa.fa_bwd(q, k, v, o, lse, do, causal=True)
        code, word = fa.fa_device_status()
    finally:
        fa.fa_debug_inject_stall(False)
        fa.fa_debug_set_wait_limit_ms(0)
    assert code == fa.FA_ERR_DEVICE_TIMEOUT, hex(word)
    assert word & 0xFF == fa.FA_ERR_DEVICE_TIMEOUT
    assert (word >> 16) == 0           # CTA 0 gave up first
    assert 20 <= (word >> 8) & 0xFF <= 32  # a backward wait site
    assert fa.fa_device_status() == (fa.FA_OK, 0)
    check_bwd(24, 1, 2, 1, 300, 300, D, "bf16", True)
    assert fa.fa_device_status() == (fa.FA_OK, 0)
    torch.cuda.synchronize()
