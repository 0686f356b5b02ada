"""GPU parity: libfa against the fp64 oracle, element by element, on small and
ragged shapes that span several tiles, every head dim and dtype, both masks,
GQA groupings, strided layouts, and the failure modes the pages list
("Write Triton Attention Kernel", Common failure modes)."""
import math

import numpy as np
import pytest

import seeded_inputs as si
from parity_util import check_full, run_gpu

pytestmark = pytest.mark.gpu

DIMS = [16, 32, 64, 128, 256]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()


@pytest.mark.parametrize("D", DIMS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dims(D, dtype, causal):
    check_full(1, 1, 2, 2, 300, 300, D, dtype, causal)


@pytest.mark.parametrize("Nq,Nkv", [(1, 1), (1, 300), (127, 127), (129, 129), (128, 1), (200, 77), (77, 200),
                                    (1000, 1000), (256, 1024), (1024, 256)])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(Nq, Nkv, causal):
    # tails on either side; causal with Nq != Nkv keeps the top-left convention
    check_full(2, 1, 2, 1, Nq, Nkv, 64, "fp16", causal)


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (2, 1), (4, 1), (8, 2), (8, 8), (32, 1), (32, 8)])
def test_gqa_groupings(Hq, Hkv):
    # distinct K/V per kv head: a wrong head stride reads another head's keys
    check_full(3, 2, Hq, Hkv, 130, 260, 32, "bf16", True)


@pytest.mark.parametrize("layout,o_layout", [("bsnd", "bnsd"), ("bnsd", "bsnd"), ("padded", "padded"),
                                             ("bsnd", "bsnd")])
@pytest.mark.parametrize("D", [64, 128])
def test_strided_layouts(layout, o_layout, D):
    check_full(4, 2, 4, 2, 200, 300, D, "fp16", False, layout=layout, o_layout=o_layout)
    check_full(4, 2, 4, 2, 200, 300, D, "bf16", True, layout=layout, o_layout=o_layout)


def test_growing_block_maxima_need_rescaling():
    # later key blocks score higher, so the running max moves at every block:
    # a missing alpha rescale of O or l is caught here
    def grow(q, k, v):
        kd = (k.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ramp = np.linspace(0.2, 3.0, k.shape[2])[None, None, :, None]
        return q, si.round_bits(kd * ramp, "bf16"), v
    check_full(5, 1, 2, 2, 256, 1024, 64, "bf16", False, transform=grow)


def test_future_keys_score_high_under_causal():
    # keys after the query score far above the past ones: masking after the
    # row max (instead of before) would shift the softmax
    def future_heavy(q, k, v):
        kd = q[:, :, : k.shape[2]].view(np.float16).astype(np.float64) * 0.5
        kd = kd * np.linspace(0.1, 4.0, k.shape[2])[None, None, :, None]
        return q, si.round_bits(kd, "fp16"), v
    check_full(6, 1, 2, 2, 384, 384, 64, "fp16", True, transform=future_heavy)


def test_unscaled_scores_of_magnitude_d():
    # scale 1: scores of size ~D stay exact in the fp32 state
    check_full(7, 1, 2, 1, 256, 512, 128, "bf16", False, scale=1.0)
    check_full(7, 1, 2, 1, 256, 512, 128, "fp16", True, scale=0.5)


def test_tiny_scale_gives_mean_of_values():
    check_full(8, 1, 1, 1, 130, 390, 64, "fp16", False, scale=1e-6)


def test_identical_rows_in_both_dtypes_and_lse_optional():
    import torch
    from exact_attention_44_gb300 import fa_fwd
    q, k, v = si.qkv(9, 1, 4, 4, 256, 256, 64, "bf16")
    qt, kt, vt = (si.as_torch(x, "bf16").cuda() for x in (q, k, v))
    o1, lse1 = fa_fwd(qt, kt, vt, causal=True)
    o2, lse2 = fa_fwd(qt, kt, vt, causal=True, want_lse=False)
    torch.cuda.synchronize()
    assert lse2 is None
    assert torch.equal(o1, o2)


def test_deterministic_bitwise():
    import torch
    from exact_attention_44_gb300 import fa_fwd
    q, k, v = si.qkv(10, 2, 8, 2, 1000, 1000, 128, "bf16")
    qt, kt, vt = (si.as_torch(x, "bf16").cuda() for x in (q, k, v))
    outs = [fa_fwd(qt, kt, vt, causal=c) for c in (True, True, False, False)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[2][0], outs[3][0]) and torch.equal(outs[2][1], outs[3][1])


def test_empty_problems_are_noops():
    import torch
    from exact_attention_44_gb300 import fa_fwd
    q = torch.empty(0, 2, 64, 64, dtype=torch.float16, device="cuda")
    o, lse = fa_fwd(q, q[:, :1], q[:, :1])
    assert o.shape == q.shape and lse.shape == (0, 2, 64)
    q = torch.empty(1, 2, 0, 64, dtype=torch.float16, device="cuda")
    k = torch.randn(1, 2, 5, 64, dtype=torch.float16, device="cuda")
    fa_fwd(q, k, k)
    torch.cuda.synchronize()


def test_device_status_is_clean_after_normal_runs():
    from exact_attention_44_gb300 import fa_device_status, fa_fwd
    q, k, v = si.qkv(11, 1, 2, 1, 300, 300, 64, "fp16")
    fa_fwd(*(si.as_torch(x, "fp16").cuda() for x in (q, k, v)), causal=True)
    code, word = fa_device_status()
    assert code == 0 and word == 0


def test_misaligned_views_are_rejected_not_computed():
    import torch
    from exact_attention_44_gb300 import FA_ERR_ALIGNMENT, FaError, fa_fwd
    base = torch.zeros(1, 1, 64, 72, dtype=torch.float16, device="cuda")
    q = base[..., 4:68]  # 8-byte offset: not 16-byte aligned
    with pytest.raises(FaError) as e:
        fa_fwd(q, q, q)
    assert e.value.code == FA_ERR_ALIGNMENT


def test_output_matches_torch_sdpa_as_a_second_opinion():
    # not the oracle: PyTorch's own attention in fp32 on the same inputs, as a
    # sanity cross-check of the harness (tolerance of the oracle comparison)
    import torch
    q, k, v = si.qkv(12, 2, 4, 4, 333, 333, 64, "fp16")
    o, lse = run_gpu(q, k, v, "fp16", 0.125, True)
    qt, kt, vt = (si.as_torch(x, "fp16").float() for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.125)
    assert np.max(np.abs(o - ref.double().numpy())) < 5e-3
    s = (qt @ kt.transpose(-1, -2)) * 0.125
    s = s.masked_fill(torch.ones(333, 333, dtype=torch.bool).triu(1), float("-inf"))
    assert np.max(np.abs(lse - torch.logsumexp(s, -1).double().numpy())) < 1e-3


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_scale_zero_gives_mean_of_kept_values(D, causal):
    # scale 0 ("1/sqrt(D) or a custom value", "Write Triton Attention Kernel",
    # Inputs 4): every kept key weighs the same, O = mean of their V and
    # lse = log of their count -- the closed form the oracle is pinned to
    import oracle
    q, k, v = si.qkv(13, 1, 2, 2, 300, 300, D, "bf16")
    o, lse = run_gpu(q, k, v, "bf16", 0.0, causal)
    check_full(13, 1, 2, 2, 300, 300, D, "bf16", causal, scale=0.0)
    vd = oracle.decode(v, "bf16")
    n = np.arange(1, 301) if causal else np.full(300, 300)
    mean = (np.cumsum(vd[0, 0], axis=0) / n[:, None]) if causal else np.broadcast_to(vd[0, 0].mean(0), (300, D))
    assert np.max(np.abs(o[0, 0] - mean)) <= 2e-2
    assert np.max(np.abs(lse[0, 0] - np.log(n))) <= 1e-5


@pytest.mark.parametrize("D", [32, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_negative_scale(D, dtype, causal):
    # a negative scale turns the softmax toward the lowest scores: the row
    # extreme that references the exponentials is then the row minimum
    check_full(14, 1, 2, 1, 260, 390, D, dtype, causal, scale=-1 / math.sqrt(D))
    check_full(15, 1, 2, 1, 200, 200, D, dtype, causal, scale=-1.0)


def test_negative_and_zero_scale_through_the_split_schedule_and_variants():
    import exact_attention_44_gb300 as fa
    fa.fa_debug_force_split(1)
    try:
        check_full(16, 1, 4, 2, 150, 1500, 128, "bf16", False, scale=-0.2, impl="splitkv")
        check_full(16, 1, 4, 2, 150, 1500, 128, "bf16", True, scale=0.0, impl="splitkv")
    finally:
        fa.fa_debug_force_split(0)


@pytest.fixture(params=[1, 2], ids=["two_chains", "one_chain"])
def softmax_kernel(request):
    # whole tiles of D <= 128 run one of two kernels (one or two softmax
    # chains); the library picks by shape, these tests force each in turn
    import exact_attention_44_gb300 as fa
    fa.fa_debug_force_chains(request.param)
    yield request.param
    fa.fa_debug_force_chains(0)


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_both_softmax_kernels_head_dims(softmax_kernel, D, dtype, causal):
    check_full(31, 1, 2, 2, 300, 300, D, dtype, causal)


@pytest.mark.parametrize("Nq,Nkv", [(1, 1), (1, 300), (129, 129), (200, 77), (77, 200), (1000, 1000), (256, 1024)])
@pytest.mark.parametrize("causal", [False, True])
def test_both_softmax_kernels_ragged(softmax_kernel, Nq, Nkv, causal):
    # odd block counts: the two chains' hand-off crosses tile boundaries
    check_full(32, 2, 2, 1, Nq, Nkv, 64, "fp16", causal)


@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (32, 8)])
def test_both_softmax_kernels_gqa(softmax_kernel, Hq, Hkv):
    check_full(33, 2, Hq, Hkv, 130, 900, 128, "bf16", True)


def test_both_softmax_kernels_rescale_and_scales(softmax_kernel):
    # block maxima that keep growing: the maximum moves in both chains, O and
    # each chain's row sum are rescaled; and the zero and negative scales
    def grow(q, k, v):
        kd = (k.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ramp = np.linspace(0.2, 3.0, k.shape[2])[None, None, :, None]
        return q, si.round_bits(kd * ramp, "bf16"), v
    check_full(34, 1, 2, 2, 256, 2048, 64, "bf16", False, transform=grow)
    check_full(34, 1, 2, 2, 256, 2048, 128, "bf16", True, transform=grow)
    check_full(35, 1, 2, 1, 300, 700, 64, "fp16", True, scale=0.0)
    check_full(35, 1, 2, 1, 300, 700, 128, "bf16", False, scale=-0.3)


def test_both_softmax_kernels_bitwise_repeatable(softmax_kernel):
    import torch
    from exact_attention_44_gb300 import fa_fwd
    q, k, v = si.qkv(36, 2, 8, 2, 1000, 1000, 64, "fp16")
    qt, kt, vt = (si.as_torch(x, "fp16").cuda() for x in (q, k, v))
    outs = [fa_fwd(qt, kt, vt, causal=c) for c in (True, True, False, False)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[2][0], outs[3][0]) and torch.equal(outs[2][1], outs[3][1])
