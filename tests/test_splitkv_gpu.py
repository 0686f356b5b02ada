"""GPU parity of fa_fwd_splitkv (key blocks of all query tiles cut into one
equal range per SM, cut tiles merged by their log-sum-exps) against the fp64
oracle, on shapes where the cuts fall inside tiles, at every head dim, both
masks, GQA, decode-like and cross lengths, plus full-size sampled configs."""
import math

import numpy as np
import pytest

import seeded_inputs as si
from parity_util import check_full, check_sampled, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    # these tests exercise the cut schedule on every shape; fa_fwd_splitkv
    # would otherwise keep whole tiles where cutting does not pay
    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()
    fa.fa_debug_force_split(1)
    yield
    fa.fa_debug_force_split(0)


@pytest.mark.parametrize("D", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dims(D, dtype, causal):
    # 2 heads x 3 tiles x (3 or fewer) key blocks: fewer pairs than SMs, so
    # every CTA holds one block and every multi-block tile is cut
    check_full(31, 1, 2, 2, 300, 300, D, dtype, causal, impl="splitkv")


@pytest.mark.parametrize("Nq,Nkv", [(1, 1), (1, 300), (1, 5000), (7, 4096), (128, 1), (129, 129), (200, 77),
                                    (77, 200), (1000, 1000), (256, 2048), (2048, 256)])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(Nq, Nkv, causal):
    check_full(32, 1, 2, 1, Nq, Nkv, 64, "fp16", causal, impl="splitkv")


@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (8, 2), (32, 8)])
def test_gqa(Hq, Hkv):
    check_full(33, 2, Hq, Hkv, 150, 700, 128, "bf16", False, impl="splitkv")


@pytest.mark.parametrize("causal", [False, True])
def test_many_tiles_few_cuts(causal):
    # more (tile, block) pairs than SMs: most tiles whole, a few cut
    check_full(34, 2, 8, 4, 640, 640, 64, "fp16", causal, impl="splitkv")


def test_layouts():
    check_full(35, 2, 4, 2, 300, 900, 64, "bf16", False, layout="bsnd", o_layout="padded", impl="splitkv")


def test_large_scores_and_rescale():
    # scores of several hundred: maxima jump across parts and blocks
    check_full(36, 1, 2, 1, 256, 3000, 64, "fp16", False, scale=3.0, impl="splitkv")


def test_bitwise_repeatable():
    q, k, v = si.qkv(37, 1, 4, 1, 333, 2000, 128, "bf16")
    a = run_gpu(q, k, v, "bf16", 0.1, False, impl="splitkv")
    b = run_gpu(q, k, v, "bf16", 0.1, False, impl="splitkv")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_lse_none_and_workspace_reuse():
    import torch
    import exact_attention_44_gb300 as fa
    q, k, v = (si.as_torch(x, "fp16").cuda() for x in si.qkv(38, 1, 2, 1, 100, 1500, 64, "fp16"))
    ws = fa.workspace_for(64)
    o1, _ = fa.fa_fwd_splitkv(q, k, v, workspace=ws, want_lse=False)
    o2, l2 = fa.fa_fwd_splitkv(q, k, v, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and l2 is not None
    assert fa.fa_device_status()[0] == 0


def test_workspace_errors():
    import torch
    import exact_attention_44_gb300 as fa
    q = torch.zeros(1, 1, 64, 64, dtype=torch.float16, device="cuda")
    need = fa.fa_fwd_splitkv_workspace_size(64)
    assert need >= 2 * torch.cuda.get_device_properties(0).multi_processor_count * 128 * 65 * 4
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_splitkv(q, q, q, workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
    assert e.value.code == fa.FA_ERR_WORKSPACE
    big = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_splitkv(q, q, q, workspace=big[16:])  # not 256-byte aligned
    assert e.value.code == fa.FA_ERR_WORKSPACE


@pytest.mark.parametrize("name,shape,causal", [
    ("cross Nq1024 Nkv8192", (1, 32, 8, 1024, 8192, 128, "bf16"), False),
    ("GQA N32768 causal", (1, 32, 8, 32768, 32768, 128, "bf16"), True),
    ("Z4 H16 N1024", (4, 16, 16, 1024, 1024, 128, "bf16"), False),
])
def test_full_size_sampled(name, shape, causal):
    check_sampled(39, *shape, causal, impl="splitkv")


def test_stall_times_out_and_recovers():
    import torch
    import exact_attention_44_gb300 as fa
    q, k, v = (si.as_torch(x, "fp16").cuda() for x in si.qkv(40, 1, 2, 1, 256, 2048, 64, "fp16"))
    fa.fa_debug_set_wait_limit_ms(100)
    fa.fa_debug_inject_stall(True)
    try:
        fa.fa_fwd_splitkv(q, k, v)
        code, word = fa.fa_device_status()
    finally:
        fa.fa_debug_inject_stall(False)
        fa.fa_debug_set_wait_limit_ms(0)
    assert code == fa.FA_ERR_DEVICE_TIMEOUT and (word >> 16) == 0
    o, lse = fa.fa_fwd_splitkv(q, k, v)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0 and torch.isfinite(o).all()


@pytest.mark.parametrize("shape,causal", [
    ((1, 8, 8, 128, 20000, 64, "bf16"), False),   # few tiles, many keys: cut
    ((1, 8, 2, 1, 9000, 128, "fp16"), False),     # decode row
    ((2, 4, 2, 640, 640, 64, "fp16"), True),      # many tiles: whole
])
def test_automatic_choice(shape, causal):
    import exact_attention_44_gb300 as fa
    fa.fa_debug_force_split(0)
    try:
        check_full(41, *shape, causal, impl="splitkv")
    finally:
        fa.fa_debug_force_split(1)


@pytest.mark.parametrize("Z,Hq,Hkv,Nq,Nkv", [(1, 8, 2, 1, 3000), (2, 8, 2, 5, 1000), (3, 16, 2, 16, 700),
                                             (1, 32, 4, 31, 2049), (2, 4, 2, 100, 513), (1, 8, 8, 1, 900)])
@pytest.mark.parametrize("impl", ["fwd", "splitkv"])
def test_gqa_packed_short_queries(Z, Hq, Hkv, Nq, Nkv, impl):
    # non-causal, Nq < 128, contiguous: the g query heads of a group run as one
    # head of g * Nq rows (the last case, g = 1, is not packed)
    check_full(42, Z, Hq, Hkv, Nq, Nkv, 128, "bf16", False, impl=impl)


def test_gqa_pack_skipped_for_other_layouts_and_causal():
    check_full(43, 2, 8, 2, 7, 800, 64, "fp16", False, layout="bsnd", impl="splitkv")
    check_full(44, 2, 8, 2, 7, 800, 64, "fp16", True, impl="splitkv")


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_few_row_tiles(D, dtype):
    # cut launches of tiles with few query rows: decode rows (GQA-packed: 4
    # query heads x 2 rows = 8 rows a tile) against thousands of keys, and 64
    # plain rows, at every head dim up to 128
    check_full(46, 2, 8, 2, 2, 3000, D, dtype, False, impl="splitkv")
    check_full(47, 1, 2, 2, 64, 2500, D, dtype, False, impl="splitkv")


def test_few_row_stall_times_out_and_recovers():
    import torch
    import exact_attention_44_gb300 as fa
    q, k, v = (si.as_torch(x, "bf16").cuda() for x in si.qkv(48, 1, 8, 2, 1, 4096, 128, "bf16"))
    fa.fa_debug_set_wait_limit_ms(100)
    fa.fa_debug_inject_stall(True)
    try:
        fa.fa_fwd_splitkv(q, k, v)
        code, word = fa.fa_device_status()
    finally:
        fa.fa_debug_inject_stall(False)
        fa.fa_debug_set_wait_limit_ms(0)
    assert code == fa.FA_ERR_DEVICE_TIMEOUT and (word >> 16) == 0
    check_full(48, 1, 8, 2, 1, 4096, 128, "bf16", False, impl="splitkv")
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
