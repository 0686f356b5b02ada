"""GPU parity of the CTA-pair forward kernel (D = 128) against the fp64 oracle.

A cluster of two CTAs takes two query tiles that see the same key blocks --
two query heads of one GQA group (even group sizes), else query blocks 2m and
2m + 1 of one head -- and multiplies each key block once for both (M = 256
over two SMs, each SM holding half of every K and V block).  The library
picks it for long tiles; these tests force it (fa_debug_force_pair) on shapes
that exercise both pairings, ragged query and key lengths, a last query block
without a partner (odd block count), causal top-left alignment with Nq != Nkv,
GQA, strided layouts, any finite scale, and more units than clusters.  Every
output row and lse is compared (parity_util.check_full)."""
import pytest

from parity_util import check_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _pair_kernel():
    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()
    fa.fa_debug_force_pair(1)
    yield
    fa.fa_debug_force_pair(0)


def _runs_on_pairs(Z, Hq, Hkv, Nq, Nkv, causal):
    import exact_attention_44_gb300 as fa
    s = fa.fa_fwd_schedule(Z, Hq, Hkv, Nq, Nkv, 128, causal, num_sms=152, l2_bytes=126 << 20)
    return s["cta_pairs"] == 1


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (4, 4), (6, 2), (3, 1)], ids=["head_pairs", "block_pairs",
                                                                          "group3_block_pairs", "group3_odd"])
def test_pairings(dtype, causal, Hq, Hkv):
    assert _runs_on_pairs(1, Hq, Hkv, 520, 600, causal)
    print(check_full(301, 1, Hq, Hkv, 520, 600, 128, dtype, causal))


@pytest.mark.parametrize("Nq,Nkv", [(128, 128), (129, 300), (300, 129), (1000, 1000), (1300, 700), (700, 1300),
                                    (255, 2049), (2049, 255)])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(Nq, Nkv, causal):
    # block pairs (Hq = Hkv) and head pairs (group 2) on the same lengths;
    # an odd number of query blocks leaves the last unit a tile past the rows
    print(check_full(302, 2, 2, 2, Nq, Nkv, 128, "bf16", causal))
    print(check_full(303, 1, 4, 2, Nq, Nkv, 128, "bf16", causal))


@pytest.mark.parametrize("causal", [False, True])
def test_many_units_per_cluster(causal):
    # 2 x 16 query heads, group 4 -> 16 virtual heads x 12 blocks = 192 units on <= 76 clusters
    print(check_full(304, 2, 16, 4, 1500, 1500, 128, "bf16", causal))


@pytest.mark.parametrize("layout", ["bsnd", "padded"])
def test_layouts(layout):
    print(check_full(305, 2, 4, 2, 400, 900, 128, "bf16", True, layout=layout, o_layout=layout))


@pytest.mark.parametrize("scale", [0.0, -0.0883883, 1.0])
def test_any_scale(scale):
    print(check_full(306, 1, 4, 2, 300, 700, 128, "bf16", True, scale=scale))
    print(check_full(307, 1, 2, 2, 300, 700, 128, "fp16", False, scale=scale))


def test_gqa_packed_rows():
    # non-causal with Nq < 128: each GQA group's rows run as one head (group
    # 1 after packing): block pairs whose odd tile lies past the packed rows
    print(check_full(308, 2, 8, 2, 24, 3000, 128, "bf16", False))
