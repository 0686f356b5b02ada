"""GPU parity at the full sizes of the workloads this path is specified on,
in the launch configuration the benchmark times.  The GPU computes every row;
the oracle checks sampled rows (tile edges, last row, random rows) of a few
GQA groups, one by one.  Config 1 is small enough to compare in full."""
import pytest

from parity_util import check_full, check_sampled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()


def test_tiny_fp16_seed0_full():
    # Z=1 H=2 N=128 D=64 fp16, seed 0, scale 1/8, non-causal
    check_full(0, 1, 2, 2, 128, 128, 64, "fp16", False, scale=1 / 8)


@pytest.mark.parametrize("causal", [False, True])
def test_z4_h16_n1024_d128_bf16(causal):
    check_sampled(0, 4, 16, 16, 1024, 1024, 128, "bf16", causal)


@pytest.mark.parametrize("D", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_sweep_z8_h16_n2048(D, dtype, causal):
    check_sampled(0, 8, 16, 16, 2048, 2048, D, dtype, causal, rows_per_head=24)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_many_heads_z128_h8_n1024_fp16(D, causal):
    check_sampled(0, 128, 8, 8, 1024, 1024, D, "fp16", causal, n_groups=4, rows_per_head=16)


def test_long_context_gqa_n32768_causal():
    check_sampled(0, 1, 32, 8, 32768, 32768, 128, "bf16", True, n_groups=2, rows_per_head=40)


def test_cross_attention_nq1024_nkv8192():
    check_sampled(0, 1, 32, 8, 1024, 8192, 128, "bf16", False, n_groups=3, rows_per_head=48)


def test_supplementary_n8192_noncausal():
    check_sampled(0, 1, 32, 8, 8192, 8192, 128, "bf16", False, n_groups=2, rows_per_head=32)
