"""GPU parity at the full sizes of the workloads this path is specified on,
in the launch configuration the benchmark times.

Every output row is compared with the fp64 oracle ("Write Triton Attention
Kernel", Correctness requirements: verify against a reference attention
implementation), except for the causal N = 32768 GQA workload, whose full
comparison is ~8.8 TFLOP of fp64 work: there every row of query heads 0 and
31 is compared, and in each other head the rows 0, 127, 128, 32767, the
first row of every 128-row tile and 512 seeded random rows."""
import pytest

from parity_util import check_full, check_full_chunked, check_heads_full_rest_sampled

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
def test_z4_h16_n1024_d128_bf16_every_row(causal):
    print(check_full_chunked(0, 4, 16, 16, 1024, 1024, 128, "bf16", causal))


@pytest.mark.parametrize("D", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_sweep_z8_h16_n2048_every_row(D, dtype, causal):
    print(check_full_chunked(0, 8, 16, 16, 2048, 2048, D, dtype, causal))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_many_heads_z128_h8_n1024_fp16_every_row(D, causal):
    # 1024 heads: several causal head groups of the persistent schedule, every head compared
    print(check_full_chunked(0, 128, 8, 8, 1024, 1024, D, "fp16", causal))


def test_long_context_gqa_n32768_causal():
    print(check_heads_full_rest_sampled(0, 1, 32, 8, 32768, 32768, 128, "bf16", True, full_heads={0, 31}))


def test_cross_attention_nq1024_nkv8192_every_row():
    print(check_full_chunked(0, 1, 32, 8, 1024, 8192, 128, "bf16", False))


def test_supplementary_n8192_noncausal_every_row():
    print(check_full_chunked(0, 1, 32, 8, 8192, 8192, 128, "bf16", False))
