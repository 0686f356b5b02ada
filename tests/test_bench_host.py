"""Host-side accounting of bench.py (CPU): the flops, bytes and workloads its
JSON line reports, checked against their closed forms."""
import bench

MAIN = bench.WORKLOADS[bench.MAIN]
Z4 = bench.WORKLOADS["z4_h16_n1024_d128_bf16"]


def test_headline_workload_is_the_largest_specified_configuration():
    # the largest configuration the path is specified on that fits one GPU:
    # Z=1, Hq=32, Hkv=8 (GQA group 4), Nq=Nkv=32768, D=128, bf16, causal
    assert MAIN == (1, 32, 8, 32768, 32768, 128, "bf16", [True])
    largest = max(bench.WORKLOADS.values(), key=bench.step_flops)
    assert bench.step_flops(MAIN) == bench.step_flops(largest)
    # the Z=4 H=16 N=1024 workload (both masks) and the target shapes are timed besides it
    assert Z4 == (4, 16, 16, 1024, 1024, 128, "bf16", [False, True])
    assert set(bench.EXTRA_SHAPES) == {"z4_h16_n1024_d128_bf16"} | set(bench.TARGET_SHAPES)


def test_flops_count_4_nq_nkv_d_per_head_halved_for_causal():
    Z, Hq, N, D = 4, 16, 1024, 128
    full = 4 * Z * Hq * N * N * D
    assert bench.flops_of(Z, Hq, N, N, D, False) == full
    assert bench.flops_of(Z, Hq, N, N, D, True) == full / 2
    assert bench.step_flops(Z4) == 1.5 * full
    # the headline: 32 heads of 32768^2 pairs, half of them kept
    assert bench.step_flops(MAIN) == 4 * 32 * 32768 * 32768 * 128 / 2
    # cross lengths: Nq x Nkv pairs
    assert bench.flops_of(1, 32, 1024, 8192, 128, False) == 4 * 32 * 1024 * 8192 * 128


def test_bytes_of_a_step_and_of_a_launch():
    Z, Hq, Hkv, Nq, Nkv, D = 4, 16, 16, 1024, 1024, 128
    h2d, d2h = bench.io_bytes(Z4)
    # Q, K, V in bf16 once per step; O (bf16) and lse (fp32) of both launches back
    assert h2d == 2 * (Z * Hq * Nq * D + 2 * Z * Hkv * Nkv * D) == 50331648
    assert d2h == 2 * (2 * Z * Hq * Nq * D + 4 * Z * Hq * Nq) == 34078720
    # per launch: read Q, K, V once, write O and lse once
    assert bench.algorithmic_bytes(Z4) == 2 * (2 * Z * Hq * Nq * D + 2 * Z * Hkv * Nkv * D) + 4 * Z * Hq * Nq
    assert bench.algorithmic_bytes(Z4) == 67371008
    # the headline: Q and O of 32 heads, K and V of 8 heads, lse of 32 heads
    assert bench.io_bytes(MAIN) == (2 * (32 + 16) * 32768 * 128, 2 * 32 * 32768 * 128 + 4 * 32 * 32768)
    # GQA: K and V have Hkv heads
    gqa = bench.WORKLOADS["z1_hq32_hkv8_n8192_d128_bf16_noncausal"]
    assert bench.algorithmic_bytes(gqa) == 2 * (2 * 32 * 8192 * 128 + 2 * 8 * 8192 * 128) + 4 * 32 * 8192


def test_every_extra_shape_is_a_known_workload():
    for name in bench.TARGET_SHAPES + bench.SPLIT_SHAPES + bench.EXTRA_SHAPES:
        assert name in bench.WORKLOADS
    for wl in bench.WORKLOADS.values():
        Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
        assert Hq % Hkv == 0 and D in (16, 32, 64, 128, 256) and dtype in ("fp16", "bf16") and flags


def test_peaks_come_from_the_measured_file_when_present():
    import json
    import os
    p = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    peaks = bench.load_peaks()
    if os.path.exists(p):
        d = json.load(open(p))
        assert peaks["source"] == "measured" and peaks["bf16_tflops"] == d["bf16_tflops"]
    else:
        assert peaks["source"] == "fallback"
