"""The shared input generator: determinism, counter-based sub-ranges, rounding, moments."""
import numpy as np
import pytest

import seeded_inputs as si


def test_splitmix64_first_outputs_seed0():
    # splitmix64 seeded with 0: the first outputs of Vigna's reference generator.
    lib = si._load()
    got = [lib.si_splitmix64_at(0, i) for i in range(3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_counter_based():
    a = si.normals(7, 0, 100_001)
    b = si.normals(7, 0, 100_001)
    assert np.array_equal(a, b)
    # any sub-range equals the slice of the full stream (odd offsets included)
    assert np.array_equal(si.normals(7, 12_345, 50_000), a[12_345:62_345])
    assert np.array_equal(si.normals(7, 1, 3), a[1:4])
    assert not np.array_equal(si.normals(8, 0, 1000), a[:1000])


def test_threads_do_not_change_values():
    assert np.array_equal(si.normals(3, 5, 300_000, nthreads=1), si.normals(3, 5, 300_000, nthreads=7))


def test_normal_moments():
    x = si.normals(0, 0, 2_000_000)
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1.0) < 5e-3
    # fourth moment of N(0,1) is 3
    assert abs((x ** 4).mean() - 3.0) < 0.05
    assert np.all(np.isfinite(x))


def test_fp16_rounding_matches_numpy():
    # numpy's float64 -> float16 conversion rounds to nearest even, subnormals included
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.standard_normal(20000),
        rng.standard_normal(5000) * 1e-5,          # subnormal range
        rng.standard_normal(2000) * 3e4,           # near overflow
        np.array([0.0, -0.0, 65504.0, 65519.9, 65520.0, 1e-8, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -24]),
        # exact ties: halfway between consecutive fp16 values
        (np.arange(1024, 1100) + 0.5) * 2.0 ** -10,
    ])
    got = si.round_bits(xs, "fp16")
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def _bf16_value(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-39,
                         (np.arange(128, 200) + 0.5) * 2.0 ** -7])
    bits = si.round_bits(xs, "bf16")
    y = _bf16_value(bits)
    assert np.all(np.signbit(y) == np.signbit(xs))
    mag = bits & 0x7FFF
    zero = mag == 0
    # a result of zero: |x| is at most half the smallest subnormal (2^-133 / 2)
    assert np.all(np.abs(xs[zero]) <= 2.0 ** -134)
    nz = ~zero
    b, x = bits[nz].astype(np.int64), xs[nz]
    up = _bf16_value((b + 1).astype(np.uint16))   # next magnitude away from zero
    dn = _bf16_value((b - 1).astype(np.uint16))   # next magnitude towards zero
    err = np.abs(x - y[nz])
    assert np.all(err <= np.abs(x - up))
    assert np.all(err <= np.abs(x - dn))
    ties = ((err == np.abs(x - up)) | (err == np.abs(x - dn))) & (err > 0)
    assert ties.sum() >= 70
    assert np.all(b[ties] % 2 == 0)


def test_qkv_one_stream_order():
    q, k, v = si.qkv(0, 1, 2, 1, 3, 5, 16, "fp16")
    assert q.shape == (1, 2, 3, 16) and k.shape == (1, 1, 5, 16) and v.shape == k.shape
    full = si.normals(0, 0, q.size + 2 * k.size, "fp16")
    assert np.array_equal(np.concatenate([q.ravel(), k.ravel(), v.ravel()]), full)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_as_torch_is_a_view_of_bits(dtype):
    torch = pytest.importorskip("torch")
    q, _, _ = si.qkv(0, 1, 1, 1, 4, 4, 16, dtype)
    t = si.as_torch(q, dtype)
    assert t.dtype == (torch.float16 if dtype == "fp16" else torch.bfloat16)
    assert np.array_equal(t.view(torch.int16).numpy().view(np.uint16), q)
