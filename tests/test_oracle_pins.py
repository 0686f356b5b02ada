"""Pins for the CPU oracle: closed forms, invariants, library routines and a brute force.

None of these re-types the oracle's own formula: each compares it with something
the pages or the mathematics fix independently of it.
  - decoding: every fp16/bf16 bit pattern against numpy / the fp32 bit layout;
  - one key: O = V[0], lse = s_00 (closed form);
  - identical keys or scale = 0: O = mean(V), lse = s + ln(Nkv) (closed form);
  - causal row 0: O = V[0]; causal row i = non-causal attention over keys 0..i;
  - V = identity exposes P itself: rows sum to 1, P >= 0, P_ij = 0 above the
    diagonal under the causal mask;
  - an mpmath brute force at 60 digits (no max shift, exact scores);
  - numpy matmul + scipy.special.softmax/logsumexp on small shapes;
  - GQA equals MHA on K/V repeated per group; key permutation invariance.
"""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si

mpmath = pytest.importorskip("mpmath")


def _bits(values, dtype):
    return si.round_bits(np.asarray(values, dtype=np.float64), dtype)


def _np_decode(bits, dtype):
    """Reference decoding through numpy's binary16 and the fp32 bit layout of bf16."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- decoding ----

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_decode_every_bit_pattern(dtype):
    allbits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode(allbits, dtype)
    want = _np_decode(allbits, dtype)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


# ------------------------------------------------------------ closed forms ----

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_single_key_gives_v0(dtype, causal):
    q, k, v = si.qkv(11, 2, 4, 2, 9, 1, 32, dtype)
    scale = 0.3
    o, lse = oracle.attention_fwd(q, k, v, dtype, scale, causal)
    K, V, Q = _np_decode(k, dtype), _np_decode(v, dtype), _np_decode(q, dtype)
    for z in range(2):
        for h in range(4):
            hk = h // 2
            assert np.array_equal(o[z, h], np.broadcast_to(V[z, hk, 0], o[z, h].shape))
            s00 = scale * np.array([math.fsum(Q[z, h, i] * K[z, hk, 0]) for i in range(9)])
            np.testing.assert_allclose(lse[z, h], s00, rtol=0, atol=1e-13)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_identical_keys_give_mean_v(dtype):
    Nkv, D = 37, 64
    q, k, v = si.qkv(5, 1, 2, 1, 6, Nkv, D, dtype)
    k[:] = k[:, :, :1, :]                 # every key equals key 0
    scale = 1 / 8
    o, lse = oracle.attention_fwd(q, k, v, dtype, scale, False)
    Q, K, V = _np_decode(q, dtype), _np_decode(k, dtype), _np_decode(v, dtype)
    mean_v = np.array([math.fsum(V[0, 0, :, d]) / Nkv for d in range(D)])
    for h in range(2):
        np.testing.assert_allclose(o[0, h], np.broadcast_to(mean_v, (6, D)), rtol=0, atol=1e-14)
        s = scale * np.array([math.fsum(Q[0, h, i] * K[0, 0, 0]) for i in range(6)])
        np.testing.assert_allclose(lse[0, h], s + math.log(Nkv), rtol=0, atol=1e-13)


def test_zero_scale_gives_uniform_attention():
    q, k, v = si.qkv(6, 1, 1, 1, 5, 19, 16, "fp16")
    o, lse = oracle.attention_fwd(q, k, v, "fp16", 0.0, False)
    V = _np_decode(v, "fp16")[0, 0]
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(V.mean(0), (5, 16)), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], math.log(19), rtol=0, atol=1e-15)
    # causal: row i averages keys 0..i, lse = ln(i + 1)
    o, lse = oracle.attention_fwd(q, k, v, "fp16", 0.0, True)
    for i in range(5):
        np.testing.assert_allclose(o[0, 0, i], V[: i + 1].mean(0), rtol=0, atol=1e-14)
        assert abs(lse[0, 0, i] - math.log(i + 1)) < 1e-15


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_causal_row0_is_v0(dtype):
    q, k, v = si.qkv(3, 2, 4, 4, 20, 20, 16, dtype)
    scale = 0.25
    o, lse = oracle.attention_fwd(q, k, v, dtype, scale, True)
    Q, K, V = _np_decode(q, dtype), _np_decode(k, dtype), _np_decode(v, dtype)
    assert np.array_equal(o[:, :, 0], V[:, :, 0])
    s00 = scale * np.array([[math.fsum(Q[z, h, 0] * K[z, h, 0]) for h in range(4)] for z in range(2)])
    np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_identity_values_expose_probabilities(causal):
    # With V = I (Nkv = D) row i of O is row i of P = softmax(S).
    D = 16
    q, k, _ = si.qkv(9, 1, 1, 1, D, D, D, "fp16")
    v = _bits(np.eye(D)[None, None], "fp16")
    P, lse = oracle.attention_fwd(q, k, v, "fp16", 0.5, causal)
    P = P[0, 0]
    assert np.all(P >= 0)
    np.testing.assert_allclose(P.sum(1), 1.0, rtol=0, atol=1e-14)
    if causal:
        assert np.all(np.triu(P, 1) == 0)
        assert np.all(np.diag(P) > 0)
    else:
        assert np.all(P > 0)


# --------------------------------------------------- brute force (mpmath) ----

@pytest.mark.parametrize("dtype,scale,causal", [("fp16", 0.25, False), ("bf16", 0.25, True),
                                                ("fp16", 200.0, False), ("bf16", 500.0, True)])
def test_mpmath_bruteforce(dtype, scale, causal):
    """Exact scores, exp without a max shift, 60 significant digits.

    The large scales give scores in the thousands, beyond the float64 range of
    exp (about 709), so an oracle without the max shift returns inf/nan there."""
    Nq, Nkv, D = 4, 6, 16
    q, k, v = si.qkv(21, 1, 1, 1, Nq, Nkv, D, dtype)
    o, lse = oracle.attention_fwd(q, k, v, dtype, scale, causal)
    Q, K, V = _np_decode(q, dtype)[0, 0], _np_decode(k, dtype)[0, 0], _np_decode(v, dtype)[0, 0]
    if scale > 100:
        assert np.max(np.abs(scale * Q @ K.T)) > 1000.0
    with mpmath.workdps(60):
        sc = mpmath.mpf(scale)
        for i in range(Nq):
            keys = range(i + 1) if causal else range(Nkv)
            s = [sc * mpmath.fsum(mpmath.mpf(Q[i, d]) * mpmath.mpf(K[j, d]) for d in range(D)) for j in keys]
            e = [mpmath.exp(x) for x in s]
            tot = mpmath.fsum(e)
            assert abs(lse[0, 0, i] - float(mpmath.log(tot))) <= 1e-13 * max(1.0, abs(float(mpmath.log(tot))))
            for d in range(D):
                ref = mpmath.fsum(e[t] * mpmath.mpf(V[j, d]) for t, j in enumerate(keys)) / tot
                assert abs(o[0, 0, i, d] - float(ref)) <= 2e-14


# -------------------------------------------------- library routines (scipy) ----

def _scipy_attention(q, k, v, dtype, scale, causal):
    from scipy.special import logsumexp, softmax

    Q, K, V = _np_decode(q, dtype), _np_decode(k, dtype), _np_decode(v, dtype)
    g = Q.shape[1] // K.shape[1]
    K = np.repeat(K, g, axis=1)
    V = np.repeat(V, g, axis=1)
    S = scale * np.matmul(Q, np.swapaxes(K, -1, -2))
    if causal:
        Nq, Nkv = S.shape[-2:]
        S = np.where(np.arange(Nkv)[None, :] <= np.arange(Nq)[:, None], S, -np.inf)
    return np.matmul(softmax(S, axis=-1), V), logsumexp(S, axis=-1)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(2, 4, 2, 37, 53, 32), (1, 8, 1, 70, 41, 16), (1, 2, 2, 129, 129, 64)])
def test_matches_scipy(dtype, causal, shape):
    Z, Hq, Hkv, Nq, Nkv, D = shape
    q, k, v = si.qkv(4, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    scale = 1 / math.sqrt(D)
    o, lse = oracle.attention_fwd(q, k, v, dtype, scale, causal)
    o_ref, lse_ref = _scipy_attention(q, k, v, dtype, scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------- invariants ----

def test_gqa_equals_mha_on_repeated_kv():
    q, k, v = si.qkv(8, 2, 8, 2, 33, 45, 32, "bf16")
    for causal in (False, True):
        o, lse = oracle.attention_fwd(q, k, v, "bf16", 0.2, causal)
        o2, lse2 = oracle.attention_fwd(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), "bf16", 0.2, causal)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    # and a different grouping of the same K/V heads is a different answer
    o3, _ = oracle.attention_fwd(q, np.tile(k, (1, 4, 1, 1)), np.tile(v, (1, 4, 1, 1)), "bf16", 0.2, False)
    assert not np.allclose(o, o3)


def test_key_permutation_invariance():
    q, k, v = si.qkv(12, 1, 2, 1, 17, 64, 32, "fp16")
    perm = np.random.default_rng(0).permutation(64)
    o, lse = oracle.attention_fwd(q, k, v, "fp16", 0.17, False)
    o2, lse2 = oracle.attention_fwd(q, k[:, :, perm], v[:, :, perm], "fp16", 0.17, False)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-13)


def test_causal_row_is_prefix_attention():
    q, k, v = si.qkv(13, 1, 2, 2, 40, 40, 16, "fp16")
    o, lse = oracle.attention_fwd(q, k, v, "fp16", 0.3, True)
    for i in (0, 1, 7, 31, 39):
        op, lp = oracle.attention_fwd(q[:, :, i:i + 1], k[:, :, : i + 1], v[:, :, : i + 1], "fp16", 0.3, False)
        assert np.array_equal(o[:, :, i], op[:, :, 0]) and np.array_equal(lse[:, :, i], lp[:, :, 0])


def test_causal_top_left_when_nq_exceeds_nkv():
    # row i keeps keys j <= i: rows i >= Nkv - 1 see every key
    q, k, v = si.qkv(14, 1, 1, 1, 30, 12, 16, "bf16")
    oc, lc = oracle.attention_fwd(q, k, v, "bf16", 0.3, True)
    on, ln = oracle.attention_fwd(q, k, v, "bf16", 0.3, False)
    assert np.array_equal(oc[0, 0, 11:], on[0, 0, 11:]) and np.array_equal(lc[0, 0, 11:], ln[0, 0, 11:])
    assert not np.allclose(oc[0, 0, :11], on[0, 0, :11])


def test_row_subset_equals_full():
    q, k, v = si.qkv(15, 2, 4, 2, 50, 60, 32, "fp16")
    o, lse = oracle.attention_fwd(q, k, v, "fp16", 0.2, True)
    rows = np.array([0, 49, 50, 199, 201, 399, 123])
    os_, ls_ = oracle.attention_fwd(q, k, v, "fp16", 0.2, True, rows=rows)
    assert np.array_equal(os_, o.reshape(-1, 32)[rows]) and np.array_equal(ls_, lse.reshape(-1)[rows])


def test_threads_do_not_change_results():
    q, k, v = si.qkv(16, 1, 4, 4, 64, 64, 32, "bf16")
    a = oracle.attention_fwd(q, k, v, "bf16", 0.2, False, nthreads=1)
    b = oracle.attention_fwd(q, k, v, "bf16", 0.2, False, nthreads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_rejects_invalid_arguments():
    q, k, v = si.qkv(0, 1, 3, 2, 4, 4, 16, "fp16")
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, k, v, "fp16", 0.1, False)          # Hq % Hkv != 0
    q, k, v = si.qkv(0, 1, 2, 1, 4, 4, 16, "fp16")
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, k, v, "fp16", float("nan"), False)
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, k, v, "fp16", 0.1, False, rows=np.array([8]))


# ------------------------------------------------- merge over disjoint key sets ----
# The sum over a union of key sets is the sum of the per-set sums: merging the
# oracle's results over key shards must reproduce its result over all keys.

@pytest.mark.parametrize("cuts", [(0, 40, 97), (0, 1, 96, 97), (0, 13, 50, 51, 97)])
def test_merge_of_key_shards_is_attention_over_their_union(cuts):
    dtype = "fp16"
    q, k, v = si.qkv(21, 2, 4, 2, 19, 97, 32, dtype)
    scale = 0.7  # score spread of a few units, so the shards' lse differ widely
    o_full, lse_full = oracle.attention_fwd(q, k, v, dtype, scale, False)
    parts = [oracle.attention_fwd(q, k[:, :, a:b], v[:, :, a:b], dtype, scale, False) for a, b in zip(cuts, cuts[1:])]
    assert max(np.ptp(np.stack([p[1] for p in parts]), axis=0).ravel()) > 2.0
    o, lse = oracle.lse_merge([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(o, o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_full, rtol=0, atol=1e-12)


def test_merge_single_part_is_identity():
    rng = np.random.default_rng(3)
    o = rng.standard_normal((3, 5, 16))
    lse = rng.standard_normal((3, 5)) * 10
    mo, ml = oracle.lse_merge([o], [lse])
    assert np.array_equal(mo, o) and np.array_equal(ml, lse)


def test_merge_two_parts_closed_form():
    # lse = log 1 and log 3: weights 1/4 and 3/4, merged lse = log 4
    rng = np.random.default_rng(4)
    o1, o2 = rng.standard_normal((2, 7, 8))
    mo, ml = oracle.lse_merge([o1, o2], [np.full(7, 0.0), np.full(7, math.log(3.0))])
    np.testing.assert_allclose(mo, (o1 + 3 * o2) / 4, rtol=0, atol=1e-14)
    np.testing.assert_allclose(ml, math.log(4.0), rtol=0, atol=1e-14)


def test_merge_equal_lse_gives_mean_and_log_count():
    rng = np.random.default_rng(5)
    parts = [rng.standard_normal((4, 8)) for _ in range(5)]
    c = 123.25  # far from 0: the shift by the maximum matters
    mo, ml = oracle.lse_merge(parts, [np.full(4, c)] * 5)
    np.testing.assert_allclose(mo, np.mean(parts, axis=0), rtol=0, atol=1e-14)
    np.testing.assert_allclose(ml, c + math.log(5.0), rtol=0, atol=1e-12)


def test_merge_ignores_empty_parts():
    rng = np.random.default_rng(6)
    a, b = rng.standard_normal((2, 6, 16))
    la, lb = rng.standard_normal((2, 6))
    junk = np.full((6, 16), 1e30)
    mo, ml = oracle.lse_merge([a, junk, b], [la, np.full(6, -np.inf), lb])
    ro, rl = oracle.lse_merge([a, b], [la, lb])
    assert np.array_equal(mo, ro) and np.array_equal(ml, rl)
    eo, el = oracle.lse_merge([a, b], [np.full(6, -np.inf)] * 2)
    assert np.all(eo == 0) and np.all(el == -np.inf)


# ---------------------------------------------- variants: window, ALiBi, varlen ----
# Each variant is pinned by reducing it to the (pinned) base definition on
# sliced or extended inputs, or by closed-form properties of its weights.

@pytest.mark.parametrize("causal", [False, True])
def test_ex_with_no_variant_is_the_base_forward(causal):
    q, k, v = si.qkv(81, 2, 4, 2, 45, 70, 16, "bf16")
    a = oracle.attention_fwd(q, k, v, "bf16", 0.3, causal)
    b = oracle.attention_fwd_ex(q, k, v, "bf16", 0.3, causal)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def _row_on_slice(q, k, v, dtype, scale, z, hq, i, lo, hi, g):
    """The base forward for one query row against keys lo..hi-1 only."""
    qs = np.ascontiguousarray(q[z:z + 1, hq:hq + 1, i:i + 1])
    ks = np.ascontiguousarray(k[z:z + 1, hq // g:hq // g + 1, lo:hi])
    vs = np.ascontiguousarray(v[z:z + 1, hq // g:hq // g + 1, lo:hi])
    o, lse = oracle.attention_fwd(qs, ks, vs, dtype, scale, False)
    return o[0, 0, 0], lse[0, 0, 0]


@pytest.mark.parametrize("window,causal", [((5, 3), False), ((0, 0), False), ((10, -1), True), ((-1, 4), False),
                                           ((7, 2), True), ((3, -1), False)])
def test_window_is_attention_over_the_window(window, causal):
    dtype, scale = "fp16", 0.4
    Z, Hq, Hkv, Nq, Nkv, D = 1, 2, 1, 37, 44, 16
    q, k, v = si.qkv(82, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    o, lse = oracle.attention_fwd_ex(q, k, v, dtype, scale, causal, window=window)
    wl, wr = window
    for hq in range(Hq):
        for i in range(Nq):
            lo = 0 if wl < 0 else max(0, i - wl)
            hi = Nkv if wr < 0 else min(Nkv, i + wr + 1)
            if causal:
                hi = min(hi, i + 1)
            if lo >= hi:
                assert np.all(o[0, hq, i] == 0) and lse[0, hq, i] == -np.inf
                continue
            ro, rl = _row_on_slice(q, k, v, dtype, scale, 0, hq, i, lo, hi, Hq // Hkv)
            np.testing.assert_allclose(o[0, hq, i], ro, rtol=0, atol=1e-12)
            assert abs(lse[0, hq, i] - rl) <= 1e-12


def test_window_with_no_key_gives_zero_and_neg_inf():
    q, k, v = si.qkv(83, 1, 1, 1, 30, 10, 16, "fp16")
    o, lse = oracle.attention_fwd_ex(q, k, v, "fp16", 0.5, False, window=(0, 0))
    # row i keeps only key i: rows 10.. have none
    assert np.all(o[0, 0, 10:] == 0) and np.all(lse[0, 0, 10:] == -np.inf)
    V = si.as_torch(v, "fp16").double().numpy()
    np.testing.assert_array_equal(o[0, 0, :10], V[0, 0, :10])


@pytest.mark.parametrize("causal", [False, True])
def test_alibi_is_an_extra_dimension_where_the_distance_has_one_sign(causal):
    # For keys j <= i the bias -s (i - j) = s j - s i: the same softmax as one
    # extra dimension with q = 1 and k_j = s j / scale (exact in fp16 here),
    # with lse shifted by -s i.  Keys j >= i (row 0) take k_j = -s j / scale.
    dtype, scale = "fp16", 0.25
    Z, Hq, Hkv, N, D = 1, 2, 1, 60, 16
    slopes = np.array([1 / 64, 1 / 32])
    q, k, v = si.qkv(84, Z, Hq, Hkv, N, N, D, dtype)
    o, lse = oracle.attention_fwd_ex(q, k, v, dtype, scale, causal, alibi=slopes)
    one = si.round_bits(np.ones((Z, 1, N, 1)), dtype)
    for hq in range(Hq):
        s = slopes[hq]
        for sign, rows in ((+1, range(N) if causal else [N - 1]), (-1, [0])):
            col = si.round_bits((sign * s / scale) * np.arange(N, dtype=np.float64).reshape(1, 1, N, 1), dtype)
            assert np.array_equal(si.as_torch(col, dtype).double().numpy().ravel(),
                                  (sign * s / scale) * np.arange(N))  # exact
            qx = np.concatenate([q[:, hq:hq + 1], one], axis=3)
            kx = np.concatenate([k, col], axis=3)
            vx = v
            bo, bl = oracle.attention_fwd(qx, kx, np.concatenate([vx, si.round_bits(np.zeros((1, 1, N, 1)), dtype)],
                                                                 axis=3), dtype, scale, causal)
            for i in rows:
                np.testing.assert_allclose(o[0, hq, i], bo[0, 0, i, :D], rtol=0, atol=1e-12)
                assert abs(lse[0, hq, i] - (bl[0, 0, i] - sign * s * i)) <= 1e-11


def test_alibi_weights_decay_geometrically_and_symmetrically():
    # Q = 0 leaves only the bias: with V = I the output row is the weight row
    # P_ij proportional to exp(-s |i - j|)
    dtype, N, s = "fp16", 16, 0.3
    q = si.round_bits(np.zeros((1, 1, N, N)), dtype)
    k = si.round_bits(np.ones((1, 1, N, N)), dtype)
    v = si.round_bits(np.eye(N).reshape(1, 1, N, N), dtype)
    P, lse = oracle.attention_fwd_ex(q, k, v, dtype, 0.7, False, alibi=[s])
    P = P[0, 0]
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    for i in range(N):
        for j in range(i, N - 1):
            assert abs(P[i, j] / P[i, j + 1] - math.exp(s)) < 1e-12
        for d in range(1, min(i, N - 1 - i) + 1):
            assert abs(P[i, i - d] - P[i, i + d]) < 1e-15
    # lse = log sum_j exp(-s |i - j|), a finite geometric sum
    i = 5
    want = math.log(sum(math.exp(-s * abs(i - j)) for j in range(N)))
    assert abs(lse[0, 0, i] - want) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_is_attention_per_sequence(causal):
    dtype, scale, D, Hq, Hkv = "bf16", 0.3, 32, 4, 2
    cu_q = np.array([0, 5, 5, 140, 200], dtype=np.int32)
    cu_k = np.array([0, 7, 30, 30, 330], dtype=np.int32)
    tq, tk = 210, 340  # packed extents; rows 200.. belong to no sequence
    q = si.normals(85, 0, Hq * tq * D, dtype).reshape(1, Hq, tq, D)
    k = si.normals(85, q.size, Hkv * tk * D, dtype).reshape(1, Hkv, tk, D)
    v = si.normals(85, q.size + k.size, Hkv * tk * D, dtype).reshape(1, Hkv, tk, D)
    o, lse = oracle.attention_fwd_ex(q, k, v, dtype, scale, causal, cu_q=cu_q, cu_k=cu_k)
    for z in range(4):
        a, b, c, d = cu_q[z], cu_q[z + 1], cu_k[z], cu_k[z + 1]
        if b == a:
            continue
        if d == c:  # no keys: every row of the sequence is empty
            assert np.all(o[0, :, a:b] == 0) and np.all(lse[0, :, a:b] == -np.inf)
            continue
        ro, rl = oracle.attention_fwd(q[:, :, a:b], k[:, :, c:d], v[:, :, c:d], dtype, scale, causal)
        np.testing.assert_allclose(o[:, :, a:b], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, :, a:b], rl, rtol=0, atol=1e-12)
    assert np.all(np.isnan(o[0, :, 200:])) and np.all(np.isnan(lse[0, :, 200:]))


# ---------------------------------------------------------------- backward ----
# The gradients are pinned by central finite differences of an independent
# float64 forward (numpy matmul + scipy softmax), by closed forms, and by the
# GQA reduction.

def _np_forward(Q, K, V, scale, causal):
    """float64 attention forward from library routines, for finite differences."""
    from scipy.special import softmax
    Z, Hq, Nq, D = Q.shape
    g = Hq // K.shape[1]
    O = np.empty_like(Q)
    for z in range(Z):
        for h in range(Hq):
            S = scale * Q[z, h] @ K[z, h // g].T
            if causal:
                S = np.where(np.arange(K.shape[2])[None, :] > np.arange(Nq)[:, None], -np.inf, S)
            O[z, h] = softmax(S, axis=1) @ V[z, h // g]
    return O


@pytest.mark.parametrize("dtype,causal,shape", [("fp16", False, (1, 2, 1, 7, 9, 8)), ("bf16", True, (2, 4, 2, 9, 6, 4)),
                                                ("fp16", True, (1, 2, 2, 5, 5, 16))])
def test_bwd_matches_finite_differences(dtype, causal, shape):
    Z, Hq, Hkv, Nq, Nkv, D = shape
    scale = 0.6
    q, k, v = si.qkv(111, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    do = si.normals(112, 0, q.size, dtype).reshape(q.shape)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, dtype, scale, causal)
    Q, K, V, G = (_np_decode(x, dtype) for x in (q, k, v, do))

    def loss(Qx, Kx, Vx):
        return float(np.sum(G * _np_forward(Qx, Kx, Vx, scale, causal)))

    rng = np.random.default_rng(7)
    h = 1e-5
    for name, X, grad in (("q", Q, dq), ("k", K, dk), ("v", V, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(n)) for n in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"q": (Xp, K, V), "k": (Q, Xp, V), "v": (Q, K, Xp)}[name]
            args_m = {"q": (Xm, K, V), "k": (Q, Xm, V), "v": (Q, K, Xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_bwd_single_key_closed_form():
    # one key: P = 1, so dS = 0 (dQ = dK = 0) and dV_0 is the sum of dO over the group's rows
    q, k, v = si.qkv(113, 2, 4, 2, 6, 1, 8, "fp16")
    do = si.normals(114, 0, q.size, "fp16").reshape(q.shape)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, "fp16", 0.9, False)
    G = _np_decode(do, "fp16")
    assert np.all(dq == 0) and np.all(dk == 0)
    for z in range(2):
        for hk in range(2):
            np.testing.assert_allclose(dv[z, hk, 0], G[z, 2 * hk:2 * hk + 2].sum(axis=(0, 1)), rtol=0, atol=1e-12)


def test_bwd_scale_zero_closed_form():
    # scale 0: uniform P over the kept keys, dQ = dK = 0, dV_j = sum over rows keeping j of dO_i / n_i
    Nq = Nkv = 7
    q, k, v = si.qkv(115, 1, 1, 1, Nq, Nkv, 8, "bf16")
    do = si.normals(116, 0, q.size, "bf16").reshape(q.shape)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, "bf16", 0.0, True)
    G = _np_decode(do, "bf16")[0, 0]
    assert np.all(dq == 0) and np.all(dk == 0)
    for j in range(Nkv):
        want = sum(G[i] / (i + 1) for i in range(j, Nq))
        np.testing.assert_allclose(dv[0, 0, j], want, rtol=0, atol=1e-12)


def test_bwd_gqa_is_mha_summed_over_the_group():
    q, k, v = si.qkv(117, 1, 4, 1, 10, 12, 8, "fp16")
    do = si.normals(118, 0, q.size, "fp16").reshape(q.shape)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, "fp16", 0.4, True)
    kr, vr = np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1)
    mq, mk, mv = oracle.attention_bwd(q, kr, vr, do, "fp16", 0.4, True)
    np.testing.assert_allclose(dq, mq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk[:, 0], mk.sum(axis=1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv[:, 0], mv.sum(axis=1), rtol=0, atol=1e-12)


def test_bwd_causal_first_row_has_no_query_gradient():
    q, k, v = si.qkv(119, 1, 2, 2, 8, 8, 8, "fp16")
    do = si.normals(120, 0, q.size, "fp16").reshape(q.shape)
    dq, _, _ = oracle.attention_bwd(q, k, v, do, "fp16", 0.7, True)
    assert np.all(dq[:, :, 0] == 0) and np.any(dq[:, :, 1] != 0)


# ------------------------------------------------------- backward, variants ----
# The window / ALiBi backward (attention_bwd_ex): without a variant it is the
# plain backward bit for bit; it matches central finite differences of an
# independent float64 forward with the same readings (numpy + scipy: kept keys
# i - left <= j <= i + right, causal j <= i, bias -slope |i - j|, a row with no
# kept key O = 0); and a window of the diagonal alone is a closed form.

def _np_forward_ex(Q, K, V, scale, causal, window, alibi):
    from scipy.special import softmax
    Z, Hq, Nq, D = Q.shape
    g = Hq // K.shape[1]
    Nkv = K.shape[2]
    i = np.arange(Nq)[:, None]
    j = np.arange(Nkv)[None, :]
    keep = np.ones((Nq, Nkv), dtype=bool)
    if causal:
        keep &= j <= i
    if window[0] >= 0:
        keep &= j >= i - window[0]
    if window[1] >= 0:
        keep &= j <= i + window[1]
    O = np.zeros_like(Q)
    for z in range(Z):
        for h in range(Hq):
            S = scale * Q[z, h] @ K[z, h // g].T
            if alibi is not None:
                S = S - alibi[h] * np.abs(i - j)
            S = np.where(keep, S, -np.inf)
            rows = keep.any(axis=1)
            P = np.zeros_like(S)
            P[rows] = softmax(S[rows], axis=1)
            O[z, h] = P @ V[z, h // g]
    return O


@pytest.mark.parametrize("dtype,causal", [("fp16", False), ("bf16", True)])
def test_bwd_ex_without_variants_is_the_plain_backward(dtype, causal):
    q, k, v = si.qkv(121, 2, 4, 2, 13, 11, 16, dtype)
    do = si.normals(122, 0, q.size, dtype).reshape(q.shape)
    plain = oracle.attention_bwd(q, k, v, do, dtype, 0.5, causal)
    ex = oracle.attention_bwd_ex(q, k, v, do, dtype, 0.5, causal, window=(-1, -1), alibi=None)
    for a, b in zip(plain, ex):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("dtype,causal,window,alibi,shape", [
    ("fp16", False, (2, 1), None, (1, 2, 1, 9, 9, 8)),
    ("bf16", True, (3, -1), [0.5, 0.125], (1, 2, 2, 8, 10, 4)),
    ("fp16", False, (-1, 2), [0.25, 1.0, 0.0, 0.75], (2, 4, 2, 7, 6, 8)),
    ("fp16", True, (1, -1), None, (1, 2, 1, 12, 5, 4)),      # rows past the keys keep none
])
def test_bwd_ex_matches_finite_differences(dtype, causal, window, alibi, shape):
    Z, Hq, Hkv, Nq, Nkv, D = shape
    scale = 0.6
    slopes = None if alibi is None else np.asarray(alibi, dtype=np.float64)
    q, k, v = si.qkv(123, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    do = si.normals(124, 0, q.size, dtype).reshape(q.shape)
    dq, dk, dv = oracle.attention_bwd_ex(q, k, v, do, dtype, scale, causal, window=window, alibi=slopes)
    Q, K, V, G = (_np_decode(x, dtype) for x in (q, k, v, do))

    def loss(Qx, Kx, Vx):
        return float(np.sum(G * _np_forward_ex(Qx, Kx, Vx, scale, causal, window, slopes)))

    rng = np.random.default_rng(8)
    h = 1e-5
    for name, X, grad in (("q", Q, dq), ("k", K, dk), ("v", V, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(n)) for n in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"q": (Xp, K, V), "k": (Q, Xp, V), "v": (Q, K, Xp)}[name]
            args_m = {"q": (Xm, K, V), "k": (Q, Xm, V), "v": (Q, K, Xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_bwd_ex_diagonal_window_closed_form():
    # window (0, 0): each query keeps only key i, so O_i = v_i, P = 1 there:
    # dV_i = dO_i (summed over the group's query heads), dS = 0, so dQ = dK = 0;
    # queries past the keys keep nothing
    q, k, v = si.qkv(125, 1, 4, 2, 9, 7, 8, "bf16")
    do = si.normals(126, 0, q.size, "bf16").reshape(q.shape)
    dq, dk, dv = oracle.attention_bwd_ex(q, k, v, do, "bf16", 0.8, False, window=(0, 0), alibi=[0.3, 0.1, 0.0, 2.0])
    G = _np_decode(do, "bf16")
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    want = np.stack([G[0, 0:2, :7].sum(axis=0), G[0, 2:4, :7].sum(axis=0)])[None]
    np.testing.assert_allclose(dv, want, rtol=0, atol=1e-12)


def test_bwd_ex_varlen_matches_finite_differences():
    # packed sequences (one without keys, one of a single row): central
    # differences of the independent numpy forward run sequence by sequence
    lens_q, lens_k = [5, 0, 1, 7], [6, 3, 0, 4]
    cq = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    Hq, Hkv, D, dtype, scale, causal, window = 4, 2, 8, "fp16", 0.7, True, (4, -1)
    slopes = np.array([0.5, 0.0, 0.25, 1.0])
    tq, tk = int(cq[-1]), int(ck[-1])
    q = si.normals(131, 0, Hq * tq * D, dtype).reshape(1, Hq, tq, D)
    k = si.normals(131, q.size, Hkv * tk * D, dtype).reshape(1, Hkv, tk, D)
    v = si.normals(131, q.size + k.size, Hkv * tk * D, dtype).reshape(1, Hkv, tk, D)
    do = si.normals(132, 0, q.size, dtype).reshape(q.shape)
    dq, dk, dv = oracle.attention_bwd_ex(q, k, v, do, dtype, scale, causal, window=window, alibi=slopes,
                                         cu_q=cq, cu_k=ck)
    Q, K, V, G = (_np_decode(x, dtype) for x in (q, k, v, do))

    def loss(Qx, Kx, Vx):
        total = 0.0
        for z in range(len(lens_q)):
            a, b, c, e = cq[z], cq[z + 1], ck[z], ck[z + 1]
            if b == a or e == c:
                continue
            O = _np_forward_ex(Qx[:, :, a:b], Kx[:, :, c:e], Vx[:, :, c:e], scale, causal, window, slopes)
            total += float(np.sum(G[:, :, a:b] * O))
        return total

    rng = np.random.default_rng(9)
    h = 1e-5
    for name, X, grad in (("q", Q, dq), ("k", K, dk), ("v", V, dv)):
        for _ in range(16):
            idx = tuple(int(rng.integers(n)) for n in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"q": (Xp, K, V), "k": (Q, Xp, V), "v": (Q, K, Xp)}[name]
            args_m = {"q": (Xm, K, V), "k": (Q, Xm, V), "v": (Q, K, Xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])
    # the sequence without keys has no query gradient
    assert np.all(dq[:, :, cq[1]:cq[2]] == 0.0) and np.all(dq[:, :, cq[2]:cq[3]] == 0.0)
