"""Property tests of the oracle on random small shapes (CPU, hypothesis).

Invariants that hold for every shape, drawn over head dims, q-heads per kv-head ratios (1, 2, 4, 7), ragged
lengths and selections at or above T:
  - selecting at least T tokens is a no-op: decode equals plain attention over the rotated rebuilt keys and the
    predicted values;
  - RoPE's inverse undoes it at any position;
  - the log-sum-exp merge is commutative and associative, including empty sets (lse = -inf);
  - the attention mass is non-negative and each sequence's mass sums to W * H_q;
  - the eviction plan holds exactly T_keep ascending tokens, every sink and recent token, and no dropped token
    outweighs a kept one (equal weights go to the lower index);
  - the int4 and int8 quantisers stay within half a step of their input at magnitudes from 1e-3 to 1e4, keep their
    codes in range, take their scales from the group's (vector's) largest entry, and map an all-zero group to 0.
"""
import numpy as np
import pytest
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

import oracle as O

SETTINGS = settings(max_examples=25, deadline=None, suppress_health_check=[HealthCheck.too_slow])


@st.composite
def decode_case(draw):
    B = draw(st.integers(1, 2))
    T = draw(st.integers(1, 37))
    H_kv = draw(st.integers(1, 2))
    g = draw(st.sampled_from([1, 2, 4, 7]))
    d = draw(st.sampled_from([8, 16]))
    r = draw(st.sampled_from([4, 8]))
    m = draw(st.sampled_from([4, 8]))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return B, T, H_kv, g, d, r, m, seed


@SETTINGS
@given(decode_case(), st.integers(0, 5))
def test_selecting_every_token_is_plain_attention(case, extra):
    B, T, H_kv, g, d, r, m, seed = case
    rng = np.random.default_rng(seed)
    q = rng.normal(0, 1, (B, H_kv * g, d))
    coef = rng.normal(0, 1, (B, T, r))
    basis = rng.normal(0, r ** -0.5, (H_kv * d, r))
    w1, w2 = rng.normal(0, d ** -0.5, (H_kv, m, d)), rng.normal(0, m ** -0.5, (H_kv, d, m))
    theta = 1e4
    res = O.decode(q, coef, basis, w1, w2, S=T + extra, theta=theta)
    k_pre = O.rebuild_keys(coef, basis, H_kv, d)
    k = O.rope_rows(k_pre, np.broadcast_to(np.arange(T)[None, :, None], (B, T, H_kv)), theta)
    v = O.predict_values(k_pre, w1, w2)
    out, lse = O.dense_decode(q, k, v)
    np.testing.assert_allclose(res.out, out, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(res.lse, lse, rtol=1e-12, atol=1e-12)


@SETTINGS
@given(st.sampled_from([8, 64, 128]), st.integers(0, 100000), st.sampled_from([1e4, 5e5]), st.integers(0, 2 ** 31 - 1))
def test_rope_inverse_undoes_rope(d, pos, theta, seed):
    x = np.random.default_rng(seed).normal(0, 1, (3, d))
    y = O.rope_rows(x, np.full(3, pos), theta)
    np.testing.assert_allclose(O.rope_rows(y, np.full(3, pos), theta, inverse=True), x, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)


def _part(rng, shape, d):
    lse = rng.normal(0, 3, shape)
    lse[rng.random(shape) < 0.25] = -np.inf
    out = np.where(np.isneginf(lse)[..., None], 0.0, rng.normal(0, 1, shape + (d,)))
    return out, lse


@SETTINGS
@given(st.integers(0, 2 ** 31 - 1))
def test_merge_is_commutative_and_associative(seed):
    rng = np.random.default_rng(seed)
    a, b, c = (_part(rng, (2, 5), 4) for _ in range(3))
    ab = O.merge_attn(*a, *b)
    ba = O.merge_attn(*b, *a)
    np.testing.assert_allclose(ab[0], ba[0], atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(ab[1]), np.isneginf(ba[1]))
    left = O.merge_attn(*ab, *c)
    right = O.merge_attn(*a, *O.merge_attn(*b, *c))
    np.testing.assert_allclose(left[0], right[0], atol=1e-10)
    fin = np.isfinite(left[1])
    np.testing.assert_array_equal(fin, np.isfinite(right[1]))
    np.testing.assert_allclose(left[1][fin], right[1][fin], atol=1e-10)


@SETTINGS
@given(st.integers(1, 2), st.integers(1, 30), st.integers(1, 4), st.sampled_from([1, 2, 4, 7]),
       st.integers(0, 2 ** 31 - 1))
def test_attention_mass_is_a_distribution_per_window_query(B, T, W, g, seed):
    rng = np.random.default_rng(seed)
    H_kv, d = 2, 8
    q = rng.normal(0, 2, (B, W, H_kv * g, d))
    k = rng.normal(0, 1, (B, T, H_kv, d))
    mass = O.attention_mass(q, k)
    assert mass.shape == (B, T) and np.all(mass >= 0)
    np.testing.assert_allclose(mass.sum(axis=1), W * H_kv * g, rtol=1e-12)


@SETTINGS
@given(st.integers(1, 60), st.data())
def test_evict_plan_keeps_the_forced_and_the_heaviest(T, data):
    n_sink = data.draw(st.integers(0, T))
    n_recent = data.draw(st.integers(0, T - n_sink))
    T_keep = data.draw(st.integers(n_sink + n_recent, T))
    mass = np.asarray(data.draw(st.lists(st.integers(0, 4), min_size=T, max_size=T)), dtype=np.float64)[None]
    keep = O.evict_plan(mass, n_sink, n_recent, T_keep)[0].tolist()
    assert len(keep) == T_keep and keep == sorted(set(keep))
    forced = set(range(n_sink)) | set(range(T - n_recent, T))
    assert forced <= set(keep)
    kept_free = [t for t in keep if t not in forced]
    dropped = [t for t in range(T) if t not in set(keep)]
    for t in kept_free:
        for u in dropped:
            assert (mass[0, t], -t) > (mass[0, u], -u)        # heavier, or as heavy and earlier


@SETTINGS
@given(st.integers(1, 6), st.sampled_from([32, 64, 128]), st.floats(-3, 4), st.integers(0, 2 ** 31 - 1))
def test_int4_quantiser_bound_range_and_zero_groups(rows, r, log_mag, seed):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 10.0 ** log_mag, (rows, r))
    x[0, :32] = 0.0                                          # an all-zero group: scale 0, codes 0
    packed, scales = O.quant_int4_g32(x)
    deq = O.dequant_int4_g32(packed, scales)
    s = np.repeat(scales, 32, axis=1)
    assert scales[0, 0] == 0 and np.all(deq[0, :32] == 0)
    assert np.all(np.abs(x - deq) <= s / 2 * (1 + 1e-3) + 1e-300)
    nz = s > 0
    assert np.all(np.abs(np.round(deq[nz] / s[nz])) <= 7)
    amax = np.abs(x).reshape(rows, r // 32, 32).max(-1)
    np.testing.assert_array_equal(scales, np.float16(amax / 7).astype(np.float64))


@SETTINGS
@given(st.integers(1, 6), st.sampled_from([64, 128]), st.floats(-3, 4), st.integers(0, 2 ** 31 - 1))
def test_int8_quantiser_bound_and_range(rows, d, log_mag, seed):
    x = np.random.default_rng(seed).normal(0, 10.0 ** log_mag, (rows, d))
    codes, sc = O.quant_int8_vec(x)
    deq = O.dequant_int8_vec(codes, sc)
    assert np.abs(codes.astype(int)).max() <= 127
    assert np.all(np.abs(x - deq) <= sc[:, None] / 2 * (1 + 1e-3) + 1e-300)
    np.testing.assert_array_equal(sc, np.float16(np.abs(x).max(axis=1) / 127).astype(np.float64))
