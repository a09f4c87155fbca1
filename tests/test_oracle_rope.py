"""Pins of the oracle's rotary positions (apply_rope, rope_chunk) to things other than themselves.

"KV cache decoding", "Position information with a cache": the query and key are rotated by an angle
of their absolute position, keys are stored rotated, the score then depends only on the distance
between the two positions, and cached keys never need updating. The formula is the RoFormer paper's
(Su et al., eq. 34), which the pages name but do not print.
"""
import math

import numpy as np
import pytest

from oracle.kvc_oracle import (OracleKVCache, apply_rope, full_recompute_attention, gqa_cached_attention,
                               rope_chunk, rope_pairs, rope_theta)

STYLES = ["half", "interleaved"]


@pytest.mark.parametrize("style", STYLES)
def test_position_zero_is_the_identity(style):
    x = np.random.default_rng(1).standard_normal((5, 16))
    assert np.array_equal(apply_rope(x, np.zeros(5), 10000.0, style), x)


@pytest.mark.parametrize("style", STYLES)
def test_two_dims_turn_by_the_position_in_radians(style):
    """d = 2 has one pair with theta_0 = base^0 = 1: the unit vector e_0 at position p becomes
    (cos p, sin p), for any base."""
    for base in (10.0, 10000.0, 500000.0):
        for p in (1, 2, 7, 4095):
            got = apply_rope(np.array([[1.0, 0.0]]), [p], base, style)[0]
            assert got[0] == pytest.approx(math.cos(p), abs=1e-15)
            assert got[1] == pytest.approx(math.sin(p), abs=1e-15)


@pytest.mark.parametrize("style", STYLES)
def test_pair_frequencies_form_a_geometric_series(style):
    """Recovered from the rotation itself (atan2 of a rotated unit vector at position 1): the first
    pair turns by 1 radian, each next one by base^(-2/d) times as much, the last by base^(-(d-2)/d)."""
    d, base = 16, 10000.0
    a, b = rope_pairs(d, style)
    ang = []
    for i in range(d // 2):
        e = np.zeros((1, d))
        e[0, a[i]] = 1.0
        r = apply_rope(e, [1], base, style)[0]
        ang.append(math.atan2(r[b[i]], r[a[i]]))
    ang = np.array(ang)
    assert ang[0] == pytest.approx(1.0, abs=1e-15)
    assert np.allclose(ang[1:] / ang[:-1], math.exp(-2.0 * math.log(base) / d), rtol=1e-12, atol=0)
    assert ang[-1] == pytest.approx(math.exp(-(d - 2) / d * math.log(base)), rel=1e-12)


@pytest.mark.parametrize("style", STYLES)
def test_rotation_preserves_each_pair_norm(style):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((6, 32))
    pos = rng.integers(0, 5000, 6)
    y = apply_rope(x, pos, 10000.0, style)
    a, b = rope_pairs(32, style)
    assert np.allclose(x[:, a] ** 2 + x[:, b] ** 2, y[:, a] ** 2 + y[:, b] ** 2, rtol=1e-13, atol=0)


@pytest.mark.parametrize("style", STYLES)
def test_scores_depend_only_on_the_distance(style):
    """q.k after rotating q to position i and k to position j is the same for (i + s, j + s)."""
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((2, 64))
    for i, j in ((10, 3), (0, 0), (4000, 17), (5, 900)):
        ref = apply_rope(q[None], [i], 10000.0, style)[0] @ apply_rope(k[None], [j], 10000.0, style)[0]
        for shift in (1, 100, 3000):
            got = apply_rope(q[None], [i + shift], 10000.0, style)[0] @ \
                apply_rope(k[None], [j + shift], 10000.0, style)[0]
            assert got == pytest.approx(ref, abs=1e-10)


def test_interleaved_is_half_on_permuted_coordinates():
    """The two layouts rotate the same pairs once the coordinates are permuted: interleaved(x) =
    P^-1 half(P x) with P gathering the even elements then the odd ones."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 12))
    pos = [0, 1, 33, 1000]
    perm = np.concatenate([np.arange(0, 12, 2), np.arange(1, 12, 2)])
    inv = np.argsort(perm)
    got = apply_rope(x[:, perm], pos, 500000.0, "half")[:, inv]
    assert np.allclose(got, apply_rope(x, pos, 500000.0, "interleaved"), rtol=0, atol=1e-15)


def test_theta_values():
    th = rope_theta(8, 10000.0)
    assert th[0] == 1.0 and len(th) == 4
    assert th[2] == pytest.approx(0.01, rel=1e-15)       # 10000^(-4/8) = 1/100


@pytest.mark.parametrize("style", STYLES)
def test_cached_rotated_keys_equal_full_recompute(style):
    """Keys rotated once at their own positions and cached, queries rotated at s + t: every step
    equals the uncached pass that rotates the whole sequence at positions 0 .. n-1 (cached keys never
    need updating)."""
    rng = np.random.default_rng(5)
    H_q, H_kv, d, n = 4, 2, 16, 30
    q = rng.standard_normal((H_q, n, d))
    k = rng.standard_normal((H_kv, n, d))
    v = rng.standard_normal((H_kv, n, d))
    base = 10000.0
    full = full_recompute_attention(apply_rope(q, np.arange(n), base, style),
                                    apply_rope(k, np.arange(n), base, style), v)
    cache = OracleKVCache(1, 1, H_kv, d, n, "f64")
    s = 0
    for T in (7, 1, 1, 5, 16):
        starts = cache.committed()
        kr = np.stack([apply_rope(k[h, s:s + T], starts[0] + np.arange(T), base, style) for h in range(H_kv)])
        cache.append(0, kr[None], v[None, :, s:s + T])
        qr = np.stack([apply_rope(q[h, s:s + T], starts[0] + np.arange(T), base, style) for h in range(H_q)])
        out = gqa_cached_attention(cache, 0, qr[None])[0]
        assert np.abs(out - full[:, s:s + T]).max() < 1e-12
        cache.commit()
        s += T


def test_rope_chunk_positions_follow_each_sequence():
    """rope_chunk rotates row t of sequence b at starts[b] + t and rounds to float32."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 2, 4, 8)).astype(np.float32)
    starts = [0, 5, 100]
    got = rope_chunk(x, starts, 10000.0, "half")
    assert got.dtype == np.float32
    for b in range(3):
        want = apply_rope(x[b], starts[b] + np.arange(4), 10000.0, "half").astype(np.float32)
        assert np.array_equal(got[b], want)
    assert np.array_equal(got[0, :, 0], x[0, :, 0])     # position 0 is the identity
