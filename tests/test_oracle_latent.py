"""Pins of the oracle's latent cache (OracleLatentCache) and multi-head latent attention
(mla_cached_attention) to things other than themselves.

* "KV cache, incremental decode, ...", §2.6 "The latent cache": the same rules as the KV cache
  (per-layer fill, committed length, rollback) and nbytes = L B N_max (r + d_R) itemsize; pinned by
  driving a latent and a (separately pinned) KV oracle with the same calls, and by hand values.
* The attention that reads the latent cache is DeepSeek-V2's MLA in its absorbed form; pinned against
  the unabsorbed computation with explicit per-head key and value up-projections (a different route
  to the same numbers), and by its reduction to single-K/V-head attention when k^R is zero.
"""
import numpy as np
import pytest

from oracle.kvc_oracle import (OracleKVCache, OracleLatentCache, apply_rope, attend, gqa_cached_attention,
                               mla_cached_attention, store_round, stored_to_f64)


def test_nbytes_by_hand():
    assert OracleLatentCache(2, 1, 4, 2, 8, "f32").nbytes() == 2 * 1 * 8 * (4 + 2) * 4      # 384
    assert OracleLatentCache(61, 1, 512, 64, 4096, "bf16").nbytes() == 61 * 4096 * 576 * 2


def test_same_rules_as_the_kv_cache():
    """Identical appends, commits and truncates give identical fills, lengths and positions, and the
    same errors (capacity, commit with unequal fills, truncate past the committed length)."""
    rng = np.random.default_rng(1)
    lat = OracleLatentCache(3, 2, 8, 4, 20, "bf16")
    kv = OracleKVCache(3, 2, 1, 8, 20, "bf16")
    for T in (5, 1, 3):
        for layer in range(3):
            c = rng.standard_normal((2, T, 8)).astype(np.float32)
            lat.append(layer, c, rng.standard_normal((2, T, 4)).astype(np.float32))
            kv.append(layer, c[:, None], c[:, None])
            assert np.array_equal(lat.seq_len(layer), kv.seq_len(layer))
            if layer < 2:
                with pytest.raises(RuntimeError):
                    lat.commit()
        lat.commit()
        kv.commit()
        assert np.array_equal(lat.committed(), kv.committed())
        assert np.array_equal(lat.positions(3), kv.positions(3))
    for c in (lat, kv):
        with pytest.raises(RuntimeError):
            c.truncate([10, 2])
        c.truncate([4, 9])
    assert np.array_equal(lat.committed(), kv.committed()) and np.array_equal(lat.fill, kv.fill)
    with pytest.raises(OverflowError):
        lat.append(0, np.zeros((2, 12, 8), np.float32), np.zeros((2, 12, 4), np.float32))


def test_rollback_then_reappend_equals_never_appended():
    rng = np.random.default_rng(2)
    a = OracleLatentCache(2, 1, 8, 4, 16, "f16")
    b = OracleLatentCache(2, 1, 8, 4, 16, "f16")
    chunks = [(rng.standard_normal((1, 6, 8)).astype(np.float32), rng.standard_normal((1, 6, 4)).astype(np.float32))
              for _ in range(3)]
    for c in (a, b):
        for layer in range(2):
            c.append(layer, *chunks[0])
        c.commit()
    for layer in range(2):
        a.append(layer, *chunks[1])
    a.commit()
    a.truncate(6)
    for c in (a, b):
        for layer in range(2):
            c.append(layer, *chunks[2])
        c.commit()
    for layer in range(2):
        for x, y in zip(a.stored_f64(layer, 0, 12), b.stored_f64(layer, 0, 12)):
            assert np.array_equal(x, y)


def test_stored_values_are_rounded_and_returned():
    c = OracleLatentCache(1, 1, 4, 2, 4, "bf16")
    x = np.array([[[1.0 + 2 ** -9, 3.14159, -2.5, 1e-3]]], np.float32)
    k = np.array([[[0.1, -7.0]]], np.float32)
    rows = c.append(0, x, k)
    assert np.array_equal(rows[0][0], stored_to_f64(store_round(x[0], "bf16"), "bf16"))
    assert np.array_equal(rows[0][1], stored_to_f64(store_round(k[0], "bf16"), "bf16"))


@pytest.mark.parametrize("T,lengths", [(1, [7, 0, 12]), (4, [3, 9, 0])])
def test_absorbed_mla_equals_explicit_per_head_projections(T, lengths):
    """Per head h: k_{h,j} = [W_uk[h] c_j ; k^R_j], v_{h,j} = W_uv[h] c_j, score = q_h . k_{h,j} * scale.
    With q_lat_h = W_uk[h]^T q_nope_h, the absorbed scores are the same, and W_uv[h] (sum_j p_j c_j)
    is the explicit output."""
    rng = np.random.default_rng(3 + T)
    B, H, r, dR, dn, dv = len(lengths), 4, 16, 8, 12, 10
    scale = 1.0 / np.sqrt(dn + dR)
    cache = OracleLatentCache(1, B, r, dR, 32, "f64")
    s0 = max(lengths)
    c_all = rng.standard_normal((B, s0 + T, r))
    kr_all = rng.standard_normal((B, s0 + T, dR))
    if s0:
        cache.append(0, c_all[:, :s0], kr_all[:, :s0])
        cache.commit()
        cache.truncate(lengths)
    c_new, kr_new = rng.standard_normal((B, T, r)), rng.standard_normal((B, T, dR))
    cache.append(0, c_new, kr_new)
    W_uk = rng.standard_normal((H, dn, r))
    W_uv = rng.standard_normal((H, dv, r))
    q_nope = rng.standard_normal((B, H, T, dn))
    q_rope = rng.standard_normal((B, H, T, dR))
    q_lat = np.einsum("bhtn,hnr->bhtr", q_nope, W_uk)
    o_lat = mla_cached_attention(cache, 0, q_lat, q_rope, scale)
    for b in range(B):
        n = lengths[b] + T
        c = np.concatenate([c_all[b, :lengths[b]], c_new[b]])
        kr = np.concatenate([kr_all[b, :lengths[b]], kr_new[b]])
        for h in range(H):
            k = np.concatenate([c @ W_uk[h].T, kr], axis=1)          # [n, dn + dR]
            v = c @ W_uv[h].T                                       # [n, dv]
            q = np.concatenate([q_nope[b, h], q_rope[b, h]], axis=1)
            want = attend(q * scale * np.sqrt(dn + dR), k, v, q_offset=lengths[b])   # attend scales by 1/sqrt(d)
            assert np.abs(o_lat[b, h] @ W_uv[h].T - want).max() < 1e-10
            assert n == k.shape[0]


def test_zero_rope_key_reduces_to_one_kv_head_attention():
    """k^R = 0 and scale 1/sqrt(r): every head attends over K = V = c, i.e. GQA with one K/V head."""
    rng = np.random.default_rng(4)
    B, H, r, T = 2, 3, 8, 2
    lat = OracleLatentCache(1, B, r, 4, 16, "f32")
    kv = OracleKVCache(1, B, 1, r, 16, "f32")
    c = rng.standard_normal((B, 9, r)).astype(np.float32)
    lat.append(0, c, np.zeros((B, 9, 4), np.float32))
    kv.append(0, c[:, None], c[:, None])
    for x in (lat, kv):
        x.commit()
        x.truncate([7, 3])
    c2 = rng.standard_normal((B, T, r)).astype(np.float32)
    lat.append(0, c2, np.zeros((B, T, 4), np.float32))
    kv.append(0, c2[:, None], c2[:, None])
    q = rng.standard_normal((B, H, T, r)).astype(np.float32)
    got = mla_cached_attention(lat, 0, q, rng.standard_normal((B, H, T, 4)).astype(np.float32), 1 / np.sqrt(r))
    assert np.abs(got - gqa_cached_attention(kv, 0, q)).max() < 1e-12


def test_cached_latent_equals_full_recompute_with_rope():
    """Keys k^R rotated once at their own positions and queries at theirs: every decode step equals a
    causal pass over the whole sequence."""
    rng = np.random.default_rng(5)
    H, r, dR, n = 2, 8, 4, 20
    c = rng.standard_normal((n, r))
    kr = apply_rope(rng.standard_normal((n, dR)), np.arange(n), 10000.0, "half")
    ql = rng.standard_normal((H, n, r))
    qr = apply_rope(rng.standard_normal((H, n, dR)), np.arange(n), 10000.0, "half")
    scale = 0.3
    cache = OracleLatentCache(1, 1, r, dR, n, "f64")
    s = 0
    for T in (6, 1, 1, 4, 8):
        cache.append(0, c[None, s:s + T], kr[None, s:s + T])
        out = mla_cached_attention(cache, 0, ql[None, :, s:s + T], qr[None, :, s:s + T], scale)[0]
        for h in range(H):
            scores = (ql[h, :s + T] @ c[:s + T].T + qr[h, :s + T] @ kr[:s + T].T) * scale
            scores = np.where(np.tril(np.ones((s + T, s + T), bool)), scores, -np.inf)
            e = np.exp(scores - scores.max(axis=1, keepdims=True))
            full = (e / e.sum(axis=1, keepdims=True)) @ c[:s + T]
            assert np.abs(out[h] - full[s:s + T]).max() < 1e-12
        cache.commit()
        s += T
