"""Pins of the paged oracle, OraclePagedKVCache, to things other than itself.

* "KV cache, incremental decode, ...", Key Takeaways and §2.5: a float16 paged cache hands back what
  the contiguous cache hands back and compares with it exactly. The contiguous oracle is pinned on its
  own (test_oracle_pins.py), so equality with it under random ragged traffic pins the paged one's
  addressing, rounding and reads.
* "KV cache decoding", "Batching caches of different lengths": a sequence takes a new block only when
  it grows into it and frees its blocks when it ends. Block counts follow from that in closed form,
  and small tables are worked out by hand below.
* "Generation and the KV Cache", "Static versus growing": the reserved positions of a preallocated
  cache are what paging recovers.
"""
import numpy as np
import pytest

from oracle.kvc_oracle import (OracleKVCache, OraclePagedKVCache, gqa_cached_attention)


def _chunk(rng, B, H, T, d):
    return (rng.standard_normal((B, H, T, d)).astype(np.float32),
            rng.standard_normal((B, H, T, d)).astype(np.float32))


def test_paged_hand_example():
    """Rows [[1, 2], [3, 4]] then [5, 6] with blocks of 2: block 0 holds the first two rows, block 1
    holds the third in its row 0; the table is [0, 1, -1, -1]."""
    c = OraclePagedKVCache(1, 1, 1, 2, 8, block=2, n_blocks=4, dtype="f32")
    k1 = np.array([[[[1, 2], [3, 4]]]], np.float32)
    rows = c.append(0, k1, k1)
    c.commit()
    assert c.table.tolist() == [[0, -1, -1, -1]]
    k2 = np.array([[[[5, 6]]]], np.float32)
    rows = c.append(0, k2, k2)
    c.commit()
    assert c.table.tolist() == [[0, 1, -1, -1]]
    assert c.k[0, 0, 0].tolist() == [[1, 2], [3, 4]]
    assert c.k[0, 1, 0].tolist() == [[5, 6], [0, 0]]
    assert rows[0][0][0].tolist() == [[1, 2], [3, 4], [5, 6]]
    assert c.seq_len().tolist() == [3]
    assert sorted(c.free) == [2, 3]
    assert c.nbytes() == 2 * 1 * 4 * 1 * 2 * 2 * 4


def test_paged_allocation_order_by_hand():
    """Lowest free block first, sequences in order, then logical blocks in order."""
    c = OraclePagedKVCache(1, 2, 1, 1, 6, block=2, n_blocks=6, dtype="f32")
    z = np.zeros((2, 1, 3, 1), np.float32)
    c.append(0, z, z)                       # 3 rows each: 2 blocks each
    c.commit()
    assert c.table.tolist() == [[0, 1, -1], [2, 3, -1]]
    c.truncate([1, 3])                      # sequence 0 keeps only block 0
    assert c.table.tolist() == [[0, -1, -1], [2, 3, -1]]
    assert sorted(c.free) == [1, 4, 5]
    z2 = np.zeros((2, 1, 2, 1), np.float32)
    c.append(0, z2, z2)                     # fills 3 and 5: sequence 0 takes 1, sequence 1 takes 4
    assert c.table.tolist() == [[0, 1, -1], [2, 3, 4]]
    c.commit()
    c.truncate([0, 0])                      # both end: every block is free again
    assert c.table.tolist() == [[-1, -1, -1], [-1, -1, -1]]
    assert sorted(c.free) == list(range(6))


def _random_traffic(dtype, seed, block, L=2, B=3, H=2, G=2, d=4, max_len=40, steps=14):
    """Identical random forwards and ragged truncates on a contiguous and a paged oracle; yields both
    after every operation."""
    rng = np.random.default_rng(seed)
    n_blocks = B * (-(-max_len // block))
    ref = OracleKVCache(L, B, H, d, max_len, dtype)
    pag = OraclePagedKVCache(L, B, H, d, max_len, block, n_blocks, dtype)
    for _ in range(steps):
        if rng.random() < 0.7:
            T = int(rng.integers(1, 7))
            if int(ref.lens.max()) + T > max_len:
                continue
            q = rng.standard_normal((B, H * G, T, d)).astype(np.float32)
            for layer in range(L):
                k, v = _chunk(rng, B, H, T, d)
                r1 = ref.append(layer, k, v)
                r2 = pag.append(layer, k, v)
                for (ka, va), (kb, vb) in zip(r1, r2):
                    assert np.array_equal(ka, kb) and np.array_equal(va, vb)
                o1 = gqa_cached_attention(ref, layer, q)
                o2 = gqa_cached_attention(pag, layer, q)
                assert np.array_equal(o1, o2)
            ref.commit()
            pag.commit()
        else:
            n = [int(rng.integers(0, int(s) + 1)) for s in ref.lens]
            ref.truncate(n)
            pag.truncate(n)
        yield ref, pag


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("block", [1, 4, 16])
def test_paged_equals_contiguous_bit_for_bit(dtype, block):
    for ref, pag in _random_traffic(dtype, seed=11 + block, block=block):
        assert np.array_equal(ref.fill, pag.fill) and np.array_equal(ref.lens, pag.lens)
        for layer in range(ref.L):
            for b in range(ref.B):
                n = int(ref.fill[layer, b])
                for h in range(ref.H):
                    ka, va = ref.stored_f64(layer, b, h, n)
                    kb, vb = pag.stored_f64(layer, b, h, n)
                    assert np.array_equal(ka, kb) and np.array_equal(va, vb)


@pytest.mark.parametrize("block", [1, 4, 16])
def test_paged_holds_exactly_the_blocks_its_rows_reach(block):
    """Each sequence holds ceil(s_b / block) blocks, mapped at logical 0 .. held-1, all distinct; the
    rest of the pool is free."""
    for ref, pag in _random_traffic("f16", seed=3 + block, block=block):
        mapped = []
        for b in range(pag.B):
            held = pag.held(b)
            assert held == -(-int(pag.lens[b]) // block)
            assert np.all(pag.table[b, :held] >= 0) and np.all(pag.table[b, held:] == -1)
            mapped += pag.table[b, :held].tolist()
        assert len(set(mapped)) == len(mapped)
        assert set(mapped) | pag.free == set(range(pag.n_blocks))
        assert not (set(mapped) & pag.free)


def test_paging_recovers_reserved_positions():
    """A 20-position answer in a 128-position cache: the contiguous cache reserves all 128, the paged
    one holds ceil(20 / 16) = 2 blocks of 16."""
    ref = OracleKVCache(1, 1, 1, 8, 128, "f32")
    pag = OraclePagedKVCache(1, 1, 1, 8, 128, block=16, n_blocks=8, dtype="f32")
    k = np.ones((1, 1, 20, 8), np.float32)
    ref.append(0, k, k)
    pag.append(0, k, k)
    assert ref.nbytes() == 2 * 128 * 8 * 4
    assert pag.held(0) * 16 == 32
    assert len(pag.free) == 6


def test_pool_exhaustion_changes_nothing():
    c = OraclePagedKVCache(2, 2, 1, 2, 32, block=4, n_blocks=5, dtype="f16")
    k = np.ones((2, 1, 8, 2), np.float32)
    c.append(0, k, k)                       # 2 + 2 blocks
    snapshot = (c.table.copy(), set(c.free), c.fill.copy(), c.k.copy())
    with pytest.raises(OverflowError):
        c.append(0, np.ones((2, 1, 4, 2), np.float32), np.ones((2, 1, 4, 2), np.float32))
    assert np.array_equal(c.table, snapshot[0]) and c.free == snapshot[1]
    assert np.array_equal(c.fill, snapshot[2]) and np.array_equal(c.k, snapshot[3])
    c.append(1, k, k)                       # layer 1 reuses the blocks layer 0 mapped
    assert len(c.free) == 1
    with pytest.raises(OverflowError):
        c.append(0, np.ones((2, 1, 30, 2), np.float32), np.ones((2, 1, 30, 2), np.float32))


def test_a_finished_sequence_frees_blocks_for_another():
    """Sequence 0 ends (truncate to 0); both then grow into the freed blocks, lowest first; reads stay
    those of the contiguous cache."""
    rng = np.random.default_rng(5)
    ref = OracleKVCache(1, 2, 1, 4, 24, "bf16")
    pag = OraclePagedKVCache(1, 2, 1, 4, 24, block=4, n_blocks=7, dtype="bf16")
    k, v = _chunk(rng, 2, 1, 12, 4)
    for c in (ref, pag):
        c.append(0, k, v)
        c.commit()
    assert pag.table.tolist() == [[0, 1, 2, -1, -1, -1], [3, 4, 5, -1, -1, -1]]
    for c in (ref, pag):
        c.truncate([0, 12])
    assert sorted(pag.free) == [0, 1, 2, 6]
    k, v = _chunk(rng, 2, 1, 4, 4)
    for c in (ref, pag):
        c.append(0, k, v)
        c.commit()
    q = rng.standard_normal((2, 1, 1, 4)).astype(np.float32)
    kk, vv = _chunk(rng, 2, 1, 1, 4)
    for c in (ref, pag):
        c.append(0, kk, vv)
    assert pag.table.tolist() == [[0, 2, -1, -1, -1, -1], [3, 4, 5, 1, 6, -1]]
    assert len(pag.free) == 0
    assert np.array_equal(gqa_cached_attention(ref, 0, q), gqa_cached_attention(pag, 0, q))
