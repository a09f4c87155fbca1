"""GPU parity of the paged cache: the library's block pool and table against the paged oracle, and
paged attention against the contiguous cache on the same rows.

Bit-exact: both pools (never-written zeros and stale rows included), the block table, the free-block
count and the lengths. Within tolerance: attention outputs against the oracle. Bit-identical:
attention outputs of a paged and a contiguous cache holding the same rows ("KV cache, incremental
decode, ...", Key Takeaways: a float16 paged cache compares with the contiguous one exactly). The
kernels and their work plan are the same for both; only the tile addresses differ.
"""
import numpy as np
import pytest

from tests.gpu_parity import Mirror, check_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    yield


PAGED_CASES = [
    # dtype, d_h, H_q, H_kv, T, lengths, block   (kernel, pieces per tile)
    ("bf16", 128, 32, 8, 1, [0, 1, 15, 16, 17, 300, 1500], 16),   # tensor-core decode, 8 pieces
    ("f16", 128, 32, 8, 1, [127, 128, 129, 700], 128),            # tensor-core decode, 1 piece
    ("bf16", 128, 32, 8, 1, [255, 256, 257, 1000], 256),          # block longer than a tile
    ("f16", 64, 9, 3, 1, [2048, 5, 129], 32),                     # decode d_h = 64, 4 pieces
    ("f16", 128, 32, 8, 8, [2048, 333], 16),                      # verify chunk on the chunk kernel
    ("bf16", 128, 32, 8, 64, [5, 700], 64),                       # prefill chunk, 2 pieces
    ("f16", 128, 8, 8, 200, [0, 129], 16),                        # G = 1, diagonal masking, 8 pieces
    ("f32", 128, 8, 2, 1, [100, 33], 16),                         # CUDA-core split-K, 32-key tiles
    ("f32", 64, 6, 2, 3, [260, 1], 16),                           # 64-key tiles, 4 pieces
    ("f16", 32, 8, 2, 1, [600, 17], 16),                          # 256-key tiles (64-byte swizzle), 16 pieces
    ("bf16", 32, 4, 1, 17, [0, 100], 1024),                       # block longer than every tile
]


@pytest.mark.parametrize("dtype,d,Hq,Hkv,T,lengths,block", PAGED_CASES)
def test_paged_attention_matches_oracle(dtype, d, Hq, Hkv, T, lengths, block):
    B = len(lengths)
    max_len = max(lengths) + T + 8
    m = Mirror(L=2, B=B, H_kv=Hkv, d_h=d, max_len=max_len, dtype=dtype, seed=7 + T, block=block)
    s0 = max(lengths)
    if s0:
        for layer in range(2):
            m.append(layer, s0)
        m.commit()
        m.truncate(np.array(lengths))          # blocks past each length go back to the pool
        m.check_state()
    m.forward(T, Hq, what=f"paged block={block} {dtype} d={d} G={Hq // Hkv} T={T}")
    m.check_state()
    m.forward(1, Hq, what=f"paged block={block} {dtype} decode after")
    m.check_state()
    m.close()


def _pair(dtype, d, Hkv, max_len, block, seed, B):
    return (Mirror(L=1, B=B, H_kv=Hkv, d_h=d, max_len=max_len, dtype=dtype, seed=seed),
            Mirror(L=1, B=B, H_kv=Hkv, d_h=d, max_len=max_len, dtype=dtype, seed=seed, block=block))


@pytest.mark.parametrize("dtype,d,Hq,Hkv,T,block", [
    ("f16", 128, 32, 8, 1, 16), ("bf16", 128, 32, 8, 1, 64), ("f16", 128, 32, 8, 8, 16),
    ("bf16", 128, 16, 8, 100, 32), ("f16", 64, 8, 2, 1, 16), ("f32", 128, 8, 2, 2, 16),
    ("f16", 32, 8, 2, 1, 16)])
def test_paged_equals_contiguous_bit_for_bit(dtype, d, Hq, Hkv, T, block):
    """Same seeds, same calls: the two caches hold the same rows, so every kernel reads the same
    values into the same tile positions and the outputs agree bit for bit."""
    lengths = np.array([1999, 0, 512, 17, 1024, 77])
    cont, paged = _pair(dtype, d, Hkv, 2100, block, seed=21, B=len(lengths))
    for m in (cont, paged):
        m.append(0, int(lengths.max()))
        m.commit()
        m.truncate(lengths)
        m.append(0, T)
    for split in (0, 256):
        outs = []
        for m in (cont, paged):
            m.n_draws = 100 + split                 # same query draw on both sides
            got, want = m.attend(0, Hq, T, split_keys=split)
            check_outputs(got, want, dtype, f"split {split}")
            outs.append(got)
        assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32)), f"split {split}"
    cont.close()
    paged.close()


def test_interleaved_blocks_after_reuse():
    """Sequences that end free blocks which others grow into, so each sequence's blocks are scattered
    and out of order in the pool; reads stay those of the oracle."""
    m = Mirror(L=2, B=4, H_kv=2, d_h=128, max_len=600, dtype="bf16", seed=4, block=16, n_blocks=80)
    for _ in range(3):
        m.forward(40, 8, what="grow")           # 120 rows each: 8 blocks each, 32 in all
    m.truncate([0, 120, 3, 120])                # sequences 0 and 2 end (2 keeps one block)
    m.check_state()
    for i in range(5):
        m.forward(33 if i % 2 else 1, 8, what=f"regrow {i}")
        m.check_state()
    table = np.array(m.kb.kvc_block_table(m.gpu)[0])
    held = table[1][table[1] >= 0]
    assert np.any(np.diff(held) < 0), "sequence 1's blocks should be out of order by now"
    m.close()


def test_pool_exhaustion_returns_capacity_and_changes_nothing():
    from kv_cached_gqa_gb300 import _binding as kb
    m = Mirror(L=2, B=2, H_kv=2, d_h=128, max_len=512, dtype="f16", seed=9, block=32, n_blocks=10)
    m.forward(100, 8, what="fill")              # 4 blocks each: 8 of 10
    m.check_state()
    T = 70                                      # 170 rows need 6 blocks each: 4 more > 2 free
    k = m.torch.zeros((2, 2, T, 128), dtype=m.torch.float32, device="cuda")
    with pytest.raises(kb.KvcError) as e:
        kb.kvc_append(m.gpu, 0, k, k)
    assert e.value.code == -2 and "block pool" in str(e.value)
    m.check_state()                             # table, pool, lengths untouched
    m.forward(20, 8, what="still usable")       # 120 rows: 4 blocks each, nothing new
    m.check_state()
    m.close()


def test_paged_noalloc_matches_oracle():
    from kv_cached_gqa_gb300 import _binding as kb
    m = Mirror(L=1, B=3, H_kv=8, d_h=128, max_len=1200, dtype="bf16", seed=12, block=16)
    m.append(0, 1100)
    m.commit()
    m.truncate(np.array([1099, 3, 640]))
    m.append(0, 1)
    q = m.draw((3, 32, 1, 128))
    from oracle.kvc_oracle import gqa_cached_attention
    want = gqa_cached_attention(m.ref, 0, q)
    out = m.torch.empty((3, 32, 1, 128), dtype=m.torch.float32, device="cuda")
    for _ in range(2):
        got = kb.gqa_cached_attn_noalloc(m.gpu, m.dev(q), 0, out).cpu().numpy()
        check_outputs(got, want, "bf16", "paged no-alloc")
    m.close()
