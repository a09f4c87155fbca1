"""GPU parity of gqa_cached_attn_append: one call that stores a layer's chunk and attends over it.

The call must equal kvc_append followed by gqa_cached_attn ("KV cache, incremental decode, ...", §2.3:
the chunk's keys and values go to positions [s, s + T), then its queries attend with
causal_mask(T, s + T, q_offset = s)). Checked three ways:
- against the oracle: stored rows bit-exact (rotated keys within the RoPE bound), outputs within the
  dtype's tolerance, lengths and positions exact;
- against the two separate calls on a second cache fed the same draws: outputs and stores
  bit-identical, since the stored rows are rounded the same way and attention reads what is stored;
- its launch count: one launch on the tensor-core decode kernel, which stores the rows itself, two
  (append, attention) on every other kernel.
"""
import numpy as np
import pytest

from tests.gpu_parity import Mirror, check_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    yield


CASES = [
    # dtype, d_h, H_q, H_kv, T, lengths, block, rope, fp8 scales, launches per call
    ("bf16", 128, 32, 8, 1, [0, 1, 127, 128, 129, 700, 2300], None, None, None, 1),
    ("f16", 64, 9, 3, 1, [2048, 5, 129], None, None, None, 1),
    ("bf16", 128, 16, 4, 4, [126, 0, 255, 300], None, None, None, 1),      # new rows straddle a tile edge
    ("f16", 128, 32, 8, 1, [15, 16, 17, 900], 16, None, None, 1),           # paged, 16-position blocks
    ("bf16", 128, 32, 8, 2, [127, 1, 1000], None, (10000.0, "half"), None, 1),
    ("f16", 64, 9, 3, 1, [300, 2], None, (500000.0, "interleaved"), None, 1),
    ("e4m3", 128, 32, 8, 1, [0, 129, 1200], None, None, ([0.5, 2.0], [1.5, 0.25]), 1),
    ("f32", 128, 8, 2, 1, [100, 33], None, None, None, 2),                  # CUDA-core split-K kernel
    ("f16", 128, 32, 8, 8, [2048, 333], None, None, None, 2),               # verify chunk: chunk kernel
    ("bf16", 128, 8, 8, 200, [0, 129], None, None, None, 2),                # prefill chunk
]


def _mirror(dtype, d, Hkv, lengths, T, block, rope, scales, seed):
    B = len(lengths)
    max_len = max(lengths) + 2 * T + 8
    return Mirror(L=2, B=B, H_kv=Hkv, d_h=d, max_len=max_len, dtype=dtype, seed=seed, block=block,
                  rope=rope, scales=scales)


def _prefill(m, lengths):
    s0 = max(lengths)
    if s0:
        for layer in range(m.L):
            m.append(layer, s0)
        m.commit()
        m.truncate(np.array(lengths))


@pytest.mark.parametrize("dtype,d,Hq,Hkv,T,lengths,block,rope,scales,launches", CASES)
def test_fused_step_matches_oracle_and_separate_calls(dtype, d, Hq, Hkv, T, lengths, block, rope, scales, launches):
    fused = _mirror(dtype, d, Hkv, lengths, T, block, rope, scales, seed=11 + T)
    sep = _mirror(dtype, d, Hkv, lengths, T, block, rope, scales, seed=11 + T)
    _prefill(fused, lengths)
    _prefill(sep, lengths)
    what = f"fused {dtype} d={d} G={Hq // Hkv} T={T} block={block} rope={rope is not None}"
    for step in range(2):                              # two forwards: the second appends after a commit
        for layer in range(fused.L):
            before = fused.kb.kvc_launch_count(fused.gpu)
            got, want = fused.append_attend(layer, T, Hq)
            n = fused.kb.kvc_launch_count(fused.gpu) - before
            # a paged cache may also launch one block-table edit when a sequence reaches a new block
            assert launches <= n <= launches + (block is not None), (n, launches)
            check_outputs(got, want, dtype, f"{what} step {step} layer {layer}")
            sep.append(layer, T)
            got_sep, _ = sep.attend(layer, Hq, T)
            assert np.array_equal(got, got_sep), f"{what}: fused and separate outputs differ"
        fused.commit()
        sep.commit()
        fused.check_state()
        (fk, fv), _ = fused.store_bits()
        (sk, sv), _ = sep.store_bits()
        np.testing.assert_array_equal(fk, sk)
        np.testing.assert_array_equal(fv, sv)
    fused.close()
    sep.close()


@pytest.mark.parametrize("split", [128, 256, 384])
def test_fused_step_with_forced_splits(split):
    """Many splits per sequence: only the split that holds a new row stores it; the others read rows
    that were already there."""
    lengths = [1000, 257, 128, 3]
    m = _mirror("bf16", 128, 8, lengths, 1, None, None, None, seed=5)
    _prefill(m, lengths)
    for layer in range(m.L):
        got, want = m.append_attend(layer, 1, 32, split_keys=split)
        check_outputs(got, want, "bf16", f"split={split} layer {layer}")
    m.commit()
    m.check_state()
    m.close()


def test_fused_call_errors_change_nothing():
    from kv_cached_gqa_gb300._binding import KvcError
    lengths = [10, 3]
    m = _mirror("f16", 128, 2, lengths, 1, None, None, None, seed=3)
    _prefill(m, lengths)
    m.append(0, 1)                                     # layer 0 already holds this step's row
    (k0, v0), _ = m.store_bits()
    lens0 = [m.kb.kvc_seq_len(m.gpu, l) for l in (-1, 0, 1)]
    k = m.dev(np.zeros((2, 2, 1, 128), np.float32))
    q = m.dev(np.zeros((2, 8, 1, 128), np.float32))
    with pytest.raises(KvcError) as e:
        m.kb.gqa_cached_attn_append(m.gpu, 0, k, k, q)
    assert e.value.code == -3                          # KVC_E_STATE
    with pytest.raises(KvcError) as e:                 # H_q not a multiple of H_kv
        m.kb.gqa_cached_attn_append(m.gpu, 1, k, k, m.dev(np.zeros((2, 3, 1, 128), np.float32)))
    assert e.value.code == -1                          # KVC_E_INVAL
    m.kb.kvc_status(m.gpu)
    (k1, v1), _ = m.store_bits()
    np.testing.assert_array_equal(k0, k1)
    np.testing.assert_array_equal(v0, v1)
    assert [m.kb.kvc_seq_len(m.gpu, l) for l in (-1, 0, 1)] == lens0
    m.close()


def test_fused_call_rejects_a_chunk_past_max_len():
    from kv_cached_gqa_gb300._binding import KvcError
    m = Mirror(L=1, B=2, H_kv=2, d_h=128, max_len=20, dtype="bf16", seed=4)
    m.append(0, 19)
    m.commit()
    (k0, v0), _ = m.store_bits()
    k = m.dev(np.zeros((2, 2, 2, 128), np.float32))
    q = m.dev(np.zeros((2, 8, 2, 128), np.float32))
    with pytest.raises(KvcError) as e:
        m.kb.gqa_cached_attn_append(m.gpu, 0, k, k, q)
    assert e.value.code == -2                          # KVC_E_CAPACITY
    (k1, v1), _ = m.store_bits()
    np.testing.assert_array_equal(k0, k1)
    np.testing.assert_array_equal(v0, v1)
    assert m.kb.kvc_seq_len(m.gpu, 0) == [19, 19]
    m.close()
