"""GPU parity of fused rotary positions: kvc_append_rope and gqa_cached_attn_rope against the oracle.

"KV cache decoding", "Position information with a cache": keys are stored already rotated by their
absolute positions and each new query is rotated by its own, so cached keys never change. The oracle
rotates in float64 (RoFormer's formula); the kernels rotate in float32 from a float64-built cos/sin
table. Stored keys are compared within one unit in the last place of the cache dtype (see
check_rotated_store), values bit-exactly, outputs within the usual tolerance.
"""
import numpy as np
import pytest

from tests.gpu_parity import Mirror, check_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    yield


ROPE_CASES = [
    # dtype, d_h, H_q, H_kv, T, lengths, base, style, block
    ("bf16", 128, 32, 8, 1, [0, 1, 500, 1500], 500000.0, "half", None),      # decode, tensor cores
    ("f16", 128, 32, 8, 8, [2048, 333], 10000.0, "half", None),              # verify chunk
    ("bf16", 128, 16, 8, 100, [0, 129], 10000.0, "interleaved", None),       # prefill chunk
    ("f16", 64, 9, 3, 1, [2048, 5, 129], 10000.0, "half", None),             # d_h = 64
    ("f32", 128, 8, 2, 1, [100, 33], 10000.0, "half", None),                 # CUDA-core split-K
    ("f32", 32, 4, 2, 17, [0, 40], 10000.0, "interleaved", None),            # d_h = 32, chunk
    ("f16", 32, 8, 2, 3, [600, 17], 500000.0, "half", None),
    ("bf16", 128, 32, 8, 1, [0, 17, 300, 1500], 500000.0, "half", 16),       # paged
    ("f16", 128, 16, 4, 40, [5, 700], 10000.0, "interleaved", 64),           # paged chunk
]


@pytest.mark.parametrize("dtype,d,Hq,Hkv,T,lengths,base,style,block", ROPE_CASES)
def test_rope_attention_matches_oracle(dtype, d, Hq, Hkv, T, lengths, base, style, block):
    B = len(lengths)
    max_len = max(lengths) + 2 * T + 8
    m = Mirror(L=2, B=B, H_kv=Hkv, d_h=d, max_len=max_len, dtype=dtype, seed=31 + T, block=block,
               rope=(base, style))
    s0 = max(lengths)
    if s0:
        for layer in range(2):
            m.append(layer, s0)              # keys rotated at positions 0 .. s0-1
        m.commit()
        m.truncate(np.array(lengths))
        m.check_state()
    for step in range(2):
        m.forward(T, Hq, what=f"rope {style} base={base:g} {dtype} d={d} T={T} step {step}")
        m.check_state()
    m.close()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rope_with_inputs_in_the_cache_dtype(dtype):
    """Keys and queries handed over in the cache dtype are widened, rotated and rounded again."""
    m = Mirror(L=1, B=2, H_kv=8, d_h=128, max_len=600, dtype=dtype, seed=5, rope=(10000.0, "half"))
    m.append(0, 500, in_dtype=dtype)
    m.commit()
    m.truncate(np.array([499, 77]))
    m.append(0, 1, in_dtype=dtype)
    got, want = m.attend(0, 32, 1, q_in=dtype)
    check_outputs(got, want, dtype, "rope, 16-bit inputs")
    m.check_state()
    m.close()


def test_rope_near_the_end_of_the_table():
    """Positions up to max_len - 1 read the last rows of the cos/sin table."""
    m = Mirror(L=1, B=2, H_kv=2, d_h=64, max_len=130, dtype="bf16", seed=8, rope=(10000.0, "half"))
    m.append(0, 129)
    m.commit()
    m.truncate(np.array([129, 60]))
    m.forward(1, 8, what="last position")
    m.check_state()
    m.close()


def test_rope_calls_need_a_table():
    from kv_cached_gqa_gb300 import _binding as kb
    import torch
    c = kb.Cache(1, 1, 2, 64, 16, kb.KVC_BF16)
    k = torch.zeros((1, 2, 1, 64), device="cuda")
    with pytest.raises(kb.KvcError) as e:
        kb.kvc_append_rope(c, 0, k, k)
    assert e.value.code == -3 and "kvc_set_rope" in str(e.value)
    with pytest.raises(kb.KvcError):
        kb.kvc_set_rope(c, 1.0)
    kb.kvc_set_rope(c, 10000.0)
    kb.kvc_append_rope(c, 0, k, k)
    out = kb.gqa_cached_attn_rope(c, torch.zeros((1, 4, 1, 64), device="cuda"), 0)
    assert torch.all(out == 0)
    c.close()
