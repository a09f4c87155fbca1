"""GPU parity of the fp8 (E4M3) cache: stored codes bit-exact against the oracle, attention within
tolerance.

The pages name cache quantisation as a decode lever without a format ("KV cache decoding", "What is
cached, what is not, and what it costs"); the reading is E4M3 codes of x / scale with one scale per layer
for K and one for V, read back as code * scale, and queries used in float16.
"""
import numpy as np
import pytest

from tests.gpu_parity import Mirror

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    yield


@pytest.mark.parametrize("in_dtype", ["f32", "f16", "bf16"])
def test_fp8_append_commit_truncate_bit_exact(in_dtype):
    # scales that are not powers of two, so the float32 division rounds
    m = Mirror(L=3, B=3, H_kv=2, d_h=64, max_len=40, dtype="e4m3", scales=([0.37, 1.0, 3.1], [0.05, 2.5, 1.0]))
    for layer in range(3):
        m.append(layer, 7, in_dtype=in_dtype)
    m.check_state()
    m.commit()
    m.truncate([2, 7, 0])
    for T in (1, 5):
        for layer in range(3):
            m.append(layer, T, in_dtype=in_dtype)
        m.commit()
        m.check_state()
    m.close()


def test_fp8_saturates_and_keeps_subnormals():
    """Scales that push rows past +-448 (saturated) and down into the subnormal codes."""
    m = Mirror(L=2, B=2, H_kv=2, d_h=128, max_len=16, dtype="e4m3", scales=([1e-3, 1e3], [5e-3, 2e2]))
    for layer in range(2):
        m.append(layer, 9)
    m.check_state()
    codes = m.gpu.k.view(m.torch.uint8).cpu().numpy()
    assert np.any((codes[0] & 0x7F) == 0x7E)          # saturated at 448
    assert np.any(((codes[1] & 0x78) == 0) & ((codes[1] & 7) != 0))   # subnormal codes
    m.close()


FP8_CASES = [
    # d_h, H_q, H_kv, T, lengths, block
    (128, 32, 8, 1, [0, 1, 63, 64, 65, 700, 1500], None),
    (64, 9, 3, 1, [2048, 5, 129], None),
    (128, 16, 2, 1, [513, 31], None),                  # G = 8
    (128, 32, 8, 3, [777, 64], None),
    (128, 32, 8, 8, [2048, 333], None),                # verify chunk
    (64, 8, 8, 17, [130, 0, 3], None),
    (128, 32, 8, 1, [0, 17, 300, 1500], 16),           # paged
    (64, 8, 2, 5, [600, 17], 64),
]


@pytest.mark.parametrize("d,Hq,Hkv,T,lengths,block", FP8_CASES)
def test_fp8_attention_matches_oracle(d, Hq, Hkv, T, lengths, block):
    B = len(lengths)
    max_len = max(lengths) + 2 * T + 8
    m = Mirror(L=2, B=B, H_kv=Hkv, d_h=d, max_len=max_len, dtype="e4m3", seed=41 + T, block=block,
               scales=([0.25, 0.7], [0.5, 0.03]))
    s0 = max(lengths)
    if s0:
        for layer in range(2):
            m.append(layer, s0)
        m.commit()
        m.truncate(np.array(lengths))
    for step in range(2):
        m.forward(T, Hq, what=f"fp8 d={d} G={Hq // Hkv} T={T} block={block} step {step}")
        m.check_state()
    m.close()


def test_fp8_query_in_float16_and_rope():
    m = Mirror(L=1, B=2, H_kv=8, d_h=128, max_len=600, dtype="e4m3", seed=3, rope=(500000.0, "half"),
               scales=([0.5], [0.5]))
    m.append(0, 500, in_dtype="bf16")
    m.commit()
    m.truncate(np.array([499, 77]))
    m.append(0, 1)
    got, want = m.attend(0, 32, 1, q_in="f16")
    from tests.gpu_parity import check_outputs
    check_outputs(got, want, "e4m3", "fp8 with RoPE, float16 query")
    m.check_state()
    m.close()


def test_fp8_scales_rules():
    from kv_cached_gqa_gb300 import _binding as kb
    import torch
    c = kb.Cache(2, 1, 2, 64, 16, kb.KVC_FP8_E4M3)
    with pytest.raises(kb.KvcError):
        kb.kvc_set_kv_scales(c, [1.0, -1.0], [1.0, 1.0])
    kb.kvc_set_kv_scales(c, [2.0, 2.0], [1.0, 1.0])
    k = torch.ones((1, 2, 1, 64), device="cuda")
    kb.kvc_append(c, 0, k, k)
    with pytest.raises(kb.KvcError) as e:
        kb.kvc_set_kv_scales(c, 1.0, 1.0)
    assert e.value.code == -3
    with pytest.raises(kb.KvcError):                   # a bfloat16 query is not the fp8 cache's query type
        kb.gqa_cached_attn(c, torch.ones((1, 4, 1, 64), device="cuda", dtype=torch.bfloat16), 0)
    c.close()
    f = kb.Cache(1, 1, 1, 64, 16, kb.KVC_BF16)
    with pytest.raises(kb.KvcError):
        kb.kvc_set_kv_scales(f, 1.0, 1.0)
    f.close()
    with pytest.raises(kb.KvcError) as e:
        kb.Cache(1, 1, 1, 32, 16, kb.KVC_FP8_E4M3)     # 32-byte fp8 rows
    assert e.value.code == -6
