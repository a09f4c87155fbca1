"""GPU parity of the latent (MLA) cache and of multi-head latent attention against the oracle.

"KV cache, incremental decode, ...", §2.6 "The latent cache": one latent c in R^r and one shared RoPE key
k^R in R^{d_R} per position, the KV cache's rules, nbytes = L B N_max (r + d_R) itemsize. The attention
that reads it is DeepSeek-V2's MLA in absorbed form. Bit-exact: both stores, lengths, positions.
Within tolerance: the attended latents.
"""
import numpy as np
import pytest

from tests.gpu_parity import LatentMirror

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    yield


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_latent_append_commit_truncate_bit_exact(dtype):
    m = LatentMirror(L=3, B=3, r=64, d_rope=16, max_len=40, dtype=dtype)
    for layer in range(3):
        m.append(layer, 7)
    m.check_state()
    m.commit()
    m.truncate([2, 7, 0])
    m.check_state()
    for T in (1, 5):
        for layer in range(3):
            m.append(layer, T, in_dtype="f32" if T == 1 else dtype)
        m.commit()
        m.check_state()
    assert m.kb.kvc_nbytes(m.gpu) == 3 * 3 * 40 * (64 + 16) * {"f32": 4, "f16": 2, "bf16": 2}[dtype]
    m.close()


MLA_CASES = [
    # dtype, r, d_R, H, T, lengths
    # r in {256, 512} with d_R = 64 and a 16-bit cache run on tensor cores, the rest on CUDA cores
    ("bf16", 512, 64, 16, 1, [0, 1, 31, 32, 33, 700, 1500]),     # DeepSeek-V2-Lite-shaped decode
    ("bf16", 512, 64, 128, 1, [300, 5]),                         # 128 heads: 8 row tiles per sequence
    ("f16", 512, 64, 16, 4, [129, 0, 64]),                       # a chunk: diagonal masking
    ("f32", 128, 32, 8, 3, [100, 33]),
    ("bf16", 64, 16, 4, 17, [0, 40]),
    ("f16", 256, 32, 32, 1, [2000, 17, 999]),                    # several key splits per sequence
    ("bf16", 256, 64, 8, 2, [100, 1000, 7, 3000]),               # tensor cores, r = 256
    ("f16", 512, 64, 32, 1, [4000, 1, 2500]),                    # tensor cores, many splits and a merge
]


@pytest.mark.parametrize("dtype,r,dR,H,T,lengths", MLA_CASES)
def test_mla_matches_oracle(dtype, r, dR, H, T, lengths):
    B = len(lengths)
    m = LatentMirror(L=2, B=B, r=r, d_rope=dR, max_len=max(lengths) + 2 * T + 8, dtype=dtype, seed=T + H)
    scale = 1.0 / np.sqrt(128 + dR)
    s0 = max(lengths)
    if s0:
        for layer in range(2):
            m.append(layer, s0)
        m.commit()
        m.truncate(np.array(lengths))
    for step in range(2):
        m.forward(T, H, scale, what=f"mla {dtype} r={r} d_R={dR} H={H} T={T} step {step}")
        m.check_state()
    m.close()


def test_mla_queries_in_the_cache_dtype():
    m = LatentMirror(L=1, B=2, r=512, d_rope=64, max_len=300, dtype="bf16", seed=2)
    m.append(0, 250, in_dtype="bf16")
    m.commit()
    m.truncate(np.array([249, 3]))
    m.append(0, 1)
    got, want = m.attend(0, 16, 1, 0.07, q_in="bf16")
    from tests.gpu_parity import check_outputs
    check_outputs(got, want, "bf16", "mla, bf16 queries")
    m.close()


def test_latent_cache_rejects_kv_calls():
    from kv_cached_gqa_gb300 import _binding as kb
    import torch
    c = kb.LatentCache(1, 1, 64, 16, 16, kb.KVC_BF16)
    kb.kvc_append(c, 0, torch.zeros((1, 1, 64), device="cuda"), torch.zeros((1, 1, 16), device="cuda"))
    with pytest.raises(kb.KvcError) as e:
        kb.gqa_cached_attn(c, torch.zeros((1, 4, 1, 64), device="cuda"), 0)
    assert e.value.code == -1
    with pytest.raises(kb.KvcError) as e:
        kb.kvc_set_rope(c, 10000.0)
    assert e.value.code == -6
    with pytest.raises(kb.KvcError):
        kb.mla_cached_attn(c, torch.zeros((1, 4, 1, 64), device="cuda"), torch.zeros((1, 4, 1, 16), device="cuda"),
                           0, -1.0)
    out = kb.mla_cached_attn(c, torch.zeros((1, 4, 1, 64), device="cuda"), torch.zeros((1, 4, 1, 16), device="cuda"),
                             0, 0.1)
    assert torch.all(out == 0)
    c.close()
