"""The allocation-free attention entry point against the regular one.

gqa_cached_attn_noalloc serves callers that cannot let the library allocate device memory (a
serving process that reserves its memory up front, memory owned by another framework's pool, a
latency-critical path): its scratch is a fixed device array inside the library. This file runs last
(pytest collects it last) and also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import kvc_synth
from tests.gpu_parity import check_outputs

pytestmark = pytest.mark.gpu


def _prefilled(kb, torch, dtype, L, B, H_kv, d, lengths, T, seed):
    cache = kb.Cache(L, B, H_kv, d, max(lengths) + T + 4, dtype)
    s0 = max(lengths)
    for layer in range(L):
        k = torch.from_numpy(kvc_synth.normal_f32((B, H_kv, s0, d), seed, 10 + layer)).cuda()
        v = torch.from_numpy(kvc_synth.normal_f32((B, H_kv, s0, d), seed, 20 + layer)).cuda()
        kb.kvc_append(cache, layer, k, v)
    kb.kvc_commit(cache)
    kb.kvc_truncate_ragged(cache, lengths)
    for layer in range(L):
        k = torch.from_numpy(kvc_synth.normal_f32((B, H_kv, T, d), seed, 30 + layer)).cuda()
        v = torch.from_numpy(kvc_synth.normal_f32((B, H_kv, T, d), seed, 40 + layer)).cuda()
        kb.kvc_append(cache, layer, k, v)
    return cache


@pytest.mark.parametrize("dtype,name,d,H_q,H_kv,T,lengths", [
    (2, "bf16", 128, 32, 8, 1, [4019, 544, 2300, 1, 0, 3000, 1500, 777]),   # tensor-core kernel, splits
    (1, "f16", 128, 32, 8, 8, [2048, 300]),                                  # tensor-core, verify chunk
    (0, "f32", 32, 4, 2, 1, [47, 1000]),                                     # CUDA-core kernel
])
def test_noalloc_matches_regular_entry_point_twice(gpu_lib, dtype, name, d, H_q, H_kv, T, lengths):
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    B = len(lengths)
    cache = _prefilled(kb, torch, dtype, 2, B, H_kv, d, lengths, T, seed=7)
    for layer in range(2):
        q = torch.from_numpy(kvc_synth.normal_f32((B, H_q, T, d), 7, 50 + layer)).cuda()
        ref = kb.gqa_cached_attn(cache, q, layer).cpu().numpy()
        for _ in range(2):                                   # two calls in a row share the array
            out = torch.full((B, H_q, T, d), float("nan"), dtype=torch.float32, device="cuda")
            kb.gqa_cached_attn_noalloc(cache, q, layer, out)
            check_outputs(out.cpu().numpy(), ref, name, f"noalloc layer {layer}")
    kb.kvc_status(cache)
    cache.close()


def test_noalloc_rejects_plans_beyond_the_fixed_array(gpu_lib):
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    B, H_kv, H_q, d = 64, 8, 32, 128                         # 64 sequences of 4096 keys: ~12 MB of partials
    cache = kb.Cache(1, B, H_kv, d, 4200, 2)
    k = torch.zeros((B, H_kv, 4096, d), dtype=torch.bfloat16, device="cuda")
    kb.kvc_append(cache, 0, k, k)
    kb.kvc_commit(cache)
    kb.kvc_append(cache, 0, k[:, :, :1].contiguous(), k[:, :, :1].contiguous())
    q = torch.zeros((B, H_q, 1, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((B, H_q, 1, d), dtype=torch.float32, device="cuda")
    with pytest.raises(kb.KvcError) as ei:
        kb.gqa_cached_attn_noalloc(cache, q, 0, out)
    assert ei.value.code == -6 and "fixed array holds" in str(ei.value)
    kb.gqa_cached_attn(cache, q, 0, out=out)                 # the regular entry point still serves it
    kb.kvc_status(cache)
    cache.close()
