"""The allocation-free attention entry point, against the oracle and against the regular one.

gqa_cached_attn_noalloc serves callers that cannot let the library allocate device memory (a
serving process that reserves its memory up front, memory owned by another framework's pool, a
latency-critical path): its scratch is a fixed device array inside the library. This file runs last
(pytest collects it last) and also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import kvc_synth
from oracle.kvc_oracle import OracleKVCache, gqa_cached_attention
from tests.gpu_parity import check_outputs

pytestmark = pytest.mark.gpu

NAMES = {0: "f32", 1: "f16", 2: "bf16"}


def _prefilled(kb, torch, dtype, L, B, H_kv, d, lengths, T, seed):
    """A GPU cache and its oracle mirror: max(lengths) rows appended and committed on every layer,
    truncated to each sequence's length, then a T-row chunk appended to every layer."""
    name = NAMES[dtype]
    max_len = max(lengths) + T + 4
    cache = kb.Cache(L, B, H_kv, d, max_len, dtype)
    ref = OracleKVCache(L, B, H_kv, d, max_len, name)
    s0 = max(lengths)
    for layer in range(L):
        k = kvc_synth.normal_f32((B, H_kv, s0, d), seed, 10 + layer)
        v = kvc_synth.normal_f32((B, H_kv, s0, d), seed, 20 + layer)
        ref.append(layer, k, v)
        kb.kvc_append(cache, layer, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    ref.commit()
    kb.kvc_commit(cache)
    ref.truncate(lengths)
    kb.kvc_truncate_ragged(cache, lengths)
    for layer in range(L):
        k = kvc_synth.normal_f32((B, H_kv, T, d), seed, 30 + layer)
        v = kvc_synth.normal_f32((B, H_kv, T, d), seed, 40 + layer)
        ref.append(layer, k, v)
        kb.kvc_append(cache, layer, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    return cache, ref


@pytest.mark.parametrize("dtype,d,H_q,H_kv,T,lengths", [
    (2, 128, 32, 8, 1, [4019, 544, 2300, 1, 0, 3000, 1500, 777]),   # tensor-core decode kernel, splits
    (1, 128, 32, 8, 8, [2048, 300]),                                 # tensor-core chunk kernel, verify chunk
    (0, 32, 4, 2, 1, [47, 1000]),                                    # CUDA-core kernel
])
def test_noalloc_matches_oracle_and_regular_entry_point_twice(gpu_lib, dtype, d, H_q, H_kv, T, lengths):
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    B, name = len(lengths), NAMES[dtype]
    cache, ref = _prefilled(kb, torch, dtype, 2, B, H_kv, d, lengths, T, seed=7)
    for layer in range(2):
        q_host = kvc_synth.normal_f32((B, H_q, T, d), 7, 50 + layer)
        q = torch.from_numpy(q_host).cuda()
        want = gqa_cached_attention(ref, layer, q_host)
        regular = kb.gqa_cached_attn(cache, q, layer).cpu().numpy()
        check_outputs(regular, want, name, f"regular layer {layer}")
        for call in range(2):                                # two calls in a row share the array
            out = torch.full((B, H_q, T, d), float("nan"), dtype=torch.float32, device="cuda")
            kb.gqa_cached_attn_noalloc(cache, q, layer, out)
            got = out.cpu().numpy()
            check_outputs(got, want, name, f"noalloc layer {layer} call {call}")
            check_outputs(got, regular, name, f"noalloc vs regular, layer {layer} call {call}")
    kb.kvc_status(cache)
    cache.close()


def test_noalloc_on_a_fresh_handle_allocates_nothing(gpu_lib):
    """On a handle that has never attended, the no-alloc call leaves the handle's workspace empty and
    the device's free memory unchanged, and still matches the oracle; a regular call on the same
    handle then grows the workspace (the plan has split units, so the scratch was really needed)."""
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    lengths, H_q, H_kv, d = [3000, 1, 1700, 0], 8, 2, 128
    B = len(lengths)
    warm, _ = _prefilled(kb, torch, 2, 1, B, H_kv, d, [40] * B, 1, seed=3)     # loads the kernels and
    q0 = torch.zeros((B, H_q, 1, d), device="cuda")                              # the array's module
    kb.gqa_cached_attn(warm, q0, 0)
    kb.gqa_cached_attn_noalloc(warm, q0, 0, torch.empty_like(q0))
    kb.kvc_status(warm)

    cache, ref = _prefilled(kb, torch, 2, 1, B, H_kv, d, lengths, 1, seed=11)
    q_host = kvc_synth.normal_f32((B, H_q, 1, d), 11, 60)
    q = torch.from_numpy(q_host).cuda()
    outs = [torch.empty((B, H_q, 1, d), dtype=torch.float32, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    launches = kb.kvc_launch_count(cache)
    for out in outs:
        kb.gqa_cached_attn_noalloc(cache, q, 0, out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert kb.kvc_workspace_bytes(cache) == 0
    assert kb.kvc_launch_count(cache) == launches + 2
    want = gqa_cached_attention(ref, 0, q_host)
    for i, out in enumerate(outs):
        check_outputs(out.cpu().numpy(), want, "bf16", f"fresh handle, call {i}")
    kb.gqa_cached_attn(cache, q, 0)
    assert kb.kvc_workspace_bytes(cache) > 0
    kb.kvc_status(cache)
    cache.close()
    warm.close()


def test_noalloc_rejects_a_latent_cache_before_any_launch(gpu_lib):
    """A latent (MLA) cache is read by mla_cached_attn; the no-alloc call refuses it on the host, as
    gqa_cached_attn does, and enqueues nothing."""
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    c = kb.LatentCache(1, 2, 128, 64, 64, kb.KVC_BF16)
    kb.kvc_append(c, 0, torch.zeros((2, 4, 128), dtype=torch.bfloat16, device="cuda"),
                  torch.zeros((2, 4, 64), dtype=torch.bfloat16, device="cuda"))
    launches = kb.kvc_launch_count(c)
    q = torch.zeros((2, 8, 4, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((2, 8, 4, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(kb.KvcError) as ei:
        kb.gqa_cached_attn_noalloc(c, q, 0, out)
    assert ei.value.code == -1 and "mla_cached_attn" in str(ei.value)
    assert kb.kvc_launch_count(c) == launches
    kb.kvc_status(c)
    c.close()


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
