"""A decode step captured once in a CUDA graph and replayed gives the results of the same step made
call by call.

Every kernel of the library reads the lengths from the device and the host mirrors only validate and
plan, so a captured step (append and attention on every layer, commit, truncate back) replays
correctly as long as it ends where it began, which is how the benchmark times its graph mode. Checked
here bit for bit against a second cache driven by eager calls with the same inputs: the outputs of
every layer after each replay, then both stores and the lengths.
"""
import numpy as np
import pytest

import kvc_synth

pytestmark = pytest.mark.gpu

DT = {"f16": 1, "bf16": 2}


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    yield


def _cache(kb, torch, dtype, L, B, H_kv, d, lengths, T, seed):
    max_len = max(lengths) + T + 8
    c = kb.Cache(L, B, H_kv, d, max_len, DT[dtype])
    s0 = max(lengths)
    for layer in range(L):
        k = torch.from_numpy(kvc_synth.normal_f32((B, H_kv, s0, d), seed, 100 + layer)).cuda()
        v = torch.from_numpy(kvc_synth.normal_f32((B, H_kv, s0, d), seed, 200 + layer)).cuda()
        kb.kvc_append(c, layer, k, v)
    kb.kvc_commit(c)
    kb.kvc_truncate_ragged(c, lengths)
    return c


@pytest.mark.parametrize("dtype,d,Hq,Hkv,T,lengths,fused", [
    ("bf16", 128, 32, 8, 1, [1000, 0, 129, 2500], False),   # tensor-core decode kernel, split keys
    ("bf16", 128, 32, 8, 1, [1000, 0, 129, 2500], True),    # the same with the append fused into it
    ("f16", 64, 9, 3, 1, [2048, 7], True),                  # decode, d_h = 64
    ("f16", 128, 32, 8, 8, [300, 2048], False),             # verify chunk on the chunk kernel
])
def test_captured_step_replays_like_eager_calls(dtype, d, Hq, Hkv, T, lengths, fused):
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    L, B, seed = 3, len(lengths), 21
    graph_cache = _cache(kb, torch, dtype, L, B, Hkv, d, lengths, T, seed)
    eager_cache = _cache(kb, torch, dtype, L, B, Hkv, d, lengths, T, seed)
    q = [torch.from_numpy(kvc_synth.normal_f32((B, Hq, T, d), seed, 300 + l)).cuda() for l in range(L)]
    k = [torch.from_numpy(kvc_synth.normal_f32((B, Hkv, T, d), seed, 400 + l)).cuda() for l in range(L)]
    v = [torch.from_numpy(kvc_synth.normal_f32((B, Hkv, T, d), seed, 500 + l)).cuda() for l in range(L)]

    def step(c, outs):
        for layer in range(L):
            if fused:
                kb.gqa_cached_attn_append(c, layer, k[layer], v[layer], q[layer], out=outs[layer])
            else:
                kb.kvc_append(c, layer, k[layer], v[layer])
                kb.gqa_cached_attn(c, q[layer], layer, out=outs[layer])
        kb.kvc_commit(c)
        kb.kvc_truncate_ragged(c, lengths)                   # the step ends where it began

    want = [torch.empty((B, Hq, T, d), dtype=torch.float32, device="cuda") for _ in range(L)]
    step(eager_cache, want)
    got = [torch.full((B, Hq, T, d), float("nan"), dtype=torch.float32, device="cuda") for _ in range(L)]
    step(graph_cache, got)                                   # eager first: the workspace is sized here
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(graph_cache, got)
    for _ in range(3):
        for o in got:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for layer in range(L):
            assert torch.equal(got[layer], want[layer]), f"layer {layer}: replayed outputs differ from eager"
    kb.kvc_status(graph_cache)
    for mine, theirs in ((graph_cache.k, eager_cache.k), (graph_cache.v, eager_cache.v)):
        np.testing.assert_array_equal(mine.view(torch.int16).cpu().numpy(), theirs.view(torch.int16).cpu().numpy())
    assert kb.kvc_seq_len(graph_cache, -1) == [int(x) for x in lengths]
    graph_cache.close()
    eager_cache.close()
