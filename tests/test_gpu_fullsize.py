"""GPU parity at the workloads' full sizes, in the launch configuration the benchmark times.

One forward (every layer: append, attend; then commit) runs on the full workload. The oracle then
recomputes sampled (layer, sequence, K/V head) groups one by one from host redraws of the same
seeded inputs: their G query heads' outputs within tolerance, and the stored rows bit-exactly.
"""
import numpy as np
import pytest

import kvc_workloads
from oracle.kvc_oracle import OracleKVCache, OracleLatentCache, gqa_cached_attention, mla_cached_attention, rope_chunk
from tests.gpu_parity import check_outputs, check_rotated_store

pytestmark = pytest.mark.gpu


def _run_and_sample(wl, samples):
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    wl.prefill()
    inputs = wl.step_inputs(0)
    outs = []
    for layer, (*qs, k, v) in enumerate(inputs):
        wl.append(layer, k, v)
        outs.append(wl.attend(qs, layer))
    kb.kvc_commit(wl.cache)
    kb.kvc_status(wl.cache)
    G = wl.H_q // wl.H_kv
    view = {"f32": torch.int32, "e4m3": torch.uint8}.get(wl.dtype, torch.int16)
    for layer, b, kvh in samples:
        s_b = int(wl.lengths[b])
        ref = OracleKVCache(1, 1, 1, wl.d_h, s_b + wl.T, wl.dtype)
        rot = (lambda x, start: rope_chunk(x, [start], wl.rope_base, wl.rope_style)) if wl.rope_base else \
            (lambda x, start: x)
        if s_b:
            kp, vp = wl.host_prefill_rows(layer, b, kvh, s_b)
            ref.append(0, rot(kp[None, None], 0), vp[None, None])
            ref.commit()
        kn, vn = wl.host_step_rows(layer, 0, b, kvh)
        ref.append(0, rot(kn[None, None], s_b), vn[None, None])
        heads = list(range(kvh * G, (kvh + 1) * G))
        qh = rot(wl.host_queries(layer, 0, b, heads)[None], s_b)[0]
        want = gqa_cached_attention(ref, 0, qh[None])
        got = outs[layer][b, kvh * G:(kvh + 1) * G].cpu().numpy()[None]
        check_outputs(got, want, wl.dtype, f"layer {layer} b {b} kvh {kvh}")
        for is_k, store, want_rows in ((True, wl.cache.k, ref.k[0, 0, 0]), (False, wl.cache.v, ref.v[0, 0, 0])):
            bits = store.view(view)             # raw bits first: no indexing on float8 tensors
            if wl.block:                        # gather the sequence's rows through its block table
                p = torch.arange(s_b + wl.T)
                blk = torch.tensor(kb.kvc_block_table(wl.cache)[0][b])[p // wl.block]
                stored = bits[layer][blk.cuda(), kvh, (p % wl.block).cuda()]
            else:
                stored = bits[layer, b, kvh, :s_b + wl.T]
            stored = stored.contiguous().cpu().numpy()
            if wl.rope_base and is_k:
                check_rotated_store(stored, want_rows.view(stored.dtype), wl.dtype)
            else:
                np.testing.assert_array_equal(stored, want_rows.view(stored.dtype))
    assert kb.kvc_seq_len(wl.cache) == [int(x) + wl.T for x in wl.lengths]
    wl.close()


def test_llama3_8b_decode_bf16_ragged_full_size():
    """Llama-3-8B-shaped decode, bf16 cache: 32 layers, H_q=32, H_kv=8, d_h=128, B=64,
    ragged s_b ~ U[512, 4096], T=1."""
    wl = kvc_workloads.GpuWorkload(kvc_workloads.spec("llama3-8b-decode-bf16"))
    lo, hi = int(np.argmin(wl.lengths)), int(np.argmax(wl.lengths))
    _run_and_sample(wl, [(0, lo, 0), (31, hi, 7), (13, 17, 3), (22, 40, 5)])


def test_smollm2_decode_fp16_full_size():
    """SmolLM2-135M-shaped attention, fp16 cache: 30 layers, H_q=9, H_kv=3, d_h=64, B=8, s=2048, T=1."""
    _run_and_sample(kvc_workloads.GpuWorkload(kvc_workloads.spec("smollm2-135m-decode-fp16")),
                    [(0, 0, 0), (29, 7, 2), (11, 3, 1)])


def test_llama3_8b_verify_chunk_fp16_full_size():
    """Speculative verify chunk, fp16: H_q=32, H_kv=8, d_h=128, B=16, s=2048, T=8."""
    _run_and_sample(kvc_workloads.GpuWorkload(kvc_workloads.spec("llama3-8b-verify-fp16")),
                    [(0, 0, 0), (31, 15, 7), (7, 9, 2)])


def test_llama3_8b_prefill_chunk_fp16_full_size():
    """Prefill chunk, fp16: H_q=32, H_kv=8, d_h=128, B=16, T=512 at s=1024."""
    _run_and_sample(kvc_workloads.GpuWorkload(kvc_workloads.spec("llama3-8b-prefill-fp16")),
                    [(0, 0, 0), (31, 15, 7), (16, 4, 3)])


def test_llama3_8b_decode_bf16_paged16_full_size():
    """The Llama-3-8B-shaped ragged decode batch in a paged cache of 16-position blocks, each
    sequence's blocks B apart in the pool."""
    wl = kvc_workloads.GpuWorkload(kvc_workloads.spec("llama3-8b-decode-bf16-paged16"))
    lo, hi = int(np.argmin(wl.lengths)), int(np.argmax(wl.lengths))
    _run_and_sample(wl, [(0, lo, 0), (31, hi, 7), (13, 17, 3)])


def test_llama3_8b_decode_bf16_rope_full_size():
    """The ragged decode batch with fused RoPE (base 500000, rotate-half): keys rotated in the append,
    queries in the attention prologue."""
    wl = kvc_workloads.GpuWorkload(kvc_workloads.spec("llama3-8b-decode-bf16-rope"))
    lo, hi = int(np.argmin(wl.lengths)), int(np.argmax(wl.lengths))
    _run_and_sample(wl, [(0, lo, 0), (31, hi, 7), (9, 30, 4)])


def test_llama3_8b_decode_fp8_full_size():
    """The ragged decode batch in an FP8 E4M3 cache (scale 1): tensor-core decode over widened tiles."""
    wl = kvc_workloads.GpuWorkload(kvc_workloads.spec("llama3-8b-decode-fp8"))
    lo, hi = int(np.argmin(wl.lengths)), int(np.argmax(wl.lengths))
    _run_and_sample(wl, [(0, lo, 0), (31, hi, 7), (20, 11, 2)])


def test_deepseek_v2_lite_mla_decode_full_size():
    """Latent attention over a latent cache, DeepSeek-V2-Lite-shaped: 27 layers, 16 heads, r = 512,
    d_R = 64, the ragged 64-sequence decode batch; sampled (layer, sequence) pairs recomputed by the oracle
    from host redraws, all 16 heads, and their stored latent and RoPE-key rows bit-exact."""
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    wl = kvc_workloads.GpuWorkload(kvc_workloads.spec("deepseek-v2-lite-mla-decode-bf16"))
    wl.prefill()
    inputs = wl.step_inputs(0)
    outs = []
    for layer, (*qs, c, kr) in enumerate(inputs):
        wl.append(layer, c, kr)
        outs.append(wl.attend(qs, layer))
    kb.kvc_commit(wl.cache)
    kb.kvc_status(wl.cache)
    lo, hi = int(np.argmin(wl.lengths)), int(np.argmax(wl.lengths))
    for layer, b in [(0, lo), (26, hi), (13, 7)]:
        s_b = int(wl.lengths[b])
        ref = OracleLatentCache(1, 1, wl.d_h, wl.d_rope, s_b + wl.T, wl.dtype)
        ref.append(0, *(x[None] for x in wl.host_prefill_latent(layer, b, s_b)))
        ref.commit()
        ref.append(0, *(x[None] for x in wl.host_step_latent(layer, 0, b)))
        ql, qr = wl.host_queries_mla(layer, 0, b, range(wl.H_q))
        want = mla_cached_attention(ref, 0, ql[None], qr[None], wl.mla_scale)
        check_outputs(outs[layer][b:b + 1].cpu().numpy(), want, wl.dtype, f"mla layer {layer} b {b}")
        for store, want_rows in ((wl.cache.k, ref.c[0, 0]), (wl.cache.v, ref.kr[0, 0])):
            got = store[layer, b, :s_b + wl.T].contiguous().view(torch.int16).cpu().numpy()
            np.testing.assert_array_equal(got, want_rows.view(np.int16))
    wl.close()
