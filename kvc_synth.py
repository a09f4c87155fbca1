"""Seeded synthetic inputs for the KV-cached GQA attention step.

This module is shared by the CPU oracle's tests and by the GPU path's tests and
benchmark. It holds no attention, cache or rounding arithmetic: it only draws
numbers and names the workload shapes.

The generator is Philox4x32-10, the counter-based generator of Salmon, Moraes,
Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011), §3.
The GPU side implements the same published definition in its own CUDA source
(`kvc_synth_fill_f32`), so a large input drawn on the device can be redrawn
here, element by element, without ever copying device data into the oracle.

An "approximately standard normal" value is the Irwin-Hall sum of twelve
24-bit uniforms, centred: x = (sum_{i<12} (w_i >> 8) - 6 * 2^24) * 2^-24,
computed exactly in int64/float64 and rounded once to float32 (round to
nearest even). Every step is exact integer arithmetic or one correctly
rounded IEEE operation, so host and device produce identical bits. It has
mean ~0 and variance 1 and is bounded by |x| < 6; it stands in for the pages'
N(0, 1) draws.

Element `i` of stream `stream` under key `seed` uses the three Philox blocks
with counter (i mod 2^32, i >> 32, stream, j) for j = 0, 1, 2 and key
(seed mod 2^32, seed >> 32).
"""
from __future__ import annotations

import numpy as np

# Philox4x32-10 constants (Salmon et al. 2011, §3.2; Random123's defaults).
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint32(0x9E3779B9)
PHILOX_W1 = np.uint32(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten Philox4x32 rounds on arrays of 32-bit counters; returns four uint32 arrays."""
    c0 = np.asarray(c0, dtype=np.uint32)
    c1 = np.asarray(c1, dtype=np.uint32)
    c2 = np.asarray(c2, dtype=np.uint32)
    c3 = np.asarray(c3, dtype=np.uint32)
    k0 = np.asarray(k0, dtype=np.uint32)
    k1 = np.asarray(k1, dtype=np.uint32)
    for r in range(10):
        p0 = PHILOX_M0 * c0.astype(np.uint64)
        p1 = PHILOX_M1 * c2.astype(np.uint64)
        hi0 = (p0 >> np.uint64(32)).astype(np.uint32)
        lo0 = (p0 & _MASK32).astype(np.uint32)
        hi1 = (p1 >> np.uint64(32)).astype(np.uint32)
        lo1 = (p1 & _MASK32).astype(np.uint32)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        if r < 9:
            k0 = ((k0.astype(np.uint64) + np.uint64(PHILOX_W0)) & _MASK32).astype(np.uint32)
            k1 = ((k1.astype(np.uint64) + np.uint64(PHILOX_W1)) & _MASK32).astype(np.uint32)
    return c0, c1, c2, c3


def normal_f32_at(idx, seed: int, stream: int) -> np.ndarray:
    """Approximately N(0,1) float32 values for the element indices `idx` (int64 array)."""
    idx = np.asarray(idx, dtype=np.uint64)
    lo = (idx & _MASK32).astype(np.uint32)
    hi = (idx >> np.uint64(32)).astype(np.uint32)
    st = np.full(idx.shape, stream & 0xFFFFFFFF, dtype=np.uint32)
    k0 = np.uint32(seed & 0xFFFFFFFF)
    k1 = np.uint32((seed >> 32) & 0xFFFFFFFF)
    total = np.zeros(idx.shape, dtype=np.int64)
    for j in range(3):
        words = philox4x32_10(lo, hi, st, np.full(idx.shape, j, np.uint32), k0, k1)
        for w in words:
            total += (w >> np.uint32(8)).astype(np.int64)
    centred = (total - 6 * (1 << 24)).astype(np.float64) * (2.0 ** -24)
    return centred.astype(np.float32)


def normal_f32(shape, seed: int, stream: int, std: float = 1.0, offset: int = 0) -> np.ndarray:
    """A seeded tensor of the given shape; element i (row-major) is drawn at index offset + i.

    `std` != 1 multiplies in float32 after drawing (used for the N(0, 0.02) weights).
    """
    n = int(np.prod(shape)) if len(shape) else 1
    x = normal_f32_at(np.arange(offset, offset + n, dtype=np.int64), seed, stream).reshape(shape)
    if std != 1.0:
        x = (x * np.float32(std)).astype(np.float32)
    return x


def uniform_ints(n: int, lo: int, hi: int, seed: int, stream: int) -> np.ndarray:
    """n integers in [lo, hi] inclusive: lo + (w0 mod (hi - lo + 1)) from block (i, 0, stream, 3).

    The modulo bias is below 2^-20 for the ranges used here.
    """
    i = np.arange(n, dtype=np.uint64)
    w0, _, _, _ = philox4x32_10((i & _MASK32).astype(np.uint32), (i >> np.uint64(32)).astype(np.uint32),
                                np.full(n, stream, np.uint32), np.full(n, 3, np.uint32),
                                np.uint32(seed & 0xFFFFFFFF), np.uint32(seed >> 32))
    return (lo + (w0.astype(np.int64) % (hi - lo + 1))).astype(np.int64)


# Stream identifiers: each logical tensor of a workload draws from its own stream.
STREAM_Q = 1
STREAM_K_PREFILL = 2
STREAM_V_PREFILL = 3
STREAM_K_STEP = 4
STREAM_V_STEP = 5
STREAM_LENGTHS = 6
STREAM_WEIGHTS = 7
STREAM_PROMPT = 8
STREAM_Q_ROPE = 9           # the RoPE part of a latent-attention query


def stream_id(base: int, layer: int = 0, step: int = 0) -> int:
    """Distinct 32-bit stream per (tensor kind, layer, step): base | layer << 8 | step << 16."""
    return (base & 0xFF) | ((layer & 0xFF) << 8) | ((step & 0xFFFF) << 16)


# The workloads the pages describe, by shape (names state what they are).
WORKLOADS = {
    "toy-gqa-fp32": dict(L=4, B=1, H_q=4, H_kv=2, d_h=32, max_len=128, dtype="f32",
                         prefill=48, decode_steps=20, seed=0),
    "tiny-decoder-fp32": dict(vocab=96, d_model=128, n_heads=4, n_layers=4, max_len=256,
                              prompt=48, new_tokens=20, weight_std=0.02, seed=0),
    "smollm2-135m-decode-fp16": dict(L=30, B=8, H_q=9, H_kv=3, d_h=64, s=2048, T=1,
                                     dtype="f16", max_len=2112, seed=0),
    "llama3-8b-decode-bf16": dict(L=32, B=64, H_q=32, H_kv=8, d_h=128, s_lo=512, s_hi=4096, T=1,
                                  dtype="bf16", max_len=4160, seed=0),
    # the decode batch above in a paged cache: blocks of 16 or 128 positions, prefilled one block per
    # sequence at a time so each sequence's blocks lie B blocks apart in the pool
    "llama3-8b-decode-bf16-paged16": dict(L=32, B=64, H_q=32, H_kv=8, d_h=128, s_lo=512, s_hi=4096, T=1,
                                          dtype="bf16", max_len=4160, block=16, seed=0),
    "llama3-8b-decode-bf16-paged128": dict(L=32, B=64, H_q=32, H_kv=8, d_h=128, s_lo=512, s_hi=4096, T=1,
                                           dtype="bf16", max_len=4160, block=128, seed=0),
    # the decode batch with fused rotary positions (keys rotated in the append, queries in the
    # attention prologue; Llama-3's base 500000, rotate-half pairs)
    "llama3-8b-decode-bf16-rope": dict(L=32, B=64, H_q=32, H_kv=8, d_h=128, s_lo=512, s_hi=4096, T=1,
                                       dtype="bf16", max_len=4160, rope_base=500000.0, rope_style="half",
                                       seed=0),
    # the decode batch in an FP8 E4M3 cache (scale 1 for every layer): half the bytes per key
    "llama3-8b-decode-fp8": dict(L=32, B=64, H_q=32, H_kv=8, d_h=128, s_lo=512, s_hi=4096, T=1,
                                 dtype="e4m3", max_len=4160, seed=0),
    # multi-head latent attention over a latent cache, DeepSeek-V2-Lite-shaped (27 layers, 16 heads,
    # latent 512, RoPE key 64, softmax scale 1/sqrt(128 + 64)); the decode batch's lengths
    "deepseek-v2-lite-mla-decode-bf16": dict(L=27, B=64, H=16, r=512, d_rope=64, s_lo=512, s_hi=4096, T=1,
                                             dtype="bf16", max_len=4160, mla_scale=192 ** -0.5, seed=0),
    # the same with DeepSeek-V3's 128 heads and 61 layers
    "deepseek-v3-mla-decode-bf16": dict(L=61, B=64, H=128, r=512, d_rope=64, s_lo=512, s_hi=4096, T=1,
                                        dtype="bf16", max_len=4160, mla_scale=192 ** -0.5, seed=0),
    "llama3-8b-verify-fp16": dict(L=32, B=16, H_q=32, H_kv=8, d_h=128, s=2048, T=8, rollback=5,
                                  dtype="f16", max_len=2112, seed=0),
    "llama3-8b-prefill-fp16": dict(L=32, B=16, H_q=32, H_kv=8, d_h=128, s=1024, T=512,
                                   dtype="f16", max_len=1536, seed=0),
}


def ragged_lengths(B: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Per-sequence committed lengths s_b drawn uniformly from the integers [lo, hi]."""
    return uniform_ints(B, lo, hi, seed, STREAM_LENGTHS)


def prompt_ids(P: int, vocab: int, seed: int) -> list[int]:
    """A seeded prompt of P token ids in [0, vocab)."""
    return [int(i) for i in uniform_ints(P, 0, vocab - 1, seed, STREAM_PROMPT)]
