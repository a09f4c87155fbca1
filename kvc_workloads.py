"""Synthetic workloads: their shapes, host redraws of their inputs, and GPU-resident instances.

Used by the GPU tests and by `bench.py`. Inputs are drawn on the device by the library's Philox
fill (`kvc_synth_fill_normal_f32`); `WorkloadSpec.host_*` redraw any slice of the same inputs on the
host with `kvc_synth`, so expected values never come from the device.

Layout of the draws (element index within each stream, row-major):
* prefill keys/values of layer l: [B, H_kv, S0, d_h] from streams (K_PREFILL | V_PREFILL, l), with
  S0 = max_b s_b; after committing S0 rows the cache is truncated to each s_b;
* step n of layer l: k_new/v_new [B, H_kv, T, d_h] from (K_STEP | V_STEP, l, n + 1), queries
  [B, H_q, T, d_h] from (Q, l, n + 1), all float32.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import kvc_synth
from kvc_synth import (STREAM_K_PREFILL, STREAM_K_STEP, STREAM_Q, STREAM_Q_ROPE, STREAM_V_PREFILL, STREAM_V_STEP,
                       stream_id)

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}
ITEMSIZE = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}


@dataclass
class WorkloadSpec:
    name: str
    L: int
    B: int
    H_q: int
    H_kv: int
    d_h: int
    max_len: int
    dtype: str
    lengths: np.ndarray
    T: int = 1
    seed: int = 0
    block: int = 0          # paged cache block (positions); 0 = contiguous cache
    rope_base: float = 0.0  # fused rotary positions (kvc_append_rope / gqa_cached_attn_rope); 0 = none
    rope_style: str = "half"
    d_rope: int = 0         # latent (MLA) workload: RoPE-key width; then H_q = heads, H_kv = 1, d_h = r
    mla_scale: float = 0.0

    @property
    def mla(self) -> bool:
        return self.d_rope > 0

    @property
    def S0(self) -> int:
        return int(self.lengths.max())

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    # -- host redraws ---------------------------------------------------------------------------
    def host_prefill_rows(self, layer, b, kvh, n):
        """Float32 draws of prefill rows [0, n) of (layer, b, kvh): ([n, d], [n, d])."""
        base = ((b * self.H_kv + kvh) * self.S0) * self.d_h
        idx = base + np.arange(n * self.d_h, dtype=np.int64)
        k = kvc_synth.normal_f32_at(idx, self.seed, stream_id(STREAM_K_PREFILL, layer)).reshape(n, self.d_h)
        v = kvc_synth.normal_f32_at(idx, self.seed, stream_id(STREAM_V_PREFILL, layer)).reshape(n, self.d_h)
        return k, v

    def host_step_rows(self, layer, step, b, kvh):
        """Draws of step `step`'s T new rows of (layer, b, kvh): ([T, d], [T, d])."""
        base = ((b * self.H_kv + kvh) * self.T) * self.d_h
        idx = base + np.arange(self.T * self.d_h, dtype=np.int64)
        k = kvc_synth.normal_f32_at(idx, self.seed, stream_id(STREAM_K_STEP, layer, step + 1))
        v = kvc_synth.normal_f32_at(idx, self.seed, stream_id(STREAM_V_STEP, layer, step + 1))
        return k.reshape(self.T, self.d_h), v.reshape(self.T, self.d_h)

    def host_queries(self, layer, step, b, heads):
        """Draws of the queries [len(heads), T, d] of sequence b at step `step`."""
        rows = []
        for h in heads:
            base = ((b * self.H_q + h) * self.T) * self.d_h
            idx = base + np.arange(self.T * self.d_h, dtype=np.int64)
            rows.append(kvc_synth.normal_f32_at(idx, self.seed, stream_id(STREAM_Q, layer, step + 1)))
        return np.stack(rows).reshape(len(heads), self.T, self.d_h)

    # -- accounting -----------------------------------------------------------------------------
    def attn_bytes(self, seqs=None) -> int:
        """Algorithmic HBM bytes of one attention call over sequences `seqs` (default all): each
        stored K and V row read once per K/V head (latent: each latent and RoPE-key row once), the
        float32 queries read, float32 outputs written."""
        lens = self.lengths if seqs is None else self.lengths[list(seqs)]
        n = len(lens)
        if self.mla:
            rows = (self.d_h + self.d_rope) * ITEMSIZE[self.dtype] * int((lens + self.T).sum())
            return rows + n * self.H_q * self.T * 4 * (2 * self.d_h + self.d_rope)
        kv = 2 * self.H_kv * self.d_h * ITEMSIZE[self.dtype] * int((lens + self.T).sum())
        return kv + 2 * n * self.H_q * self.T * self.d_h * 4

    def append_bytes(self) -> int:
        """Float32 chunk read plus rounded rows written, for K and V (latent and RoPE key), one layer."""
        if self.mla:
            return self.B * self.T * (self.d_h + self.d_rope) * (4 + ITEMSIZE[self.dtype])
        n = self.B * self.H_kv * self.T * self.d_h
        return 2 * n * (4 + ITEMSIZE[self.dtype])

    def step_bytes(self) -> int:
        return self.L * (self.attn_bytes() + self.append_bytes())

    def attn_flops(self) -> int:
        """Multiply-adds of QK^T and PV counted as 2 flops each, unmasked pairs only, one layer."""
        pairs = 0
        for s in self.lengths:
            pairs += self.T * int(s) + self.T * (self.T + 1) // 2
        if self.mla:
            return 2 * (2 * self.d_h + self.d_rope) * self.H_q * pairs
        return 4 * self.d_h * self.H_q * pairs

    # -- latent (MLA) host redraws: latent [B, S0, r] / RoPE key [B, S0, d_R] per layer, step chunks
    #    [B, T, r] / [B, T, d_R], queries [B, H, T, r] / [B, H, T, d_R] --------------------------------
    def host_prefill_latent(self, layer, b, n):
        c = kvc_synth.normal_f32_at(b * self.S0 * self.d_h + np.arange(n * self.d_h, dtype=np.int64), self.seed,
                                    stream_id(STREAM_K_PREFILL, layer)).reshape(n, self.d_h)
        kr = kvc_synth.normal_f32_at(b * self.S0 * self.d_rope + np.arange(n * self.d_rope, dtype=np.int64),
                                     self.seed, stream_id(STREAM_V_PREFILL, layer)).reshape(n, self.d_rope)
        return c, kr

    def host_step_latent(self, layer, step, b):
        T = self.T
        c = kvc_synth.normal_f32_at(b * T * self.d_h + np.arange(T * self.d_h, dtype=np.int64), self.seed,
                                    stream_id(STREAM_K_STEP, layer, step + 1)).reshape(T, self.d_h)
        kr = kvc_synth.normal_f32_at(b * T * self.d_rope + np.arange(T * self.d_rope, dtype=np.int64), self.seed,
                                     stream_id(STREAM_V_STEP, layer, step + 1)).reshape(T, self.d_rope)
        return c, kr

    def host_queries_mla(self, layer, step, b, heads):
        ql, qr = [], []
        for h in heads:
            row = (b * self.H_q + h) * self.T
            ql.append(kvc_synth.normal_f32_at(row * self.d_h + np.arange(self.T * self.d_h, dtype=np.int64),
                                              self.seed, stream_id(STREAM_Q, layer, step + 1)))
            qr.append(kvc_synth.normal_f32_at(row * self.d_rope + np.arange(self.T * self.d_rope, dtype=np.int64),
                                              self.seed, stream_id(STREAM_Q_ROPE, layer, step + 1)))
        return (np.stack(ql).reshape(len(heads), self.T, self.d_h),
                np.stack(qr).reshape(len(heads), self.T, self.d_rope))


def spec(name: str, seed: int = 0) -> WorkloadSpec:
    w = kvc_synth.WORKLOADS[name]
    if "s_lo" in w:
        lengths = kvc_synth.ragged_lengths(w["B"], w["s_lo"], w["s_hi"], seed)
    else:
        lengths = np.full(w["B"], w["s"], dtype=np.int64)
    if "r" in w:                        # latent (MLA) workload
        return WorkloadSpec(name, w["L"], w["B"], w["H"], 1, w["r"], w["max_len"], w["dtype"], lengths, T=w["T"],
                            seed=seed, d_rope=w["d_rope"], mla_scale=w["mla_scale"])
    return WorkloadSpec(name, w["L"], w["B"], w["H_q"], w["H_kv"], w["d_h"], w["max_len"], w["dtype"],
                        lengths, T=w["T"], seed=seed, block=w.get("block", 0),
                        rope_base=w.get("rope_base", 0.0), rope_style=w.get("rope_style", "half"))


class GpuWorkload:
    """A workload's cache on the GPU (prefilled through the public API) and its step inputs."""

    def __init__(self, sp: WorkloadSpec, device="cuda"):
        import torch
        from kv_cached_gqa_gb300 import _binding as kb
        self.torch, self.kb, self.spec, self.device = torch, kb, sp, device
        if sp.mla:
            self.cache = kb.LatentCache(sp.L, sp.B, sp.d_h, sp.d_rope, sp.max_len, DTYPE_CODE[sp.dtype], device=device)
        elif sp.block:
            n_blocks = sp.B * (-(-sp.max_len // sp.block))
            self.cache = kb.PagedCache(sp.L, sp.B, sp.H_kv, sp.d_h, sp.max_len, sp.block, n_blocks,
                                       DTYPE_CODE[sp.dtype], device=device)
        else:
            self.cache = kb.Cache(sp.L, sp.B, sp.H_kv, sp.d_h, sp.max_len, DTYPE_CODE[sp.dtype], device=device)
        if sp.rope_base:
            kb.kvc_set_rope(self.cache, sp.rope_base, sp.rope_style)

    def append(self, layer, k, v):
        """The workload's append: kvc_append, or kvc_append_rope when it rotates keys."""
        (self.kb.kvc_append_rope if self.spec.rope_base else self.kb.kvc_append)(self.cache, layer, k, v)

    def attend(self, qs, layer, out=None):
        """The workload's attention over its query tensors `qs`: gqa_cached_attn(_rope) of qs[0], or
        mla_cached_attn of (q_lat, q_rope)."""
        if self.spec.mla:
            return self.kb.mla_cached_attn(self.cache, qs[0], qs[1], layer, self.spec.mla_scale, out=out)
        fn = self.kb.gqa_cached_attn_rope if self.spec.rope_base else self.kb.gqa_cached_attn
        return fn(self.cache, qs[0], layer, out=out)

    def append_attend(self, layer, k, v, qs, out=None):
        """The workload's layer step in one call: gqa_cached_attn_append (rotating keys and queries when
        the workload uses RoPE). K/V workloads only."""
        return self.kb.gqa_cached_attn_append(self.cache, layer, k, v, qs[0], out=out, rope=bool(self.spec.rope_base))

    def __getattr__(self, name):                      # shape fields and host redraws of the spec
        return getattr(self.__dict__["spec"], name)

    def draw(self, shape, stream, std=1.0):
        t = self.torch.empty(shape, dtype=self.torch.float32, device=self.device)
        self.kb.synth_fill_normal(t, self.spec.seed, stream, std=std)
        return t

    def prefill(self):
        """Append S0 rows to every layer, commit, then truncate each sequence to s_b. A paged cache
        takes the rows one block of positions per append, so layer 0's appends hand each sequence one
        block in turn (the later layers reuse the same blocks) and a sequence's blocks end up B blocks
        apart in the pool."""
        sp, kb = self.spec, self.kb
        shape = (sp.B, sp.H_kv, sp.S0, sp.d_h)
        chunk = sp.block or sp.S0
        for layer in range(sp.L):
            if sp.mla:
                c = self.draw((sp.B, sp.S0, sp.d_h), stream_id(STREAM_K_PREFILL, layer))
                kr = self.draw((sp.B, sp.S0, sp.d_rope), stream_id(STREAM_V_PREFILL, layer))
                self.append(layer, c, kr)
                del c, kr
                continue
            k = self.draw(shape, stream_id(STREAM_K_PREFILL, layer))
            v = self.draw(shape, stream_id(STREAM_V_PREFILL, layer))
            for c0 in range(0, sp.S0, chunk):
                c1 = min(sp.S0, c0 + chunk)
                if c0 == 0 and c1 == sp.S0:
                    self.append(layer, k, v)
                else:
                    self.append(layer, k[:, :, c0:c1].contiguous(), v[:, :, c0:c1].contiguous())
            del k, v
        kb.kvc_commit(self.cache)
        kb.kvc_truncate_ragged(self.cache, [int(x) for x in sp.lengths])

    def step_inputs(self, step):
        """Float32 device tensors of every layer for step `step`: (q, k_new, v_new), or for a latent
        workload (q_lat, q_rope, c_new, kr_new); the last two are what the append takes."""
        sp = self.spec
        out = []
        for layer in range(sp.L):
            if sp.mla:
                out.append((self.draw((sp.B, sp.H_q, sp.T, sp.d_h), stream_id(STREAM_Q, layer, step + 1)),
                            self.draw((sp.B, sp.H_q, sp.T, sp.d_rope), stream_id(STREAM_Q_ROPE, layer, step + 1)),
                            self.draw((sp.B, sp.T, sp.d_h), stream_id(STREAM_K_STEP, layer, step + 1)),
                            self.draw((sp.B, sp.T, sp.d_rope), stream_id(STREAM_V_STEP, layer, step + 1))))
                continue
            q = self.draw((sp.B, sp.H_q, sp.T, sp.d_h), stream_id(STREAM_Q, layer, step + 1))
            k = self.draw((sp.B, sp.H_kv, sp.T, sp.d_h), stream_id(STREAM_K_STEP, layer, step + 1))
            v = self.draw((sp.B, sp.H_kv, sp.T, sp.d_h), stream_id(STREAM_V_STEP, layer, step + 1))
            out.append((q, k, v))
        return out

    def close(self):
        self.cache.close()
