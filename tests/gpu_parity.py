"""Helpers for the GPU parity tests: run the same operations on the library and on the oracle.

Inputs are float32 draws of `kvc_synth` made on the host and copied to the device, so the oracle and
the GPU see the same values; expected values come from `oracle/` only.
"""
from __future__ import annotations

import numpy as np

import kvc_synth
from oracle.kvc_oracle import (OracleKVCache, OracleLatentCache, OraclePagedKVCache, gqa_cached_attention,
                               mla_cached_attention, rope_chunk, set_fp8_scales, store_round, stored_to_f64)

DT = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}
QUERY_DT = {"f32": "f32", "f16": "f16", "bf16": "bf16", "e4m3": "f16"}   # the type a query is used in
FP32_ATOL = 1e-5        # float32 caches: absolute, every output element
REL_16 = 2e-3           # 16-bit caches: max |o - r| / max |r| over each (b, query head)


def check_outputs(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    """Compare [B, H_q, T, d_h] outputs with the tolerance the cache dtype allows."""
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if dtype == "f32":
        err = np.abs(got - want).max()
        assert err <= FP32_ATOL, f"{what}: max abs error {err:.3e} > {FP32_ATOL}"
        return err
    num = np.abs(got - want).max(axis=(2, 3))
    den = np.abs(want).max(axis=(2, 3))
    rel = (num / np.maximum(den, 1e-30)).max()
    assert rel <= REL_16, f"{what}: relative max-abs error {rel:.3e} > {REL_16}"
    return rel


def check_rotated_store(got_bits, want_bits, dtype):
    """Keys rotated on the GPU (float32 arithmetic from float32 cos/sin) against the oracle's float64
    rotation rounded to float32, then to the cache dtype. The float32 rotation of a pair (x, y) is off
    by at most about 4 * 2^-24 * (|x| + |y|), i.e. 2^-21 of the row's largest magnitude m; each side
    then rounds once to the cache dtype. So |got - want| <= ulp(want) + 2^-21 m for 16-bit caches
    (where x cos and y sin nearly cancel, the result is small and that is many of its own ulps) and
    2^-20 m for float32 caches; most elements must agree exactly."""
    if dtype == "f32":
        g = got_bits.view(np.float32).astype(np.float64)
        w = want_bits.view(np.float32).astype(np.float64)
        m = np.abs(w).max(axis=-1, keepdims=True)
        assert np.all(np.abs(g - w) <= 2.0 ** -20 * m), "rotated float32 keys differ"
        return
    if dtype == "e4m3":                      # codes: compare in code space (the scale cancels)
        from oracle.kvc_oracle import e4m3_decode
        g, w = e4m3_decode(got_bits.view(np.uint8)), e4m3_decode(want_bits.view(np.uint8))
        _, ex = np.frexp(np.abs(w))
        ulp = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
        m = np.abs(w).max(axis=-1, keepdims=True)
        err = np.abs(g - w)
        assert np.all(err <= ulp + 2.0 ** -21 * m), "rotated fp8 keys off by more than one grid step"
        assert np.count_nonzero(err) / err.size < 5e-3
        return
    npdt = np.float16 if dtype == "f16" else None
    if npdt is not None:
        g = got_bits.view(np.float16).astype(np.float64)
        w = want_bits.view(np.float16).astype(np.float64)
        ulp = np.spacing(np.abs(want_bits.view(np.float16))).astype(np.float64)
    else:
        g = (got_bits.astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        w = (want_bits.astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ulp = np.spacing(np.abs(w).astype(np.float32)).astype(np.float64) * 2.0 ** 16
    m = np.abs(w).max(axis=-1, keepdims=True)
    err = np.abs(g - w)
    bound = ulp + 2.0 ** -21 * m
    assert np.all(err <= bound), f"rotated keys off by {float((err / bound).max()):.2f} x the bound"
    frac = np.count_nonzero(err) / err.size
    assert frac < 5e-3, f"{frac:.2e} of rotated keys differ from the oracle"


class Mirror:
    """A GPU cache and an oracle cache driven by the same calls (paged when `block` is given: a pool of
    `n_blocks` blocks, by default enough for every sequence at max_len)."""

    def __init__(self, L, B, H_kv, d_h, max_len, dtype, seed=0, block=None, n_blocks=None, rope=None,
                 scales=None, owned=False):
        import torch
        from kv_cached_gqa_gb300 import _binding as kb
        self.torch, self.kb = torch, kb
        self.L, self.B, self.H, self.d, self.max_len, self.dtype, self.seed = L, B, H_kv, d_h, max_len, dtype, seed
        self.paged = block is not None
        if self.paged:
            n_blocks = n_blocks or B * (-(-max_len // block))
            self.gpu = kb.PagedCache(L, B, H_kv, d_h, max_len, block, n_blocks, DT[dtype])
            self.ref = OraclePagedKVCache(L, B, H_kv, d_h, max_len, block, n_blocks, dtype)
        else:   # owned: the library allocates and zero-fills the store (kvc_create)
            self.gpu = (kb.OwnedCache if owned else kb.Cache)(L, B, H_kv, d_h, max_len, DT[dtype])
            self.ref = OracleKVCache(L, B, H_kv, d_h, max_len, dtype)
        self.n_draws = 0
        self.rope = rope                      # (base, style): keys and queries rotated by position
        if rope is not None:
            kb.kvc_set_rope(self.gpu, rope[0], rope[1])
        if scales is not None:                # fp8: (k_scale, v_scale) per layer
            set_fp8_scales(self.ref, *scales)
            kb.kvc_set_kv_scales(self.gpu, self.ref.k_scale, self.ref.v_scale)

    def draw(self, shape):
        self.n_draws += 1
        return kvc_synth.normal_f32(shape, self.seed, 1000 + self.n_draws)

    def dev(self, x, dtype=None):
        t = self.torch.from_numpy(np.ascontiguousarray(x)).cuda()
        return t if dtype is None else t.to(dtype)

    def append(self, layer, T, in_dtype="f32"):
        k = self.draw((self.B, self.H, T, self.d))
        v = self.draw((self.B, self.H, T, self.d))
        # the oracle stores what the GPU receives: the float32 draws, or their 16-bit rounding
        def given(x):
            return x if in_dtype == "f32" else stored_to_f64(store_round(x, in_dtype), in_dtype).astype(np.float32)
        k_in = given(k)
        if self.rope is not None:
            k_in = rope_chunk(k_in, self.ref.seq_len(layer), *self.rope)
        self.ref.append(layer, k_in, given(v))
        if in_dtype == "f32":
            kd, vd = self.dev(k), self.dev(v)
        else:
            # input already in the cache dtype: hand the oracle's own rounding of it to both sides
            tdt = self.kb.torch_dtype(DT[in_dtype])
            kd, vd = self.dev(k).to(tdt), self.dev(v).to(tdt)
        if self.rope is not None:
            self.kb.kvc_append_rope(self.gpu, layer, kd, vd)
        else:
            self.kb.kvc_append(self.gpu, layer, kd, vd)

    def attend(self, layer, H_q, T, q_in="f32", split_keys=0):
        q = self.draw((self.B, H_q, T, self.d))
        if self.rope is not None:
            q_in_vals = q if q_in == "f32" else stored_to_f64(store_round(q, q_in), q_in).astype(np.float32)
            want = gqa_cached_attention(self.ref, layer, rope_chunk(q_in_vals, self.ref.committed(), *self.rope))
        else:
            want = gqa_cached_attention(self.ref, layer, q)
        qd = self.dev(q) if q_in == "f32" else self.dev(q).to(self.kb.torch_dtype(DT[q_in]))
        if split_keys:
            self.kb.kvc_set_split_keys(self.gpu, split_keys)
        attn = self.kb.gqa_cached_attn_rope if self.rope is not None else self.kb.gqa_cached_attn
        got = attn(self.gpu, qd, layer).cpu().numpy()
        if split_keys:
            self.kb.kvc_set_split_keys(self.gpu, 0)
        return got, want

    def append_attend(self, layer, T, H_q, split_keys=0):
        """The draws of append() then attend(), handed to the GPU in one gqa_cached_attn_append call
        (the oracle appends, then attends): (got, want)."""
        k = self.draw((self.B, self.H, T, self.d))
        v = self.draw((self.B, self.H, T, self.d))
        k_in = k if self.rope is None else rope_chunk(k, self.ref.seq_len(layer), *self.rope)
        self.ref.append(layer, k_in, v)
        q = self.draw((self.B, H_q, T, self.d))
        q_att = q if self.rope is None else rope_chunk(q, self.ref.committed(), *self.rope)
        want = gqa_cached_attention(self.ref, layer, q_att)
        if split_keys:
            self.kb.kvc_set_split_keys(self.gpu, split_keys)
        got = self.kb.gqa_cached_attn_append(self.gpu, layer, self.dev(k), self.dev(v), self.dev(q),
                                             rope=self.rope is not None).cpu().numpy()
        if split_keys:
            self.kb.kvc_set_split_keys(self.gpu, 0)
        return got, want

    def commit(self):
        self.ref.commit()
        self.kb.kvc_commit(self.gpu)

    def truncate(self, n):
        self.ref.truncate(n)
        if np.ndim(n):
            self.kb.kvc_truncate_ragged(self.gpu, list(n))
        else:
            self.kb.kvc_truncate(self.gpu, int(n))

    def set_lengths(self, n):
        self.ref.set_lengths(n)
        self.kb.kvc_set_lengths(self.gpu, list(n))

    def forward(self, T, H_q, check=True, what=""):
        """One forward over every layer: append, attend, then commit."""
        errs = []
        for layer in range(self.L):
            self.append(layer, T)
            got, want = self.attend(layer, H_q, T)
            if check:
                errs.append(check_outputs(got, want, self.dtype, f"{what} layer {layer}"))
        self.commit()
        return errs

    def store_bits(self):
        """GPU store as raw bits and the oracle store as raw bits (same dtype/shape)."""
        torch = self.torch
        view, npview = {"f32": (torch.int32, np.int32), "e4m3": (torch.uint8, np.uint8)}.get(
            self.dtype, (torch.int16, np.int16))
        gk = self.gpu.k.view(view).cpu().numpy()
        gv = self.gpu.v.view(view).cpu().numpy()
        rk = self.ref.k.view(npview)
        rv = self.ref.v.view(npview)
        return (gk, gv), (rk, rv)

    def check_state(self):
        (gk, gv), (rk, rv) = self.store_bits()
        if self.rope is None:
            np.testing.assert_array_equal(gk, rk)
        else:
            check_rotated_store(gk, rk, self.dtype)
        np.testing.assert_array_equal(gv, rv)
        assert self.kb.kvc_seq_len(self.gpu, -1) == [int(x) for x in self.ref.committed()]
        for layer in range(self.L):
            assert self.kb.kvc_seq_len(self.gpu, layer) == [int(x) for x in self.ref.seq_len(layer)]
        pos = self.kb.kvc_positions(self.gpu, 3).cpu().numpy()
        np.testing.assert_array_equal(pos, self.ref.positions(3))
        if self.paged:
            table, n_free = self.kb.kvc_block_table(self.gpu)
            np.testing.assert_array_equal(np.array(table), self.ref.table)
            assert n_free == len(self.ref.free)

    def close(self):
        self.gpu.close()


class LatentMirror:
    """A GPU latent (MLA) cache and the oracle's, driven by the same calls."""

    def __init__(self, L, B, r, d_rope, max_len, dtype, seed=0):
        import torch
        from kv_cached_gqa_gb300 import _binding as kb
        self.torch, self.kb = torch, kb
        self.L, self.B, self.r, self.dR, self.max_len, self.dtype, self.seed = L, B, r, d_rope, max_len, dtype, seed
        self.gpu = kb.LatentCache(L, B, r, d_rope, max_len, DT[dtype])
        self.ref = OracleLatentCache(L, B, r, d_rope, max_len, dtype)
        self.n_draws = 0

    def draw(self, shape):
        self.n_draws += 1
        return kvc_synth.normal_f32(shape, self.seed, 5000 + self.n_draws)

    def dev(self, x, dtype=None):
        t = self.torch.from_numpy(np.ascontiguousarray(x)).cuda()
        return t if dtype is None else t.to(dtype)

    def append(self, layer, T, in_dtype="f32"):
        c, kr = self.draw((self.B, T, self.r)), self.draw((self.B, T, self.dR))

        def given(x):
            return x if in_dtype == "f32" else stored_to_f64(store_round(x, in_dtype), in_dtype).astype(np.float32)
        self.ref.append(layer, given(c), given(kr))
        tdt = None if in_dtype == "f32" else self.kb.torch_dtype(DT[in_dtype])
        self.kb.kvc_append(self.gpu, layer, self.dev(c, tdt), self.dev(kr, tdt))

    def attend(self, layer, H, T, scale, q_in="f32"):
        ql, qr = self.draw((self.B, H, T, self.r)), self.draw((self.B, H, T, self.dR))
        want = mla_cached_attention(self.ref, layer, ql, qr, scale)
        tdt = None if q_in == "f32" else self.kb.torch_dtype(DT[q_in])
        got = self.kb.mla_cached_attn(self.gpu, self.dev(ql, tdt), self.dev(qr, tdt), layer, scale).cpu().numpy()
        return got, want

    def commit(self):
        self.ref.commit()
        self.kb.kvc_commit(self.gpu)

    def truncate(self, n):
        self.ref.truncate(n)
        self.kb.kvc_truncate_ragged(self.gpu, [int(x) for x in np.broadcast_to(n, (self.B,))])

    def forward(self, T, H, scale, what=""):
        for layer in range(self.L):
            self.append(layer, T)
            got, want = self.attend(layer, H, T, scale)
            check_outputs(got, want, self.dtype, f"{what} layer {layer}")
        self.commit()

    def check_state(self):
        torch = self.torch
        view, npview = (torch.int32, np.int32) if self.dtype == "f32" else (torch.int16, np.int16)
        np.testing.assert_array_equal(self.gpu.k.view(view).cpu().numpy(), self.ref.c.view(npview))
        np.testing.assert_array_equal(self.gpu.v.view(view).cpu().numpy(), self.ref.kr.view(npview))
        assert self.kb.kvc_seq_len(self.gpu, -1) == [int(x) for x in self.ref.committed()]
        for layer in range(self.L):
            assert self.kb.kvc_seq_len(self.gpu, layer) == [int(x) for x in self.ref.seq_len(layer)]
        np.testing.assert_array_equal(self.kb.kvc_positions(self.gpu, 2).cpu().numpy(), self.ref.positions(2))

    def close(self):
        self.gpu.close()
