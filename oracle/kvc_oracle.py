"""CPU oracle for the KV-cached grouped-query attention step of autoregressive decoding.

TEST INFRASTRUCTURE ONLY. Only `tests/`, `__graft_entry__.smoke()` and the CPU
baseline leg of `bench.py` may import this module. The GPU library never calls
it, links it or shares code with it; the product path fails loudly when its
CUDA extension is missing rather than falling back to anything here.

It computes the plain definitions, in float64, one (sequence, head) at a time:

* the cache store and its bookkeeping: per-layer fill counts, a committed
  length that moves once per forward, truncate for rollback, and the storage
  dtype that rounds on the way in ("KV cache, incremental decode, incremental
  UTF-8 detokenizer, generate", §2.3 "Committed length, positions, and the
  mask", §2.4 "Rollback", §2.5 "Storage dtype", §4 "The interface");
* the bottom-right-aligned causal mask, mask(T)_ij = [j <= s + i] for
  0 <= i < T, 0 <= j < s + T (same page, §2.3 equation);
* scaled dot-product attention over the cache, softmax(q K^T / sqrt(d_h)) V,
  with masked scores removed ("Generation and the KV Cache", fence 3 "a toy
  KV cache equals recomputation"; "KV cache decoding", step 6);
* grouped-query head sharing, query head h reading K/V head h // G in the
  order [0, 0, 1, 1] for 4 query and 2 K/V heads ("Heads, GQA and K/V cache",
  "Four queries, two sets of K/V");
* the uncached full recompute that the cached path must equal ("KV cache
  decoding", "Why the causal mask makes caching exact");
* the paged cache: fixed-size blocks and a per-sequence block table ("KV cache decoding",
  "Batching caches of different lengths");
* the MLA latent cache and the absorbed multi-head latent attention that reads it ("KV cache,
  incremental decode, ...", §2.6; the attention is DeepSeek-V2's, which the pages name through MLA);
* rotary positions applied to the keys before they are stored and to the queries before they
  attend ("KV cache decoding", "Position information with a cache"; the formula is the RoFormer
  paper's, which the pages name but do not print).

Readings where the pages are silent (the library follows the same ones):
* rounding to float16/bfloat16 is round-to-nearest-even; NaN inputs are out of scope;
* a query for a 16-bit cache is rounded to the cache dtype before use;
* `commit` is explicit and requires every layer's fill to agree per sequence;
* `truncate(n)` requires n <= the committed length and leaves stale rows in place;
* the paged cache hands out the lowest-numbered free block first and frees, on truncate, every
  block wholly past the new length;
* RoPE: theta_i = base^(-2i/d) with pairs (i, i + d/2) or (2i, 2i + 1); a rotated row is rounded to
  float32 before the cache dtype;
* fp8 caches store E4M3 codes of x / scale (one K and one V scale per layer; round to nearest even,
  saturating at 448); a query meets an fp8 cache rounded to float16.

Parity status: every function here is pinned by `tests/test_oracle_pins.py`.
"""
from __future__ import annotations

import numpy as np

DTYPES = ("f32", "f16", "bf16", "f64", "e4m3")
ITEMSIZE = {"f32": 4, "f16": 2, "bf16": 2, "f64": 8, "e4m3": 1}
E4M3_MAX = 448.0


# ----------------------------------------------------------------------------------------------
# Storage rounding ("KV cache, incremental decode, ...", §2.5 "Storage dtype": values are
# converted on the way in and the stored values are what every later read returns).
# ----------------------------------------------------------------------------------------------

def e4m3_encode(x) -> np.ndarray:
    """float32 values -> FP8 E4M3 codes (uint8): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
    subnormals below 2^-6 in steps of 2^-9, no infinities, largest finite 448. Round to nearest even on
    the value grid, then saturate to +-448 (NaN inputs are out of scope)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    _, ex = np.frexp(a)                             # a = m * 2^ex, m in [0.5, 1): binade exponent ex - 1
    e = np.maximum(ex - 1, -6)                      # below 2^-6 the grid is the subnormal one
    quantum = np.ldexp(1.0, e - 3)                  # 3 mantissa bits
    r = np.minimum(np.rint(a / quantum) * quantum, E4M3_MAX)   # a / quantum is exact: a power of two
    # encode the (now representable) magnitude
    _, rex = np.frexp(r)
    normal = r >= 2.0 ** -6
    exp_field = np.where(normal, rex - 1 + 7, 0)
    man = np.where(normal, np.rint((r / np.ldexp(1.0, rex - 1) - 1.0) * 8), np.rint(r / 2.0 ** -9))
    code = (exp_field.astype(np.int64) << 3) | man.astype(np.int64)
    return (code | (neg.astype(np.int64) << 7)).astype(np.uint8)


def e4m3_decode(c) -> np.ndarray:
    """FP8 E4M3 codes -> float64 values (codes 0x7F / 0xFF are NaN)."""
    c = np.asarray(c, dtype=np.uint8).astype(np.int64)
    exp_field = (c >> 3) & 15
    man = c & 7
    mag = np.where(exp_field == 0, man * 2.0 ** -9, (1.0 + man / 8.0) * np.ldexp(1.0, exp_field - 7))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where(c & 0x80, -mag, mag)


def store_round(x, dtype: str) -> np.ndarray:
    """Convert float32 input values to the cache's stored representation.

    f32 -> float32 copy; f16 -> IEEE half (NumPy's astype, round to nearest even);
    bf16 -> uint16 bit patterns, rounding float32 to its top 16 bits to nearest even;
    e4m3 -> uint8 FP8 E4M3 codes (round to nearest even, saturating; a cache's scale is applied by
    the caller); f64 -> float64 (the NumPy default store of the "KV cache decoding" listing).
    """
    x = np.asarray(x)
    if dtype == "f64":
        return x.astype(np.float64)
    x = x.astype(np.float32)
    if dtype == "e4m3":
        return e4m3_encode(x)
    if dtype == "f32":
        return x.copy()
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        # keep the top 16 bits; add half an ulp minus one, plus the kept lsb, so ties go to even
        u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
        return u.astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def stored_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of stored elements (an fp8 cache's scale is applied by the caller)."""
    if dtype == "e4m3":
        return e4m3_decode(a)
    if dtype == "bf16":
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def storage_np_dtype(dtype: str):
    return {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "f64": np.float64, "e4m3": np.uint8}[dtype]


# ----------------------------------------------------------------------------------------------
# The offset causal mask ("KV cache, incremental decode, ...", §2.3 equation; "KV cache decoding",
# step 3: row i of a chunk at positions t..t+m-1 may attend to columns 0..t+i).
# ----------------------------------------------------------------------------------------------

def offset_causal_mask(T: int, s: int) -> np.ndarray:
    """Boolean [T, s + T]: entry (i, j) is True when key j is visible to query i, i.e. j <= s + i."""
    if T < 0 or s < 0:
        raise ValueError("T and s must be non-negative")
    i = np.arange(T)[:, None]
    j = np.arange(s + T)[None, :]
    return j <= s + i


def kv_bytes(layers: int, heads: int, head_dim: int, seq_len: int, batch: int = 1,
             bytes_per_value: int = 2) -> int:
    """K plus V bytes: 2 * layers * heads * head_dim * seq_len * batch * bytes ("KV cache decoding",
    "What is cached, what is not, and what it costs"; "Heads, GQA and K/V cache", "Memory and the
    window limit"; "Generation and the KV Cache", "Memory")."""
    return 2 * layers * heads * head_dim * seq_len * batch * bytes_per_value


# ----------------------------------------------------------------------------------------------
# FP8 storage. The pages name cache quantisation as a decode lever ("KV cache decoding", "What is
# cached, what is not, and what it costs") but give no format. Reading: E4M3 codes with one scale per
# layer for K and one for V, stored = e4m3(x / scale) (float32 division, round to nearest even,
# saturating), read back as code * scale.
# ----------------------------------------------------------------------------------------------

def set_fp8_scales(cache, k_scale, v_scale) -> None:
    """Per-layer K and V scales of an fp8 cache, fixed while it holds no rows."""
    if cache.dtype != "e4m3":
        raise ValueError("scales belong to fp8 caches")
    if np.any(cache.fill != 0):
        raise RuntimeError("scales change only while the cache is empty")
    k = np.broadcast_to(np.asarray(k_scale, dtype=np.float32), (cache.L,)).copy()
    v = np.broadcast_to(np.asarray(v_scale, dtype=np.float32), (cache.L,)).copy()
    if not (np.all(np.isfinite(k)) and np.all(k > 0) and np.all(np.isfinite(v)) and np.all(v > 0)):
        raise ValueError("scales must be positive and finite")
    cache.k_scale, cache.v_scale = k, v


def quantize_rows(x, dtype: str, scale) -> np.ndarray:
    """Stored form of float32 rows: store_round, after dividing by the layer's scale for fp8."""
    if dtype == "e4m3":
        return store_round(np.asarray(x, dtype=np.float32) / np.float32(scale), dtype)
    return store_round(x, dtype)


# ----------------------------------------------------------------------------------------------
# The cache ("KV cache, incremental decode, ...", §4 "The interface": seq_len, update, positions,
# mask, truncate, nbytes; "Generation and the KV Cache": k, v of shape (L, B, H, max_len, d_head)).
# ----------------------------------------------------------------------------------------------

class OracleKVCache:
    """Preallocated (L, B, H_kv, max_len, d_h) store with per-layer fills and committed lengths.

    Every method validates before it mutates: on any error nothing changes ("KV cache,
    incremental decode, ...", §4 test_update_copies_and_checks).
    """

    def __init__(self, n_layers: int, batch: int, n_kv_heads: int, d_head: int, max_len: int,
                 dtype: str = "f32"):
        if dtype not in DTYPES:
            raise ValueError(f"unknown dtype {dtype!r}")
        if min(n_layers, batch, n_kv_heads, d_head, max_len) <= 0:
            raise ValueError("all sizes must be positive")
        self.L, self.B, self.H, self.d, self.max_len, self.dtype = (
            n_layers, batch, n_kv_heads, d_head, max_len, dtype)
        shape = (n_layers, batch, n_kv_heads, max_len, d_head)
        self.k = np.zeros(shape, dtype=storage_np_dtype(dtype))
        self.v = np.zeros(shape, dtype=storage_np_dtype(dtype))
        self.fill = np.zeros((n_layers, batch), dtype=np.int64)   # per-layer fill counts
        self.lens = np.zeros(batch, dtype=np.int64)               # committed lengths s_b
        self.k_scale = np.ones(n_layers, dtype=np.float32)        # fp8 caches: stored = e4m3(x / scale)
        self.v_scale = np.ones(n_layers, dtype=np.float32)

    # -- lengths ---------------------------------------------------------------------------
    def seq_len(self, layer: int | None = None) -> np.ndarray:
        """Committed length as the minimum fill over layers (§2.3), or one layer's fill count."""
        if layer is None:
            return self.fill.min(axis=0).copy()
        return self.fill[layer].copy()

    def committed(self) -> np.ndarray:
        return self.lens.copy()

    def positions(self, T: int) -> np.ndarray:
        """[B, T] absolute positions [s_b, s_b + T) of the next chunk (what RoPE rotates by)."""
        return self.lens[:, None] + np.arange(T)[None, :]

    def mask(self, T: int, b: int = 0) -> np.ndarray:
        """causal_mask(T, s + T, q_offset=s) for sequence b, read from the committed length."""
        return offset_causal_mask(T, int(self.lens[b]))

    # -- writes ----------------------------------------------------------------------------
    def append(self, layer: int, k_new, v_new):
        """Write a [B, H_kv, T, d_h] chunk at each sequence's fill of this layer; return all rows.

        Returns, per sequence, the stored (rounded) keys and values [H_kv, fill, d_h] as float64:
        the past and the new chunk both come back as stored ("KV cache, incremental decode, ...",
        §2.5; "KV cache decoding", step 5).
        """
        if not 0 <= layer < self.L:
            raise ValueError("layer out of range")
        k_new = np.asarray(k_new)
        v_new = np.asarray(v_new)
        if k_new.ndim != 4 or k_new.shape != v_new.shape:
            raise ValueError("k_new and v_new must both be [B, H_kv, T, d_h]")
        B, H, T, d = k_new.shape
        if (B, H, d) != (self.B, self.H, self.d):
            raise ValueError("shape mismatch")
        if np.any(self.fill[layer] + T > self.max_len):
            raise OverflowError("append would exceed max_len")
        kq = quantize_rows(k_new, self.dtype, self.k_scale[layer])   # copies: the caller may reuse its buffers
        vq = quantize_rows(v_new, self.dtype, self.v_scale[layer])
        for b in range(B):
            f = int(self.fill[layer, b])
            self.k[layer, b, :, f:f + T] = kq[b]
            self.v[layer, b, :, f:f + T] = vq[b]
        self.fill[layer] += T
        return [(self._read(layer, self.k[layer, b, :, :self.fill[layer, b]], True),
                 self._read(layer, self.v[layer, b, :, :self.fill[layer, b]], False))
                for b in range(B)]

    def _read(self, layer, stored, is_k):
        """Float64 values of stored elements of one layer (times the layer's scale for fp8)."""
        x = stored_to_f64(stored, self.dtype)
        if self.dtype == "e4m3":
            x = x * float(self.k_scale[layer] if is_k else self.v_scale[layer])
        return x

    def commit(self) -> None:
        """Advance every committed length to its fill, once per forward after the last layer."""
        if np.any(self.fill != self.fill[0][None, :]):
            raise RuntimeError("commit with unequal per-layer fills")
        self.lens = self.fill[0].copy()

    def truncate(self, n) -> None:
        """Set every layer's fill and the committed length to n (scalar or per sequence).

        Nothing is freed or zeroed; the next append overwrites from n (§2.4 "Rollback").
        """
        n = np.broadcast_to(np.asarray(n, dtype=np.int64), (self.B,)).copy()
        if np.any(n < 0):
            raise ValueError("negative length")
        if np.any(n > self.lens):
            raise RuntimeError("truncate beyond the committed length")
        self.fill[:, :] = n[None, :]
        self.lens = n

    def set_lengths(self, n) -> None:
        """Set every layer's fill and the committed length to n_b, growing or shrinking, without writing
        a row: positions [0, n_b) then hold whatever the store holds there (zeros never written, rows a
        truncate left behind). Lengths are bookkeeping only (§2.3; §2.4: nothing is copied)."""
        n = np.broadcast_to(np.asarray(n, dtype=np.int64), (self.B,)).copy()
        if np.any(n < 0) or np.any(n > self.max_len):
            raise ValueError("length outside [0, max_len]")
        self.fill[:, :] = n[None, :]
        self.lens = n

    # -- sizes -----------------------------------------------------------------------------
    def nbytes(self) -> int:
        """Capacity: 2 * L * B * H_kv * max_len * d_h * itemsize (§2.5)."""
        return 2 * self.L * self.B * self.H * self.max_len * self.d * ITEMSIZE[self.dtype]

    def filled_bytes(self) -> int:
        """Bytes of the committed part: 2 * L * H_kv * d_h * itemsize * sum_b s_b."""
        return 2 * self.L * self.H * self.d * ITEMSIZE[self.dtype] * int(self.lens.sum())

    def stored_f64(self, layer: int, b: int, kvh: int, n: int):
        """Float64 view of the first n stored rows of one (layer, sequence, K/V head)."""
        return (self._read(layer, self.k[layer, b, kvh, :n], True),
                self._read(layer, self.v[layer, b, kvh, :n], False))


# ----------------------------------------------------------------------------------------------
# The paged cache ("KV cache decoding", "Batching caches of different lengths": the cache kept in
# fixed-size blocks with a table from each request to its blocks, a new block taken only when the
# sequence grows into it and its blocks freed when it ends; "KV cache, incremental decode, ...",
# Key Takeaways and §2.5: a float16 paged cache stores what the contiguous one stores and compares
# with it exactly).
# ----------------------------------------------------------------------------------------------

class OraclePagedKVCache:
    """Block pool (L, n_blocks, H_kv, block, d_h) plus a block table (B, ceil(max_len / block)).

    Position p of sequence b lives at row p % block of physical block table[b, p // block], the same
    block in every layer. Readings where the pages leave the policy open:
    * blocks are handed out lowest-numbered free block first, sequences in order, then logical
      blocks in order, when an append's new fill reaches them;
    * truncate returns every block wholly past the new length; a partly filled block stays;
    * a pool too small for an append raises OverflowError, like the max_len check, changing nothing.
    Lengths, commit and the errors are those of OracleKVCache.
    """

    def __init__(self, n_layers: int, batch: int, n_kv_heads: int, d_head: int, max_len: int,
                 block: int, n_blocks: int, dtype: str = "f32"):
        if dtype not in DTYPES:
            raise ValueError(f"unknown dtype {dtype!r}")
        if min(n_layers, batch, n_kv_heads, d_head, max_len, block, n_blocks) <= 0:
            raise ValueError("all sizes must be positive")
        self.L, self.B, self.H, self.d, self.max_len, self.dtype = (
            n_layers, batch, n_kv_heads, d_head, max_len, dtype)
        self.block, self.n_blocks = block, n_blocks
        self.max_blocks = -(-max_len // block)
        shape = (n_layers, n_blocks, n_kv_heads, block, d_head)
        self.k = np.zeros(shape, dtype=storage_np_dtype(dtype))
        self.v = np.zeros(shape, dtype=storage_np_dtype(dtype))
        self.table = np.full((batch, self.max_blocks), -1, dtype=np.int64)
        self.free = set(range(n_blocks))
        self.fill = np.zeros((n_layers, batch), dtype=np.int64)
        self.lens = np.zeros(batch, dtype=np.int64)
        self.k_scale = np.ones(n_layers, dtype=np.float32)
        self.v_scale = np.ones(n_layers, dtype=np.float32)

    # -- blocks ----------------------------------------------------------------------------
    def held(self, b: int) -> int:
        """Logical blocks sequence b holds (they are always 0 .. held-1)."""
        return int(np.sum(self.table[b] >= 0))

    def blocks_for(self, n: int) -> int:
        return -(-int(n) // self.block)

    def take_block(self) -> int:
        """Remove and return the lowest-numbered free block."""
        blk = min(self.free)
        self.free.remove(blk)
        return blk

    def where(self, b: int, p):
        """(physical block, row) of position(s) p of sequence b."""
        p = np.asarray(p)
        return self.table[b, p // self.block], p % self.block

    # -- lengths (as OracleKVCache) -------------------------------------------------------------
    def seq_len(self, layer: int | None = None) -> np.ndarray:
        if layer is None:
            return self.fill.min(axis=0).copy()
        return self.fill[layer].copy()

    def committed(self) -> np.ndarray:
        return self.lens.copy()

    def positions(self, T: int) -> np.ndarray:
        return self.lens[:, None] + np.arange(T)[None, :]

    # -- writes ----------------------------------------------------------------------------
    def append(self, layer: int, k_new, v_new):
        """Write a [B, H_kv, T, d_h] chunk at each sequence's fill, taking blocks as it grows."""
        if not 0 <= layer < self.L:
            raise ValueError("layer out of range")
        k_new = np.asarray(k_new)
        v_new = np.asarray(v_new)
        if k_new.ndim != 4 or k_new.shape != v_new.shape:
            raise ValueError("k_new and v_new must both be [B, H_kv, T, d_h]")
        B, H, T, d = k_new.shape
        if (B, H, d) != (self.B, self.H, self.d):
            raise ValueError("shape mismatch")
        if np.any(self.fill[layer] + T > self.max_len):
            raise OverflowError("append would exceed max_len")
        need = [max(0, self.blocks_for(self.fill[layer, b] + T) - self.held(b)) for b in range(B)]
        if sum(need) > len(self.free):
            raise OverflowError("block pool exhausted")
        for b in range(B):
            for i in range(self.held(b), self.held(b) + need[b]):
                self.table[b, i] = self.take_block()
        kq = quantize_rows(k_new, self.dtype, self.k_scale[layer])
        vq = quantize_rows(v_new, self.dtype, self.v_scale[layer])
        for b in range(B):
            blk, row = self.where(b, int(self.fill[layer, b]) + np.arange(T))
            self.k[layer, blk, :, row] = kq[b].transpose(1, 0, 2)     # [T, H, d] rows
            self.v[layer, blk, :, row] = vq[b].transpose(1, 0, 2)
        self.fill[layer] += T
        out = []
        for b in range(B):
            n = int(self.fill[layer, b])
            ks = np.stack([self.stored_f64(layer, b, h, n)[0] for h in range(H)])
            vs = np.stack([self.stored_f64(layer, b, h, n)[1] for h in range(H)])
            out.append((ks, vs))
        return out

    def commit(self) -> None:
        if np.any(self.fill != self.fill[0][None, :]):
            raise RuntimeError("commit with unequal per-layer fills")
        self.lens = self.fill[0].copy()

    def truncate(self, n) -> None:
        """Set every fill and committed length to n; blocks wholly past n go back to the pool."""
        n = np.broadcast_to(np.asarray(n, dtype=np.int64), (self.B,)).copy()
        if np.any(n < 0):
            raise ValueError("negative length")
        if np.any(n > self.lens):
            raise RuntimeError("truncate beyond the committed length")
        for b in range(self.B):
            for i in range(self.blocks_for(n[b]), self.max_blocks):
                if self.table[b, i] >= 0:
                    self.free.add(int(self.table[b, i]))
                    self.table[b, i] = -1
        self.fill[:, :] = n[None, :]
        self.lens = n

    # -- sizes and reads -------------------------------------------------------------------
    def nbytes(self) -> int:
        """Pool capacity: 2 * L * n_blocks * H_kv * block * d_h * itemsize."""
        return 2 * self.L * self.n_blocks * self.H * self.block * self.d * ITEMSIZE[self.dtype]

    def stored_f64(self, layer: int, b: int, kvh: int, n: int):
        """Float64 rows 0 .. n-1 of one (layer, sequence, K/V head), gathered through the table."""
        blk, row = self.where(b, np.arange(n))
        return (self._read(layer, self.k[layer, blk, kvh, row], True),
                self._read(layer, self.v[layer, blk, kvh, row], False))

    _read = OracleKVCache._read


# ----------------------------------------------------------------------------------------------
# Rotary positions ("KV cache decoding", "Position information with a cache": the query and the key
# are rotated by an angle that depends on their absolute position, keys are stored already rotated
# and the new query is rotated by its position, so the score depends only on the distance and cached
# keys never change. The pages name RoPE without its formula; this is the published one, Su et al.,
# "RoFormer: Enhanced Transformer with Rotary Position Embedding", eq. 34: pair i of a d-wide vector
# turns by position * theta_i, theta_i = base^(-2i/d).)
# ----------------------------------------------------------------------------------------------

ROPE_STYLES = ("half", "interleaved")


def rope_theta(d: int, base: float) -> np.ndarray:
    """Angular frequency of each of the d/2 pairs: theta_i = base^(-2i/d), i = 0 .. d/2 - 1."""
    return float(base) ** (-2.0 * np.arange(d // 2, dtype=np.float64) / d)


def rope_pairs(d: int, style: str):
    """Element indices (a_i, b_i) of the pairs that rotate together: (i, i + d/2) for "half" (the
    Llama-family layout), (2i, 2i + 1) for "interleaved" (the RoFormer paper's layout)."""
    i = np.arange(d // 2)
    if style == "half":
        return i, i + d // 2
    if style == "interleaved":
        return 2 * i, 2 * i + 1
    raise ValueError(f"unknown RoPE style {style!r}")


def apply_rope(x, positions, base: float, style: str) -> np.ndarray:
    """Rotate the last axis of x [..., n, d] row by row, row j at absolute position positions[j],
    in float64: (x_a, x_b) -> (x_a cos - x_b sin, x_b cos + x_a sin) with angle position * theta_i."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_theta(d, base)[None, :]
    c, sn = np.cos(ang), np.sin(ang)
    a, b = rope_pairs(d, style)
    out = x.copy()
    out[..., a] = x[..., a] * c - x[..., b] * sn
    out[..., b] = x[..., b] * c + x[..., a] * sn
    return out


def rope_chunk(x, starts, base: float, style: str) -> np.ndarray:
    """A [B, H, T, d] chunk whose row t of sequence b sits at absolute position starts[b] + t,
    rotated in float64 and rounded to float32 (what a fused append stores, before the cache dtype;
    what a fused attention uses as its query)."""
    x = np.asarray(x)
    B, H, T, d = x.shape
    out = np.empty(x.shape, dtype=np.float32)
    for b in range(B):
        out[b] = apply_rope(x[b], int(starts[b]) + np.arange(T), base, style).astype(np.float32)
    return out


# ----------------------------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------------------------

def softmax_rows(scores: np.ndarray) -> np.ndarray:
    """Row softmax with the row maximum subtracted first; -inf entries get weight 0."""
    m = np.max(scores, axis=-1, keepdims=True)
    e = np.exp(scores - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_offset: int) -> np.ndarray:
    """One head: softmax(mask(q k^T / sqrt(d))) v with query i at absolute position q_offset + i.

    q [T, d], k and v [N, d] with N = q_offset + T, all float64.
    """
    T, d = q.shape
    N = k.shape[0]
    if N != q_offset + T:
        raise ValueError("key count must equal q_offset + T")
    scores = (q @ k.T) / np.sqrt(d)
    scores = np.where(offset_causal_mask(T, q_offset), scores, -np.inf)
    return softmax_rows(scores) @ v


def query_as_f64(q, dtype: str) -> np.ndarray:
    """A float32 query rounded to the cache dtype (16-bit caches) or to float16 (fp8 caches, whose
    values float16 holds exactly), as float64."""
    q = np.asarray(q)
    if dtype == "e4m3":
        return q.astype(np.float32).astype(np.float16).astype(np.float64)
    if dtype in ("f16", "bf16"):
        return stored_to_f64(store_round(q, dtype), dtype)
    if dtype == "f32":
        return q.astype(np.float32).astype(np.float64)
    return q.astype(np.float64)


def gqa_cached_attention(cache, layer: int, q, T: int | None = None) -> np.ndarray:
    """Attend a chunk's queries over every stored row of one layer (OracleKVCache or OraclePagedKVCache).

    q is [B, H_q, T, d_h]. The layer must already hold the chunk (fill = s_b + T, with s_b the
    committed length). Query head h of sequence b reads K/V head h // G, G = H_q / H_kv, and
    query t sees stored rows j <= s_b + t. Returns [B, H_q, T, d_h] float64.
    """
    q = np.asarray(q)
    B, H_q, Tq, d = q.shape
    T = Tq if T is None else T
    if T != Tq or B != cache.B or d != cache.d or H_q % cache.H:
        raise ValueError("query shape does not match the cache")
    G = H_q // cache.H
    q64 = query_as_f64(q, cache.dtype)
    out = np.zeros((B, H_q, T, d), dtype=np.float64)
    for b in range(B):
        N = int(cache.fill[layer, b])
        s = N - T
        if s != int(cache.lens[b]):
            raise RuntimeError("the layer must hold exactly the committed rows plus this chunk")
        for h in range(H_q):
            k, v = cache.stored_f64(layer, b, h // G, N)
            out[b, h] = attend(q64[b, h], k, v, q_offset=s)
    return out


# ----------------------------------------------------------------------------------------------
# The latent cache ("KV cache, incremental decode, ...", §2.6 "The latent cache": MLA caches one
# compressed latent c in R^r and one shared RoPE key k^R in R^{d_R} per position instead of per-head
# K and V; it follows the same rules (per-layer fill, committed length, rollback) on [B, T, r] and
# [B, T, d_R] chunks, and its nbytes is L B N_max (r + d_R) times the item size).
# ----------------------------------------------------------------------------------------------

class OracleLatentCache:
    """Per layer a latent store C [B, max_len, r] and a RoPE-key store KR [B, max_len, d_R]."""

    def __init__(self, n_layers: int, batch: int, r: int, d_rope: int, max_len: int, dtype: str = "f32"):
        if dtype not in DTYPES or dtype == "e4m3":
            raise ValueError(f"unsupported dtype {dtype!r}")
        if min(n_layers, batch, r, d_rope, max_len) <= 0:
            raise ValueError("all sizes must be positive")
        self.L, self.B, self.r, self.d_rope, self.max_len, self.dtype = n_layers, batch, r, d_rope, max_len, dtype
        self.c = np.zeros((n_layers, batch, max_len, r), dtype=storage_np_dtype(dtype))
        self.kr = np.zeros((n_layers, batch, max_len, d_rope), dtype=storage_np_dtype(dtype))
        self.fill = np.zeros((n_layers, batch), dtype=np.int64)
        self.lens = np.zeros(batch, dtype=np.int64)

    seq_len = OracleKVCache.seq_len
    committed = OracleKVCache.committed
    positions = OracleKVCache.positions
    commit = OracleKVCache.commit
    truncate = OracleKVCache.truncate
    set_lengths = OracleKVCache.set_lengths

    def append(self, layer: int, c_new, kr_new):
        """Write a [B, T, r] latent chunk and a [B, T, d_R] RoPE-key chunk at each sequence's fill;
        return the stored rows (rounded) of every sequence as float64."""
        if not 0 <= layer < self.L:
            raise ValueError("layer out of range")
        c_new, kr_new = np.asarray(c_new), np.asarray(kr_new)
        if c_new.ndim != 3 or kr_new.ndim != 3 or c_new.shape[:2] != kr_new.shape[:2]:
            raise ValueError("c_new [B, T, r] and kr_new [B, T, d_R] expected")
        B, T, r = c_new.shape
        if (B, r, kr_new.shape[2]) != (self.B, self.r, self.d_rope):
            raise ValueError("shape mismatch")
        if np.any(self.fill[layer] + T > self.max_len):
            raise OverflowError("append would exceed max_len")
        cq, kq = store_round(c_new, self.dtype), store_round(kr_new, self.dtype)
        for b in range(B):
            f = int(self.fill[layer, b])
            self.c[layer, b, f:f + T] = cq[b]
            self.kr[layer, b, f:f + T] = kq[b]
        self.fill[layer] += T
        return [self.stored_f64(layer, b, int(self.fill[layer, b])) for b in range(B)]

    def nbytes(self) -> int:
        """L * B * N_max * (r + d_R) * itemsize."""
        return self.L * self.B * self.max_len * (self.r + self.d_rope) * ITEMSIZE[self.dtype]

    def stored_f64(self, layer: int, b: int, n: int):
        return (stored_to_f64(self.c[layer, b, :n], self.dtype), stored_to_f64(self.kr[layer, b, :n], self.dtype))


def mla_cached_attention(cache: OracleLatentCache, layer: int, q_lat, q_rope, scale: float) -> np.ndarray:
    """Multi-head latent attention over the latent cache, in the absorbed form of DeepSeek-V2 (§2.1):
    head h's score for key j is (q_lat_h . c_j + q_rope_h . k^R_j) * scale, with q_lat_h the head's
    no-RoPE query already multiplied by its key up-projection; query t of sequence b sees keys
    j <= s_b + t; the output is the latent sum_j softmax_j c_j [B, H, T, r] (the value up-projection is
    applied after). A query for a 16-bit cache is rounded to the cache dtype first.
    """
    q_lat, q_rope = np.asarray(q_lat), np.asarray(q_rope)
    B, H, T, r = q_lat.shape
    if q_rope.shape != (B, H, T, cache.d_rope) or B != cache.B or r != cache.r:
        raise ValueError("query shapes do not match the cache")
    ql, qr = query_as_f64(q_lat, cache.dtype), query_as_f64(q_rope, cache.dtype)
    out = np.zeros((B, H, T, r), dtype=np.float64)
    for b in range(B):
        N = int(cache.fill[layer, b])
        s = N - T
        if s != int(cache.lens[b]):
            raise RuntimeError("the layer must hold exactly the committed rows plus this chunk")
        c, kr = cache.stored_f64(layer, b, N)
        for h in range(H):
            scores = (ql[b, h] @ c.T + qr[b, h] @ kr.T) * scale
            scores = np.where(offset_causal_mask(T, s), scores, -np.inf)
            out[b, h] = softmax_rows(scores) @ c
    return out


def full_recompute_attention(q_all: np.ndarray, k_all: np.ndarray, v_all: np.ndarray) -> np.ndarray:
    """Uncached path: causal attention of every position of a whole sequence, q_offset = 0.

    q_all [H_q, n, d], k_all and v_all [H_kv, n, d] (float64, already as stored). Query head h
    uses K/V head h // G. Returns [H_q, n, d].
    """
    H_q, n, d = q_all.shape
    G = H_q // k_all.shape[0]
    return np.stack([attend(q_all[h], k_all[h // G], v_all[h // G], q_offset=0) for h in range(H_q)])
