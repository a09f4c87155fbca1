"""Plant the pages' pitfalls in the oracle (on the CPU) and check that the pins catch each one.

"KV cache, incremental decode, ...", §5 "Pitfalls" lists the mistakes; each mutant below is one
of them, patched into a copy of the oracle's behaviour for the duration of one test.
"""
import numpy as np
import pytest

import oracle.kvc_oracle as ko
from tests import test_oracle_pins as pins


def _fails(test, *args):
    with pytest.raises(AssertionError):
        test(*args)


def test_mask_without_offset_is_caught(monkeypatch):
    """Pitfall 3: a decode mask without the offset."""
    orig = ko.attend

    def attend_no_offset(q, k, v, q_offset):
        T, d = q.shape
        scores = (q @ k.T) / np.sqrt(d)
        mask = np.zeros((T, k.shape[0]), bool)
        mask[:, :T] = np.tril(np.ones((T, T), bool))
        return ko.softmax_rows(np.where(mask, scores, -np.inf)) @ v

    monkeypatch.setattr(ko, "attend", attend_no_offset)
    _fails(pins.test_cached_equals_full_recompute_every_step)
    monkeypatch.setattr(ko, "attend", orig)


def test_wrong_gqa_mapping_is_caught(monkeypatch):
    """K/V head h % H_kv instead of h // G."""
    def gqa_mod(cache, layer, q, T=None):
        B, Hq, T, d = q.shape
        out = np.zeros((B, Hq, T, d))
        for b in range(B):
            N = int(cache.fill[layer, b])
            for h in range(Hq):
                k, v = cache.stored_f64(layer, b, h % cache.H, N)
                out[b, h] = ko.attend(ko.query_as_f64(q[b, h], cache.dtype), k, v, N - T)
        return out

    monkeypatch.setattr(pins, "gqa_cached_attention", gqa_mod)
    _fails(pins.test_gqa_head_mapping_is_contiguous_groups)


def test_update_returning_only_the_new_chunk_is_caught(monkeypatch):
    """Pitfall 4."""
    orig = ko.OracleKVCache.append

    def append_new_only(self, layer, k_new, v_new):
        T = np.asarray(k_new).shape[2]
        rows = orig(self, layer, k_new, v_new)
        return [(k[:, -T:], v[:, -T:]) for k, v in rows]

    monkeypatch.setattr(ko.OracleKVCache, "append", append_new_only)
    _fails(pins.test_hand_example)


def test_truncating_one_layer_only_is_caught(monkeypatch):
    """Pitfall 6."""
    def truncate_first_layer(self, n):
        n = np.broadcast_to(np.asarray(n, dtype=np.int64), (self.B,)).copy()
        self.fill[0, :] = n
        self.lens = n

    monkeypatch.setattr(ko.OracleKVCache, "truncate", truncate_first_layer)
    with pytest.raises((AssertionError, RuntimeError)):
        pins.test_truncate_then_reappend_same_rows_restores_whole_buffer()


def test_float16_cache_returning_the_raw_chunk_is_caught(monkeypatch):
    """Pitfall 8."""
    orig = ko.OracleKVCache.append

    def append_raw(self, layer, k_new, v_new):
        rows = orig(self, layer, k_new, v_new)
        T = np.asarray(k_new).shape[2]
        out = []
        for b, (k, v) in enumerate(rows):
            k = k.copy()
            v = v.copy()
            k[:, -T:] = np.asarray(k_new)[b]
            v[:, -T:] = np.asarray(v_new)[b]
            out.append((k, v))
        return out

    monkeypatch.setattr(ko.OracleKVCache, "append", append_raw)
    _fails(pins.test_float16_cache_rounds_what_it_stores)


def test_dropped_scale_is_caught(monkeypatch):
    """Scores without the 1 / sqrt(d_h) factor."""
    def attend_unscaled(q, k, v, q_offset):
        T = q.shape[0]
        scores = q @ k.T
        return ko.softmax_rows(np.where(ko.offset_causal_mask(T, q_offset), scores, -np.inf)) @ v

    monkeypatch.setattr(pins, "attend", attend_unscaled)
    _fails(pins.test_hand_softmax)


def test_bf16_truncation_instead_of_rounding_is_caught(monkeypatch):
    orig = ko.store_round

    def truncating(x, dtype):
        if dtype == "bf16":
            return (np.asarray(x, np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
        return orig(x, dtype)

    monkeypatch.setattr(pins, "store_round", truncating)
    _fails(pins.test_storage_rounding_golden, "bf16")


# ---- the paged oracle ("KV cache decoding", "Batching caches of different lengths") ------------------
from tests import test_oracle_paged as paged_pins


def test_paged_rows_reversed_within_a_block_are_caught(monkeypatch):
    """Rows stored from the end of each block: reads stay consistent, the layout does not."""
    def where_reversed(self, b, p):
        p = np.asarray(p)
        return self.table[b, p // self.block], self.block - 1 - p % self.block

    monkeypatch.setattr(ko.OraclePagedKVCache, "where", where_reversed)
    _fails(paged_pins.test_paged_hand_example)


def test_paged_truncate_that_frees_nothing_is_caught(monkeypatch):
    """Blocks kept past the new length: the memory paging should recover stays taken."""
    def truncate_keep_blocks(self, n):
        n = np.broadcast_to(np.asarray(n, dtype=np.int64), (self.B,)).copy()
        self.fill[:, :] = n[None, :]
        self.lens = n

    monkeypatch.setattr(ko.OraclePagedKVCache, "truncate", truncate_keep_blocks)
    _fails(paged_pins.test_paged_holds_exactly_the_blocks_its_rows_reach, 4)


def test_paged_highest_block_first_is_caught(monkeypatch):
    """A different allocation order than the stated lowest-free-first reading."""
    def take_highest(self):
        blk = max(self.free)
        self.free.remove(blk)
        return blk

    monkeypatch.setattr(ko.OraclePagedKVCache, "take_block", take_highest)
    _fails(paged_pins.test_paged_allocation_order_by_hand)


# ---- rotary positions ("KV cache decoding", "Position information with a cache") ---------------------
from tests import test_oracle_rope as rope_pins


def test_rope_at_position_zero_is_caught(monkeypatch):
    """The pages' classic bug: the new token rotated as if it sat at position 0."""
    orig = ko.rope_chunk

    def rope_from_zero(x, starts, base, style):
        return orig(x, [0] * len(starts), base, style)

    monkeypatch.setattr(rope_pins, "rope_chunk", rope_from_zero)
    _fails(rope_pins.test_rope_chunk_positions_follow_each_sequence)


def test_rope_turning_the_wrong_way_is_caught(monkeypatch):
    orig = ko.apply_rope

    def backwards(x, positions, base, style):
        return orig(x, -np.asarray(positions, dtype=np.float64), base, style)

    monkeypatch.setattr(rope_pins, "apply_rope", backwards)
    _fails(rope_pins.test_two_dims_turn_by_the_position_in_radians, "half")


def test_rope_frequency_off_by_two_is_caught(monkeypatch):
    """theta_i = base^(-i/d) instead of base^(-2i/d)."""
    monkeypatch.setattr(ko, "rope_theta", lambda d, base: float(base) ** (-np.arange(d // 2) / d))
    _fails(rope_pins.test_pair_frequencies_form_a_geometric_series, "half")


# ---- fp8 storage (E4M3 with per-layer scales) ---------------------------------------------------------
from tests import test_oracle_fp8 as fp8_pins


def test_e4m3_truncating_instead_of_rounding_is_caught(monkeypatch):
    def truncating(x):
        x = np.asarray(x, dtype=np.float32).astype(np.float64)
        a = np.abs(x)
        _, ex = np.frexp(a)
        q = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
        return ko.e4m3_encode((np.sign(x) * np.minimum(np.floor(a / q) * q, 448.0)).astype(np.float32))

    monkeypatch.setattr(fp8_pins, "e4m3_encode", truncating)
    _fails(fp8_pins.test_encode_matches_torch_in_range, 1.0)


def test_e4m3_without_saturation_is_caught(monkeypatch):
    orig = ko.e4m3_encode

    def wrapping(x):
        x = np.asarray(x, dtype=np.float32)
        out = orig(x)
        return np.where(np.abs(x) > 448, np.uint8(0x7F) | (out & 0x80), out).astype(np.uint8)   # NaN code

    monkeypatch.setattr(fp8_pins, "e4m3_encode", wrapping)
    _fails(fp8_pins.test_hand_worked_codes)


def test_fp8_scale_multiplied_instead_of_divided_is_caught(monkeypatch):
    orig = ko.quantize_rows

    def multiplied(x, dtype, scale):
        if dtype == "e4m3":
            return ko.store_round(np.asarray(x, dtype=np.float32) * np.float32(scale), dtype)
        return orig(x, dtype, scale)

    monkeypatch.setattr(ko, "quantize_rows", multiplied)
    _fails(fp8_pins.test_fp8_cache_stores_codes_of_x_over_scale, ko.OracleKVCache)


# ---- the latent cache and multi-head latent attention ------------------------------------------------
from tests import test_oracle_latent as latent_pins


def test_mla_without_the_rope_key_term_is_caught(monkeypatch):
    """Scores from the latent alone, dropping q_rope . k^R."""
    def mla_no_rope(cache, layer, q_lat, q_rope, scale):
        return ko.mla_cached_attention(cache, layer, q_lat, np.zeros_like(np.asarray(q_rope)), scale)

    monkeypatch.setattr(latent_pins, "mla_cached_attention", mla_no_rope)
    _fails(latent_pins.test_absorbed_mla_equals_explicit_per_head_projections, 1, [7, 0, 12])


def test_set_lengths_moving_only_the_committed_length_is_caught(monkeypatch):
    """set_lengths that leaves the per-layer fills where they were: the next append writes at the old
    fill, not at the new length."""
    def set_lengths_committed_only(self, n):
        self.lens = np.broadcast_to(np.asarray(n, dtype=np.int64), (self.B,)).copy()

    monkeypatch.setattr(ko.OracleKVCache, "set_lengths", set_lengths_committed_only)
    _fails(pins.test_set_lengths_over_zero_rows_matches_the_closed_form)


def test_set_lengths_that_zeroes_the_rows_it_uncovers_is_caught(monkeypatch):
    """set_lengths that clears the rows it declares filled (as if they were new) loses what a truncate
    left behind."""
    orig = ko.OracleKVCache.set_lengths

    def set_lengths_zeroing(self, n):
        old = self.lens.copy()
        orig(self, n)
        for b in range(self.B):
            self.k[:, b, :, old[b]:self.lens[b]] = 0
            self.v[:, b, :, old[b]:self.lens[b]] = 0

    monkeypatch.setattr(ko.OracleKVCache, "set_lengths", set_lengths_zeroing)
    _fails(pins.test_set_lengths_after_truncate_restores_the_rows_left_behind)
