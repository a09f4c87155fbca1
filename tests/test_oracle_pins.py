"""Pins for the CPU oracle: values the pages print, closed forms, identities and brute force.

Each test ties one oracle function to something other than the oracle itself, chosen so that a
plausible mistake (a dropped term, a wrong sign or index, a transposed operand, a wrong offset)
fails at least one of them. `test_oracle_mutants.py` plants such mistakes and checks they fail.
"""
import math

import numpy as np
import pytest

import kvc_synth
from oracle.kvc_oracle import (OracleKVCache, attend, full_recompute_attention, gqa_cached_attention,
                               kv_bytes, offset_causal_mask, store_round, stored_to_f64)
from oracle.tiny_decoder import DecoderShape, build_tiny_decoder, greedy
from tests.conftest import golden


# -- the hand example ("KV cache, incremental decode, ...", §3) --------------------------------

def test_hand_example():
    g = golden("hand_example.json")
    c = g["cache"]
    cache = OracleKVCache(c["n_layers"], c["batch"], c["n_kv_heads"], c["d_head"], c["max_len"], c["dtype"])
    k = np.array(g["prefill_keys"], np.float32)[None, None]
    (kk, _), = cache.append(0, k, k)
    assert cache.seq_len(0)[0] == g["after_prefill"]["fill"]
    np.testing.assert_array_equal(kk[0], g["after_prefill"]["returned_rows"])
    cache.commit()
    assert cache.seq_len()[0] == g["after_prefill"]["s"] == cache.committed()[0]
    assert cache.positions(1)[0, 0] == g["after_prefill"]["next_position"]
    k2 = np.array(g["decode_key"], np.float32)[None, None, None]
    (kk, _), = cache.append(0, k2, k2)
    np.testing.assert_array_equal(kk[0], g["after_decode"]["returned_rows"])
    cache.commit()
    assert cache.committed()[0] == g["after_decode"]["s"]
    assert cache.positions(1)[0, 0] == g["next_query_position"]
    np.testing.assert_array_equal(cache.mask(1)[0].astype(int), g["next_query_mask_row"])
    assert cache.nbytes() == g["storage_bytes"]


# -- memory formulas -----------------------------------------------------------------------------

def test_memory_formulas():
    g = golden("memory_formulas.json")
    for case in g["cases"]:
        n = kv_bytes(case["layers"], case["heads"], case["head_dim"], case["seq_len"], case["batch"],
                     case["bytes_per_value"])
        assert n == case["bytes"], case["citation"]
        if "elements" in case:
            assert n // case["bytes_per_value"] == case["elements"]
    for case in g["approximate"]:
        n = kv_bytes(case["layers"], case["heads"], case["head_dim"], case["seq_len"], case["batch"],
                     case["bytes_per_value"])
        assert abs(n - case["about_bytes"]) <= case["rel_tol"] * case["about_bytes"], case["citation"]


def test_nbytes_is_capacity_and_halves_in_float16():
    g = golden("memory_formulas.json")["cases"][0]
    full = OracleKVCache(g["layers"], g["batch"], g["heads"], g["head_dim"], g["seq_len"], "f32")
    assert full.nbytes() == g["bytes"]                       # capacity: max_len = 128 positions
    assert full.k.nbytes + full.v.nbytes == full.nbytes()
    half = OracleKVCache(g["layers"], g["batch"], g["heads"], g["head_dim"], g["seq_len"], "f16")
    assert half.nbytes() * 2 == full.nbytes()
    f64 = OracleKVCache(g["layers"], g["batch"], g["heads"], g["head_dim"], g["seq_len"], "f64")
    assert f64.nbytes() == golden("memory_formulas.json")["cases"][1]["bytes"]


# -- the mask ------------------------------------------------------------------------------------

def test_mask_brute_force_small():
    """Every T <= 4, s <= 5 against the §2.3 predicate evaluated element by element."""
    for T in range(0, 5):
        for s in range(0, 6):
            m = offset_causal_mask(T, s)
            assert m.shape == (T, s + T)
            for i in range(T):
                for j in range(s + T):
                    assert m[i, j] == (j <= s + i)


def test_mask_special_cases_and_counts():
    # s = 0 is the usual lower triangle; T = 1 is one row of all True ("KV cache decoding", step 3)
    for T in range(1, 9):
        np.testing.assert_array_equal(offset_causal_mask(T, 0), np.tril(np.ones((T, T), bool)))
    for s in range(0, 40):
        assert offset_causal_mask(1, s).all()
    # the same mask as a lower triangle shifted right by s (the diagonal moves by the cache length)
    for T in range(1, 7):
        for s in range(0, 9):
            np.testing.assert_array_equal(offset_causal_mask(T, s), np.tril(np.ones((T, s + T), bool), k=s))
            # closed form: row i sees s + i + 1 keys; T s + T (T + 1) / 2 in all
            assert offset_causal_mask(T, s).sum() == T * s + T * (T + 1) // 2
    # without the offset a decode query would see only key 0 (§2.3, last sentence)
    assert offset_causal_mask(1, 0).sum() == 1 and offset_causal_mask(1, 7).sum() == 8


# -- storage rounding ----------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_storage_rounding_golden(dtype):
    for e in golden("storage_rounding.json")[dtype]:
        x = np.array([int(e["f32_bits"], 16)], np.uint32).view(np.float32)
        with np.errstate(over="ignore"):
            got = store_round(x, dtype).view(np.uint16)[0]
        assert int(got) == int(e["stored"], 16), e["note"]


def test_bf16_rounding_matches_torch_on_random_values():
    torch = pytest.importorskip("torch")
    x = kvc_synth.normal_f32((200000,), 3, 11) * np.float32(7.3)
    ours = store_round(x, "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(stored_to_f64(ours, "bf16"), torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_float16_cache_rounds_what_it_stores():
    """Past and new chunk both come back rounded ("KV cache, incremental decode, ...", §2.5)."""
    x1 = kvc_synth.normal_f32((1, 2, 5, 8), 0, 21)
    x2 = kvc_synth.normal_f32((1, 2, 1, 8), 0, 22)
    for dtype in ("f16", "bf16"):
        cache = OracleKVCache(1, 1, 2, 8, 16, dtype)
        cache.append(0, x1, x1)
        cache.commit()
        (k, v), = cache.append(0, x2, x2)
        both = np.concatenate([x1, x2], axis=2)[0]
        if dtype == "f16":
            expect = both.astype(np.float16).astype(np.float64)
        else:
            torch = pytest.importorskip("torch")
            expect = torch.from_numpy(np.ascontiguousarray(both)).to(torch.bfloat16).double().numpy()
        np.testing.assert_array_equal(k, expect)
        np.testing.assert_array_equal(v, expect)
        assert not np.array_equal(k, both.astype(np.float64))      # rounding really happened


# -- attention identities --------------------------------------------------------------------------

def test_hand_softmax():
    g = golden("hand_softmax.json")
    k = np.array(g["keys"], float)
    v = np.array(g["values"], float)
    q1 = np.array([math.sqrt(2) * math.log(2), 0.0])
    np.testing.assert_allclose(attend(q1[None], k, v, q_offset=1)[0], g["expected"]["decode_s1_T1"], atol=1e-14)
    out = attend(np.stack([np.array([5.0, -3.0]), q1]), k, v, q_offset=0)
    np.testing.assert_allclose(out[0], g["expected"]["chunk_s0_T2_row0"], atol=0)
    np.testing.assert_allclose(out[1], g["expected"]["chunk_s0_T2_row1"], atol=1e-14)


def test_single_key_returns_its_value_and_equal_scores_average():
    rng = np.random.default_rng(0)
    for d in (2, 8, 32):
        v = rng.standard_normal((1, d))
        np.testing.assert_array_equal(attend(rng.standard_normal((1, d)), rng.standard_normal((1, d)), v, 0), v)
        # a zero query gives equal scores, so each row averages the values it can see
        k = rng.standard_normal((6, d))
        vv = rng.standard_normal((6, d))
        out = attend(np.zeros((3, d)), k, vv, q_offset=3)
        for i in range(3):
            np.testing.assert_allclose(out[i], vv[:3 + i + 1].mean(axis=0), atol=1e-14)


def test_softmax_is_shift_invariant_and_scaled_by_sqrt_d():
    """Scores are q.k / sqrt(d): scaling q by sqrt(d) / sqrt(d') is the same as using d' instead."""
    rng = np.random.default_rng(1)
    d = 16
    q, k, v = rng.standard_normal((1, d)), rng.standard_normal((5, d)), rng.standard_normal((5, d))
    s = (q @ k.T)[0] / math.sqrt(d)
    w = np.exp(s - s.max())
    w /= w.sum()
    np.testing.assert_allclose(attend(q, k, v, 4)[0], w @ v, atol=1e-14)


def test_gqa_head_mapping_is_contiguous_groups():
    """4 query heads on 2 K/V heads use K/V heads [0, 0, 1, 1] ("Heads, GQA and K/V cache")."""
    cache = OracleKVCache(1, 1, 2, 4, 4, "f64")
    vals = np.array([[[[1.0, 1, 1, 1]], [[2.0, 2, 2, 2]]]])        # one key per K/V head
    cache.append(0, vals, vals)                                    # the chunk is the only row
    q = np.random.default_rng(2).standard_normal((1, 4, 1, 4))
    out = gqa_cached_attention(cache, 0, q)
    np.testing.assert_array_equal(out[0, :, 0, 0], [1.0, 1.0, 2.0, 2.0])


# -- the cache's behaviour --------------------------------------------------------------------------

def _toy_run(dtype="f32", store="f32"):
    """Toy GQA workload: prefill T=48, then 20 decode steps; cached and full-recompute outputs."""
    w = kvc_synth.WORKLOADS["toy-gqa-fp32"]
    L, B, Hq, Hkv, d, n_max = w["L"], w["B"], w["H_q"], w["H_kv"], w["d_h"], w["max_len"]
    n = w["prefill"] + w["decode_steps"]
    q = kvc_synth.normal_f32((L, B, Hq, n, d), w["seed"], kvc_synth.STREAM_Q)
    k = kvc_synth.normal_f32((L, B, Hkv, n, d), w["seed"], kvc_synth.STREAM_K_PREFILL)
    v = kvc_synth.normal_f32((L, B, Hkv, n, d), w["seed"], kvc_synth.STREAM_V_PREFILL)
    cache = OracleKVCache(L, B, Hkv, d, n_max, store)
    chunks = [(0, w["prefill"])] + [(w["prefill"] + i, 1) for i in range(w["decode_steps"])]
    cached = np.zeros((L, B, Hq, n, d))
    for s, T in chunks:
        for layer in range(L):
            cache.append(layer, k[layer, :, :, s:s + T], v[layer, :, :, s:s + T])
            cached[layer, :, :, s:s + T] = gqa_cached_attention(cache, layer, q[layer, :, :, s:s + T])
        cache.commit()
    full = np.zeros_like(cached)
    for layer in range(L):
        for b in range(B):
            kk = stored_to_f64(store_round(k[layer, b], store), store)
            vv = stored_to_f64(store_round(v[layer, b], store), store)
            full[layer, b] = full_recompute_attention(q[layer, b].astype(np.float64), kk, vv)
    return cache, cached, full


def test_cached_equals_full_recompute_every_step():
    """Within 1e-5 at every step ("KV cache, incremental decode, ...", key takeaways); float64
    arithmetic over the same stored values agrees far closer ("KV cache decoding", ~1e-15)."""
    cache, cached, full = _toy_run()
    assert np.abs(cached - full).max() < 1e-12
    assert np.abs(cached.astype(np.float32) - full).max() < 1e-5
    assert cache.committed()[0] == 68


def test_chunked_prefill_equals_whole():
    """Chunks of 3, 1, 5, 2 positions equal one forward (§4 test_chunked_prefill_equals_whole)."""
    d, Hq, Hkv = 8, 4, 2
    q = kvc_synth.normal_f32((1, Hq, 11, d), 5, 1)
    k = kvc_synth.normal_f32((1, Hkv, 11, d), 5, 2)
    v = kvc_synth.normal_f32((1, Hkv, 11, d), 5, 3)
    whole = OracleKVCache(1, 1, Hkv, d, 16, "f32")
    whole.append(0, k, v)
    out_whole = gqa_cached_attention(whole, 0, q)
    parts = OracleKVCache(1, 1, Hkv, d, 16, "f32")
    s = 0
    outs = []
    for T in (3, 1, 5, 2):
        parts.append(0, k[:, :, s:s + T], v[:, :, s:s + T])
        outs.append(gqa_cached_attention(parts, 0, q[:, :, s:s + T]))
        parts.commit()
        s += T
    np.testing.assert_array_equal(parts.k, whole.k)
    np.testing.assert_allclose(np.concatenate(outs, axis=2), out_whole, atol=1e-12)


def test_page_fence3_toy_cache_equals_recompute():
    """The worked fence of "Generation and the KV Cache": torch.manual_seed(35), d = 8, T = 6,
    prefill 2 then one token at a time, equal to one-shot attention within 1e-5."""
    torch = pytest.importorskip("torch")
    torch.manual_seed(35)
    d, T = 8, 6
    Wq, Wk, Wv = (torch.randn(d, d) / math.sqrt(d) for _ in range(3))
    x = torch.randn(T, d).double().numpy()
    Wq, Wk, Wv = (w.double().numpy() for w in (Wq, Wk, Wv))
    full = attend(x @ Wq, x @ Wk, x @ Wv, q_offset=0)
    cache = OracleKVCache(1, 1, 1, d, T, "f64")
    outs = []
    for lo, hi in ((0, 2), (2, 3), (3, 4), (4, 5), (5, 6)):
        cache.append(0, (x[lo:hi] @ Wk)[None, None], (x[lo:hi] @ Wv)[None, None])
        outs.append(gqa_cached_attention(cache, 0, (x[lo:hi] @ Wq)[None, None])[0, 0])
        cache.commit()
    assert np.abs(np.concatenate(outs) - full).max() < 1e-5


def test_update_copies_and_checks():
    """Inputs copied, shapes and capacity checked, nothing changed on error (§4)."""
    cache = OracleKVCache(2, 2, 2, 4, 6, "f32")
    x = kvc_synth.normal_f32((2, 2, 4, 4), 0, 9)
    cache.append(0, x, x)
    before = (cache.k.copy(), cache.v.copy(), cache.fill.copy(), cache.lens.copy())
    x[:] = 123.0                                                # caller reuses its buffer
    np.testing.assert_array_equal(cache.k, before[0])
    for bad in (np.zeros((2, 2, 3, 5), np.float32), np.zeros((1, 2, 1, 4), np.float32),
                np.zeros((2, 3, 1, 4), np.float32)):
        with pytest.raises(ValueError):
            cache.append(1, bad, bad)
    with pytest.raises(OverflowError):
        cache.append(0, np.zeros((2, 2, 3, 4), np.float32), np.zeros((2, 2, 3, 4), np.float32))
    with pytest.raises(ValueError):
        cache.append(2, x, x)
    with pytest.raises(RuntimeError):
        cache.commit()                                          # layer 1 has not been appended
    with pytest.raises(RuntimeError):
        cache.truncate(1)                                       # nothing committed yet
    for a, b in zip(before, (cache.k, cache.v, cache.fill, cache.lens)):
        np.testing.assert_array_equal(a, b)


def test_seq_len_moves_only_after_the_last_layer():
    cache = OracleKVCache(3, 1, 1, 2, 8, "f32")
    x = np.ones((1, 1, 2, 2), np.float32)
    for layer in range(3):
        assert cache.seq_len()[0] == 0
        cache.append(layer, x, x)
        assert cache.seq_len(layer)[0] == 2
    assert cache.seq_len()[0] == 2
    cache.commit()
    assert cache.committed()[0] == 2
    # every layer placed the chunk at the same positions
    for layer in range(3):
        np.testing.assert_array_equal(cache.k[layer, 0, 0, :2], 1.0)


def test_truncate_rolls_back_on_every_layer():
    """truncate then append equals never having appended (§4 test_truncate_rolls_back)."""
    L, B, H, d = 3, 2, 2, 4
    base = kvc_synth.normal_f32((B, H, 5, d), 1, 1)
    draft = kvc_synth.normal_f32((B, H, 4, d), 1, 2)
    final = kvc_synth.normal_f32((B, H, 2, d), 1, 3)
    a = OracleKVCache(L, B, H, d, 16, "f16")
    b = OracleKVCache(L, B, H, d, 16, "f16")
    for c in (a, b):
        for layer in range(L):
            c.append(layer, base, base)
        c.commit()
    for layer in range(L):
        a.append(layer, draft, draft)
    a.commit()
    a.truncate(5)
    for c in (a, b):
        for layer in range(L):
            c.append(layer, final, final)
        c.commit()
    np.testing.assert_array_equal(a.k[:, :, :, :7], b.k[:, :, :, :7])
    np.testing.assert_array_equal(a.fill, b.fill)
    q = kvc_synth.normal_f32((B, 4, 1, d), 1, 4)
    for c in (a, b):
        for layer in range(L):
            c.append(layer, final[:, :, :1], final[:, :, :1])
    for layer in range(L):
        np.testing.assert_array_equal(gqa_cached_attention(a, layer, q), gqa_cached_attention(b, layer, q))


def test_truncate_then_reappend_same_rows_restores_whole_buffer():
    """Speculative verify: keep 3 of 8 drafts, re-append the same 5, get the pre-truncate store."""
    B, H, d = 2, 2, 8
    base = kvc_synth.normal_f32((B, H, 6, d), 2, 1)
    drafts = kvc_synth.normal_f32((B, H, 8, d), 2, 2)
    c = OracleKVCache(2, B, H, d, 20, "bf16")
    for layer in range(2):
        c.append(layer, base, base)
    c.commit()
    for layer in range(2):
        c.append(layer, drafts, drafts)
    c.commit()
    before = (c.k.copy(), c.v.copy())
    c.truncate(6 + 3)
    for layer in range(2):
        c.append(layer, drafts[:, :, 3:], drafts[:, :, 3:])
    c.commit()
    np.testing.assert_array_equal(c.k, before[0])
    np.testing.assert_array_equal(c.v, before[1])
    assert (c.committed() == 14).all()


def test_set_lengths_over_zero_rows_matches_the_closed_form():
    """A fresh cache's unfilled slots are zero ("KV cache decoding", KVCache listing). Declaring n_b of
    them filled, then appending one row (k, v), gives a query scores 0 for the n_b zero keys and
    s = q.k / sqrt(d) for its own: the output is e^s / (n_b + e^s) * v."""
    B, d = 3, 4
    c = OracleKVCache(2, B, 1, d, 16, "f64")
    c.set_lengths([3, 0, 5])
    np.testing.assert_array_equal(c.committed(), [3, 0, 5])
    np.testing.assert_array_equal(c.seq_len(1), [3, 0, 5])
    np.testing.assert_array_equal(c.positions(2), [[3, 4], [0, 1], [5, 6]])
    k = np.arange(B * d, dtype=np.float64).reshape(B, 1, 1, d) / 10
    v = np.arange(B * d, dtype=np.float64).reshape(B, 1, 1, d) - 5
    c.append(0, k, v)
    assert c.k[0, 0, 0, 3].tolist() == k[0, 0, 0].tolist() and c.k[0, 2, 0, 5].tolist() == k[2, 0, 0].tolist()
    q = np.ones((B, 1, 1, d))
    out = gqa_cached_attention(c, 0, q)
    for b, n in enumerate([3, 0, 5]):
        e = math.exp(float(q[b, 0, 0] @ k[b, 0, 0]) / math.sqrt(d))
        np.testing.assert_allclose(out[b, 0, 0], e / (n + e) * v[b, 0, 0], rtol=1e-13)


def test_set_lengths_after_truncate_restores_the_rows_left_behind():
    """Truncate clears nothing (§2.4), so moving the lengths back over the same rows makes the cache
    answer as if it had never been truncated."""
    B, H, d = 2, 2, 8
    past = kvc_synth.normal_f32((B, H, 9, d), 4, 1)
    new = kvc_synth.normal_f32((B, H, 1, d), 4, 2)
    q = kvc_synth.normal_f32((B, 4, 1, d), 4, 3)
    kept, moved = OracleKVCache(1, B, H, d, 12, "f16"), OracleKVCache(1, B, H, d, 12, "f16")
    for c in (kept, moved):
        c.append(0, past, past)
        c.commit()
    kept.truncate([9, 6])
    moved.truncate([2, 0])
    moved.set_lengths([9, 6])
    for c in (kept, moved):
        c.append(0, new, new)
    np.testing.assert_array_equal(gqa_cached_attention(moved, 0, q), gqa_cached_attention(kept, 0, q))
    np.testing.assert_array_equal(moved.k, kept.k)


def test_set_lengths_rejects_out_of_range_and_changes_nothing():
    c = OracleKVCache(2, 2, 1, 4, 8, "bf16")
    c.set_lengths([4, 2])
    for bad in ([9, 0], [-1, 3]):
        with pytest.raises(ValueError):
            c.set_lengths(bad)
        np.testing.assert_array_equal(c.committed(), [4, 2])
        np.testing.assert_array_equal(c.seq_len(0), [4, 2])
    c.set_lengths([8, 0])                                       # both ends of the range are allowed
    np.testing.assert_array_equal(c.seq_len(1), [8, 0])


def test_ragged_lengths_each_sequence_writes_at_its_own_position():
    c = OracleKVCache(1, 3, 1, 2, 10, "f32")
    c.append(0, np.ones((3, 1, 6, 2), np.float32), np.ones((3, 1, 6, 2), np.float32))
    c.commit()
    c.truncate([2, 6, 0])
    new = np.arange(3 * 2, dtype=np.float32).reshape(3, 1, 1, 2) + 10
    c.append(0, new, new)
    c.commit()
    np.testing.assert_array_equal(c.committed(), [3, 7, 1])
    np.testing.assert_array_equal(c.k[0, 0, 0, 2], [10, 11])
    np.testing.assert_array_equal(c.k[0, 1, 0, 6], [12, 13])
    np.testing.assert_array_equal(c.k[0, 2, 0, 0], [14, 15])
    np.testing.assert_array_equal(c.positions(2), [[3, 4], [7, 8], [1, 2]])


# -- the tiny decoder ("KV cache decoding": "Correctness tests", "Prefill and decode") ---------------

@pytest.fixture(scope="module")
def tiny_runs():
    """The page's experiment: a 48-id prompt, 160 greedy ids, without and then with the cache."""
    g = golden("work_counters.json")
    model = build_tiny_decoder(DecoderShape(**g["model"]))
    prompt = kvc_synth.prompt_ids(g["P"], g["model"]["vocab"], 1)
    runs = {}
    for use_cache in (False, True):
        model.tally.positions = model.tally.scores = 0
        seq, logits, cache = greedy(model, prompt, g["N"], use_cache)
        runs[use_cache] = dict(seq=seq, logits=logits, cache=cache,
                               positions=model.tally.positions, scores=model.tally.scores)
    return g, model, prompt, runs


def test_tiny_decoder_equality_and_counters(tiny_runs):
    g, model, prompt, runs = tiny_runs
    plain, cached = runs[False], runs[True]
    assert plain["seq"] == cached["seq"]
    assert np.abs(plain["logits"] - cached["logits"]).max() < g["gap_bound"]
    assert np.ptp(plain["logits"]) > 1.0                      # the logits are not all near zero
    # the page's printed counts for this run
    assert (plain["scores"], cached["scores"]) == (g["scores_uncached"], g["scores_cached"])
    assert (plain["positions"], cached["positions"]) == (g["positions_uncached"], g["positions_cached"])
    # and the closed forms behind them, for the page's larger example too
    P, N = g["large"]["P"], g["large"]["N"]
    assert N * P + N * (N - 1) // 2 == g["large"]["positions_uncached"]
    assert P + N - 1 == g["large"]["positions_cached"]


def test_tiny_decoder_cache_state(tiny_runs):
    g, model, prompt, runs = tiny_runs
    cache, s = runs[True]["cache"], model.shape
    assert cache.k.shape == (s.n_layers, 1, s.n_heads, s.max_len, s.d_head)
    filled = int(cache.committed()[0])
    assert filled == g["P"] + g["N"] - 1                      # the id picked last was never run
    assert cache.filled_bytes() == kv_bytes(s.n_layers, s.n_heads, s.d_head, filled, bytes_per_value=8)
    assert not cache.k[:, :, :, filled:].any() and not cache.v[:, :, :, filled:].any()


def test_tiny_decoder_rows_of_a_prefix_ignore_later_tokens(tiny_runs):
    """A position's stored key and value are the same whether 0 or 20 tokens follow it
    ("Why the causal mask makes caching exact")."""
    g, model, prompt, runs = tiny_runs
    P, seq = g["P"], runs[False]["seq"]
    stores = []
    for extra in (0, 20):
        cache = model.new_cache()
        model(seq[:P + extra], cache)
        stores.append(cache)
    for a, b in ((stores[0].k, stores[1].k), (stores[0].v, stores[1].v)):
        assert np.abs(a[..., :P, :] - b[..., :P, :]).max() <= 1e-12


@pytest.mark.parametrize("pieces", [[30, 18], [1] * 48, [7, 1, 23, 17], [47, 1]])
def test_tiny_decoder_prompt_in_pieces(tiny_runs, pieces):
    """Running the prompt in consecutive pieces fills the same cache, and its last piece gives the
    same last-row logits, as one pass over the whole prompt ("Prefill and decode"; the page checks
    30 + 18 and one id at a time, the other splits put several ids on a non-empty cache too)."""
    g, model, prompt, runs = tiny_runs
    whole = model.new_cache()
    model(prompt, whole)
    split = model.new_cache()
    start = 0
    for n in pieces:
        last = model(prompt[start:start + n], split)[-1]
        start += n
    assert start == g["P"] == int(split.committed()[0])
    assert np.abs(split.k - whole.k).max() <= 1e-12 and np.abs(split.v - whole.v).max() <= 1e-12
    assert np.abs(last - runs[False]["logits"][0]).max() <= 1e-9
