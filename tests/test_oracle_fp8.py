"""Pins of the oracle's fp8 storage (e4m3_encode, e4m3_decode, scales) to things other than itself.

The pages name cache quantisation as a decode lever ("KV cache decoding", "What is cached, what is not,
and what it costs") without a format. The reading is FP8 E4M3 (OCP 8-bit floating point, E4M3: bias 7,
no infinities, largest finite 448) with one scale per layer for K and one for V. Pinned against
PyTorch's own float8_e4m3fn conversions (a library routine), hand-worked codes, and error bounds.
"""
import numpy as np
import pytest

from oracle.kvc_oracle import (OracleKVCache, OraclePagedKVCache, e4m3_decode, e4m3_encode,
                               gqa_cached_attention, set_fp8_scales)

torch = pytest.importorskip("torch")


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8).copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_encode(x):
    return torch.from_numpy(np.asarray(x, np.float32).copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got, want = e4m3_decode(codes), _torch_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)])
    assert np.count_nonzero(np.isnan(got)) == 2                       # 0x7F and 0xFF only


@pytest.mark.parametrize("scale", [1.0, 1e-2, 30.0])
def test_encode_matches_torch_in_range(scale):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(400000) * scale).astype(np.float32)
    x = np.concatenate([x, (rng.standard_normal(20000) * 2.0 ** -8).astype(np.float32)])   # subnormals
    x = x[np.abs(x) < 440]
    assert np.array_equal(e4m3_encode(x), _torch_encode(x))


def test_hand_worked_codes():
    cases = {
        0.0: 0x00, 1.0: 0x38, 1.125: 0x39, 448.0: 0x7E, -448.0: 0xFE, 2.0 ** -6: 0x08,
        2.0 ** -9: 0x01,                      # smallest subnormal
        1.0625: 0x38,                         # halfway between 1 and 1.125: to even (1.0)
        1.1875: 0x3A,                         # halfway between 1.125 and 1.25: to even (1.25)
        2.0 ** -10: 0x00,                     # halfway between 0 and 2^-9: to even (0)
        3 * 2.0 ** -10: 0x02,                 # halfway between 2^-9 and 2^-8: to even (2^-8)
        1.9375: 0x40,                         # rounds up into the next binade: 2.0
        449.0: 0x7E, 464.0: 0x7E, 500.0: 0x7E, 1e9: 0x7E, -1e9: 0xFE,   # saturate at +-448
    }
    for x, code in cases.items():
        assert int(e4m3_encode(np.float32(x))) == code, (x, hex(int(e4m3_encode(np.float32(x)))), hex(code))


def test_every_value_encodes_to_itself():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = e4m3_decode(codes).astype(np.float32)
    back = e4m3_encode(vals)
    assert np.array_equal(back[codes != 0x80], codes[codes != 0x80])
    assert e4m3_decode(back[codes == 0x80])[0] == 0.0                 # -0 reads as zero either way


def test_encode_is_monotonic():
    x = np.sort(np.random.default_rng(8).uniform(-500, 500, 100000).astype(np.float32))
    v = e4m3_decode(e4m3_encode(x))
    assert np.all(np.diff(v) >= 0)


@pytest.mark.parametrize("cls", [OracleKVCache, OraclePagedKVCache])
def test_fp8_cache_stores_codes_of_x_over_scale(cls):
    """Row values read back within half a step of the E4M3 grid times the scale: relative 2^-4 for
    normals, absolute 2^-10 * scale below 2^-6 * scale; the stored codes are e4m3(x / scale)."""
    args = (2, 2, 2, 8, 16) if cls is OracleKVCache else (2, 2, 2, 8, 16, 4, 8)
    c = cls(*args, dtype="e4m3")
    set_fp8_scales(c, [0.5, 3.0], [2.0, 0.25])
    rng = np.random.default_rng(9)
    k = rng.standard_normal((2, 2, 5, 8)).astype(np.float32) * 4
    v = rng.standard_normal((2, 2, 5, 8)).astype(np.float32)
    for layer in range(2):
        rows = c.append(layer, k, v)
        for b in range(2):
            ks, vs = rows[b]
            for x, got, sc in ((k[b], ks, c.k_scale[layer]), (v[b], vs, c.v_scale[layer])):
                err = np.abs(got - x.astype(np.float64))
                bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * sc)
                assert np.all(err <= bound + 1e-12)
    c1 = cls(*args, dtype="e4m3")
    set_fp8_scales(c1, 0.5, 0.5)
    c1.append(0, k, v)
    want = e4m3_encode((k / np.float32(0.5)).astype(np.float32))
    if cls is OracleKVCache:
        assert np.array_equal(c1.k[0, :, :, :5], want)


def test_scales_only_while_empty_and_positive():
    c = OracleKVCache(1, 1, 1, 4, 8, "e4m3")
    with pytest.raises(ValueError):
        set_fp8_scales(c, 0.0, 1.0)
    c.append(0, np.ones((1, 1, 1, 4), np.float32), np.ones((1, 1, 1, 4), np.float32))
    with pytest.raises(RuntimeError):
        set_fp8_scales(c, 2.0, 2.0)
    with pytest.raises(ValueError):
        set_fp8_scales(OracleKVCache(1, 1, 1, 4, 8, "f16"), 1.0, 1.0)


def test_fp8_attention_reads_dequantised_rows_and_a_float16_query():
    """With one key the output is that key's value as stored (code * scale); the query only matters
    through float16 rounding."""
    c = OracleKVCache(1, 1, 1, 4, 4, "e4m3")
    set_fp8_scales(c, 2.0, 0.125)
    v = np.array([[[[1.0, -3.0, 0.3, 100.0]]]], np.float32)
    c.append(0, np.ones((1, 1, 1, 4), np.float32), v)
    out = gqa_cached_attention(c, 0, np.ones((1, 2, 1, 4), np.float32))
    want = e4m3_decode(e4m3_encode(v[0, 0, 0] / np.float32(0.125))) * 0.125
    assert np.array_equal(out[0, 0, 0], want) and np.array_equal(out[0, 1, 0], want)
    assert not np.array_equal(want, v[0, 0, 0])            # 0.3 and 100 are not on the grid
