"""Float64 oracle of a small decoder-only transformer whose attention reads a KV cache.

TEST INFRASTRUCTURE ONLY: the rules of `oracle/kvc_oracle.py` apply here too (only `tests/`,
`__graft_entry__.smoke()` and the CPU baseline leg of `bench.py` use it; the library never does).

It is the oracle of the tiny-decoder workload: 96 token ids, model width 128, 4 heads of 32 (every
head has its own keys and values), 4 layers, a learned table of 256 absolute positions. The page
that defines it is "KV cache decoding" (problem statement, the table of shapes, its numbered steps
and "Why the causal mask makes caching exact"). What one call computes, in the page's notation
(t = tokens the cache already holds, m = new tokens in this call; t = 0 without a cache):

* the new tokens' hidden rows are their token-table rows plus position-table rows t .. t+m-1
  (the position comes from the cache length, never from 0);
* every layer normalises the rows, projects them to queries, keys and values, stores the keys and
  values in cache slots t .. t+m-1 and reads back all t+m of them, lets row i attend to keys
  0 .. t+i with scores q.k / sqrt(d_head), mixes the heads' outputs back into the residual stream,
  then normalises again and adds a ReLU MLP four times as wide (which acts on each row alone);
* after the last layer the cache's length becomes t+m (one commit per call, not per layer);
* a final normalisation and the vocabulary projection give (m, vocab) logits.

The attention of each head is `kvc_oracle.attend`, the same offset-masked softmax the cache oracle
uses, so the cache under test is an `OracleKVCache` with one sequence. Work is tallied the way the
page's correctness tests count it: positions pushed through the stack, and t+m scores for each of
the m rows, of every head, in every layer.

Parameters are drawn by `kvc_synth` from one seed. `init="pages"` scales a weight matrix with
`rows` input features by 1/sqrt(rows) and leaves the embedding tables at unit variance, as the
page does; `init="baseline"` draws every weight and table with standard deviation 0.02. Every
normalisation has gain 1 and bias 0.

Parity status: pinned by `tests/test_oracle_pins.py` (the page's printed score and position counts,
cached == uncached at every step, prefix rows unchanged by later tokens, any split of the prompt into
chunks giving the same cache and logits).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

import kvc_synth
from oracle.kvc_oracle import OracleKVCache, attend


@dataclass(frozen=True)
class DecoderShape:
    vocab: int = 96
    d_model: int = 128
    n_heads: int = 4
    n_layers: int = 4
    max_len: int = 256

    @property
    def d_head(self) -> int:
        return self.d_model // self.n_heads


@dataclass
class DecoderWeights:
    """Every parameter as a plain float64 array; per-layer ones are stacked on a leading layer axis."""
    token_table: np.ndarray       # [vocab, d_model]
    position_table: np.ndarray    # [max_len, d_model]
    w_qkv: np.ndarray             # [n_layers, 3, d_model, d_model]: query, key, value projections
    w_mix: np.ndarray             # [n_layers, d_model, d_model]: heads back into the residual stream
    w_up: np.ndarray              # [n_layers, d_model, 4 d_model]
    w_down: np.ndarray            # [n_layers, 4 d_model, d_model]
    norm_gain: np.ndarray         # [n_layers, 2, d_model]: before attention, before the MLP
    norm_bias: np.ndarray         # [n_layers, 2, d_model]
    final_gain: np.ndarray        # [d_model]
    final_bias: np.ndarray        # [d_model]
    w_vocab: np.ndarray           # [d_model, vocab]


@dataclass
class WorkTally:
    positions: int = 0            # token positions pushed through the stack
    scores: int = 0               # attention scores computed


@dataclass
class TinyDecoder:
    shape: DecoderShape
    weights: DecoderWeights
    cache_dtype: str = "f64"
    tally: WorkTally = field(default_factory=WorkTally)

    def new_cache(self) -> OracleKVCache:
        s = self.shape
        return OracleKVCache(s.n_layers, 1, s.n_heads, s.d_head, s.max_len, dtype=self.cache_dtype)

    def __call__(self, ids, cache: OracleKVCache | None = None) -> np.ndarray:
        return decoder_logits(self.shape, self.weights, ids, cache, self.tally)


def build_tiny_decoder(shape: DecoderShape = DecoderShape(), seed: int = 0, init: str = "pages",
                       cache_dtype: str = "f64") -> TinyDecoder:
    """Draw every parameter from `seed` (one `kvc_synth` stream per array, in a fixed order)."""
    if shape.d_model % shape.n_heads:
        raise ValueError("d_model must be a multiple of n_heads")
    if init not in ("pages", "baseline"):
        raise ValueError(f"unknown init {init!r}")
    serial = iter(range(1 << 16))

    def gaussian(dims, fan_in=None):
        std = 0.02 if init == "baseline" else (1.0 if fan_in is None else 1.0 / np.sqrt(fan_in))
        stream = kvc_synth.stream_id(kvc_synth.STREAM_WEIGHTS, step=next(serial))
        return kvc_synth.normal_f32(dims, seed, stream).astype(np.float64) * std

    L, D, V = shape.n_layers, shape.d_model, shape.vocab
    weights = DecoderWeights(
        token_table=gaussian((V, D)),
        position_table=gaussian((shape.max_len, D)),
        w_qkv=np.stack([np.stack([gaussian((D, D), D) for _ in range(3)]) for _ in range(L)]),
        w_mix=np.stack([gaussian((D, D), D) for _ in range(L)]),
        w_up=np.stack([gaussian((D, 4 * D), D) for _ in range(L)]),
        w_down=np.stack([gaussian((4 * D, D), 4 * D) for _ in range(L)]),
        norm_gain=np.ones((L, 2, D)),
        norm_bias=np.zeros((L, 2, D)),
        final_gain=np.ones(D),
        final_bias=np.zeros(D),
        w_vocab=gaussian((D, V), D),
    )
    return TinyDecoder(shape, weights, cache_dtype)


def layer_norm(x, gain, bias, eps=1e-5):
    """LayerNorm over the feature axis: each row is normalised on its own."""
    centred = x - x.mean(axis=-1, keepdims=True)
    return gain * centred / np.sqrt((centred ** 2).mean(axis=-1, keepdims=True) + eps) + bias


def decoder_logits(shape: DecoderShape, w: DecoderWeights, ids, cache: OracleKVCache | None = None,
                   tally: WorkTally | None = None) -> np.ndarray:
    """Logits [m, vocab] of m new token ids.

    Without a cache `ids` is the whole sequence (t = 0) and nothing is kept. With a cache holding t
    tokens the ids sit at positions t .. t+m-1; their keys and values are stored and their queries
    see all t+m stored rows of each layer.
    """
    ids = np.asarray(ids, dtype=np.int64)
    m = len(ids)
    t = 0 if cache is None else int(cache.lens[0])
    if t + m > shape.max_len:
        raise OverflowError("the sequence would pass max_len")
    dh = shape.d_head
    head_cols = [slice(j * dh, (j + 1) * dh) for j in range(shape.n_heads)]

    x = w.token_table[ids] + w.position_table[t:t + m]
    for layer in range(shape.n_layers):
        a = layer_norm(x, w.norm_gain[layer, 0], w.norm_bias[layer, 0])
        q, k, v = (a @ w.w_qkv[layer, n] for n in range(3))
        if cache is None:
            keys = [k[:, c] for c in head_cols]
            values = [v[:, c] for c in head_cols]
        else:
            k_heads = np.stack([k[:, c] for c in head_cols])[None]     # [1, H, m, d_head]
            v_heads = np.stack([v[:, c] for c in head_cols])[None]
            (keys, values), = cache.append(layer, k_heads, v_heads)    # [H, t+m, d_head] as stored
        mixed = np.concatenate([attend(q[:, c], keys[j], values[j], q_offset=t)
                                for j, c in enumerate(head_cols)], axis=1)
        x = x + mixed @ w.w_mix[layer]
        b = layer_norm(x, w.norm_gain[layer, 1], w.norm_bias[layer, 1])
        x = x + np.maximum(b @ w.w_up[layer], 0.0) @ w.w_down[layer]
        if tally is not None:
            tally.scores += shape.n_heads * m * (t + m)
    if cache is not None:
        cache.commit()
    if tally is not None:
        tally.positions += m
    return layer_norm(x, w.final_gain, w.final_bias) @ w.w_vocab


def greedy(model: TinyDecoder, prompt, n_new: int, use_cache: bool):
    """Extend `prompt` by n_new argmax tokens.

    use_cache=False runs the whole sequence through the model for every new token; use_cache=True
    runs the prompt once and then only the token picked last. Returns (prompt + new ids, the logits
    row each new id was picked from [n_new, vocab], the cache or None). The token picked last is
    never run, so the cache ends up holding len(prompt) + n_new - 1 positions.
    """
    seq = [int(i) for i in prompt]
    cache = model.new_cache() if use_cache else None
    feed = list(seq)
    rows = []
    for _ in range(n_new):
        last = model(feed if use_cache else seq, cache)[-1]
        rows.append(last)
        seq.append(int(np.argmax(last)))
        feed = seq[-1:]
    return seq, np.stack(rows), cache
