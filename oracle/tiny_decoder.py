"""A tiny decoder-only transformer in float64 NumPy, run with and without a KV cache.

TEST INFRASTRUCTURE ONLY (see `oracle/kvc_oracle.py`). It is the oracle for the
tiny-decoder workload: vocab 96, d_model 128, 4 heads (MHA), 4 layers, learned
positional embedding, max_len 256 ("KV cache decoding", problem statement and
the TinyDecoder listing). Its structure, from that page's steps 1-7:

* x = tok_emb[ids] + pos_emb[t : t + m], t the cached length (step 2);
* per layer: pre-LN (eps 1e-5), q/k/v projections of the m new tokens (step 4),
  append k/v to the cache and read back all t + m rows (step 5), scores
  q k^T / sqrt(d_head) under the offset causal mask, softmax, weighted sum of v,
  output projection and residual, then pre-LN and a ReLU 4x MLP (step 6);
* the length is committed once, after the last layer (step 7);
* final LN and the output projection give (m, vocab) logits.

Work counters follow step 10 and the "Correctness tests" list of that page:
positions pushed through the stack, and attention scores n_heads * m * (t + m)
per layer.

Weights are drawn by `kvc_synth` (seeded). `init="pages"` uses the page's
scales (weights N(0, 1/sqrt(rows)), embeddings N(0, 1)); `init="baseline"`
uses N(0, 0.02) for every weight and embedding. LayerNorm gains are 1 and
biases 0 in both.
"""
from __future__ import annotations

import numpy as np

import kvc_synth
from oracle.kvc_oracle import OracleKVCache, attend


def layer_norm(x, gain, bias, eps=1e-5):
    """Normalise each position over its features; never mixes positions."""
    mean = x.mean(axis=-1, keepdims=True)
    var = x.var(axis=-1, keepdims=True)
    return gain * (x - mean) / np.sqrt(var + eps) + bias


class TinyDecoder:
    def __init__(self, vocab=96, d_model=128, n_heads=4, n_layers=4, max_len=256, seed=0,
                 init="pages", cache_dtype="f64"):
        assert d_model % n_heads == 0
        self.vocab, self.d_model, self.max_len = vocab, d_model, max_len
        self.n_heads, self.n_layers, self.d_head = n_heads, n_layers, d_model // n_heads
        self.cache_dtype = cache_dtype
        counter = [0]

        def draw(shape, std):
            stream = kvc_synth.stream_id(kvc_synth.STREAM_WEIGHTS, step=counter[0])
            counter[0] += 1
            return kvc_synth.normal_f32(shape, seed, stream).astype(np.float64) * std

        def w(rows, cols):
            return draw((rows, cols), 1.0 / np.sqrt(rows) if init == "pages" else 0.02)

        emb_std = 1.0 if init == "pages" else 0.02
        self.tok_emb = draw((vocab, d_model), emb_std)
        self.pos_emb = draw((max_len, d_model), emb_std)
        self.layers = [{
            "w_q": w(d_model, d_model), "w_k": w(d_model, d_model),
            "w_v": w(d_model, d_model), "w_o": w(d_model, d_model),
            "w_1": w(d_model, 4 * d_model), "w_2": w(4 * d_model, d_model),
            "g1": np.ones(d_model), "b1": np.zeros(d_model),
            "g2": np.ones(d_model), "b2": np.zeros(d_model),
        } for _ in range(n_layers)]
        self.g_out, self.b_out = np.ones(d_model), np.zeros(d_model)
        self.w_out = w(d_model, vocab)
        self.positions = 0   # positions pushed through the stack
        self.scores = 0      # attention scores computed

    def new_cache(self) -> OracleKVCache:
        return OracleKVCache(self.n_layers, 1, self.n_heads, self.d_head, self.max_len,
                             dtype=self.cache_dtype)

    def _split(self, x):
        """(m, d_model) -> (h, m, d_head)."""
        return x.reshape(x.shape[0], self.n_heads, self.d_head).transpose(1, 0, 2)

    def forward(self, ids, cache: OracleKVCache | None = None) -> np.ndarray:
        """m new token ids -> (m, vocab) logits; with a cache holding t tokens they sit at t..t+m-1."""
        t = 0 if cache is None else int(cache.lens[0])
        m = len(ids)
        if t + m > self.max_len:
            raise OverflowError("sequence is longer than max_len")
        x = self.tok_emb[ids] + self.pos_emb[t:t + m]
        for i, p in enumerate(self.layers):
            h = layer_norm(x, p["g1"], p["b1"])
            q = self._split(h @ p["w_q"])
            k = self._split(h @ p["w_k"])
            v = self._split(h @ p["w_v"])
            if cache is not None:
                (k, v), = cache.append(i, k[None], v[None])
            heads = np.stack([attend(q[j], k[j], v[j], q_offset=t) for j in range(self.n_heads)])
            x = x + heads.transpose(1, 0, 2).reshape(m, self.d_model) @ p["w_o"]
            h = layer_norm(x, p["g2"], p["b2"])
            x = x + np.maximum(h @ p["w_1"], 0.0) @ p["w_2"]
            self.scores += self.n_heads * m * (t + m)
        if cache is not None:
            cache.commit()
        self.positions += m
        return layer_norm(x, self.g_out, self.b_out) @ self.w_out


def generate_no_cache(model: TinyDecoder, prompt, n_new):
    """Greedy decoding that pushes the whole sequence through the model at every step."""
    ids, step_logits = list(prompt), []
    for _ in range(n_new):
        logits = model.forward(ids)[-1]
        step_logits.append(logits)
        ids.append(int(np.argmax(logits)))
    return ids, np.array(step_logits)


def generate_with_cache(model: TinyDecoder, prompt, n_new):
    """Greedy decoding with a KV cache: one prefill pass, then one token per call."""
    cache = model.new_cache()
    ids, step_logits = list(prompt), []
    new = list(prompt)
    for _ in range(n_new):
        logits = model.forward(new, cache)[-1]
        step_logits.append(logits)
        new = [int(np.argmax(logits))]
        ids.append(new[0])
    return ids, np.array(step_logits), cache


def teacher_forced_logits(model: TinyDecoder, ids, P: int):
    """Uncached last-row logits for every prefix ids[:P + i], i = 0 .. len(ids) - P - 1."""
    return np.array([model.forward(list(ids[:P + i]))[-1] for i in range(len(ids) - P)])
