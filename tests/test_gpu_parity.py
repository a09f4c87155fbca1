"""GPU parity: the library (through its C ABI) against the float64 oracle on seeded inputs.

Bit-exact: cache contents (the whole store, never-written zeros included) and lengths.
Within tolerance: attention outputs, 1e-5 absolute for float32 caches and 2e-3 relative
(max-abs over each query head's T x d_h outputs) for float16/bfloat16 caches.
"""
import numpy as np
import pytest

import kvc_synth
from oracle.kvc_oracle import OracleKVCache, full_recompute_attention, gqa_cached_attention, store_round, stored_to_f64
from tests.gpu_parity import Mirror, check_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    import torch
    torch.backends.cuda.matmul.allow_tf32 = False
    torch.backends.cudnn.allow_tf32 = False
    yield


def test_synth_fill_matches_host_bits():
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    for n, off, stream, std in ((1000, 0, 1, 1.0), (4097, 123456789, 77, 1.0), (333, 2 ** 33 + 5, 9, 0.02)):
        t = torch.empty(n, dtype=torch.float32, device="cuda")
        kb.synth_fill_normal(t, 5, stream, std=std, offset=off)
        host = kvc_synth.normal_f32((n,), 5, stream, std=std, offset=off)
        np.testing.assert_array_equal(t.cpu().numpy().view(np.uint32), host.view(np.uint32))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_append_commit_truncate_bit_exact(dtype):
    m = Mirror(L=3, B=3, H_kv=2, d_h=64, max_len=40, dtype=dtype)
    for layer in range(3):
        m.append(layer, 7)
    m.check_state()
    m.commit()
    m.truncate([2, 7, 0])                 # ragged
    m.check_state()
    for T in (1, 5):
        for layer in range(3):
            m.append(layer, T, in_dtype="f32" if T == 1 else dtype)
        m.commit()
        m.check_state()
    m.truncate(3)
    for layer in range(3):
        m.append(layer, 2)
    m.check_state()
    m.close()


def test_toy_gqa_fp32_cached_equals_oracle_and_full_recompute():
    """Cached GQA attention, fp32: B=1, L=4, H_q=4, H_kv=2, d_h=32, max_len=128; prefill T=48 then
    20 decode steps, each checked against the oracle and against full recompute."""
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    w = kvc_synth.WORKLOADS["toy-gqa-fp32"]
    L, B, Hq, Hkv, d, n_max = w["L"], w["B"], w["H_q"], w["H_kv"], w["d_h"], w["max_len"]
    n = w["prefill"] + w["decode_steps"]
    q = kvc_synth.normal_f32((L, B, Hq, n, d), w["seed"], kvc_synth.STREAM_Q)
    k = kvc_synth.normal_f32((L, B, Hkv, n, d), w["seed"], kvc_synth.STREAM_K_PREFILL)
    v = kvc_synth.normal_f32((L, B, Hkv, n, d), w["seed"], kvc_synth.STREAM_V_PREFILL)
    gpu = kb.Cache(L, B, Hkv, d, n_max, 0)
    ref = OracleKVCache(L, B, Hkv, d, n_max, "f32")
    from oracle.kvc_oracle import gqa_cached_attention
    full = np.zeros((L, B, Hq, n, d))
    for layer in range(L):
        full[layer, 0] = full_recompute_attention(q[layer, 0].astype(np.float64), k[layer, 0].astype(np.float64),
                                                  v[layer, 0].astype(np.float64))
    s = 0
    for T in [w["prefill"]] + [1] * w["decode_steps"]:
        for layer in range(L):
            sl = slice(s, s + T)
            kd = torch.from_numpy(np.ascontiguousarray(k[layer, :, :, sl])).cuda()
            vd = torch.from_numpy(np.ascontiguousarray(v[layer, :, :, sl])).cuda()
            qd = torch.from_numpy(np.ascontiguousarray(q[layer, :, :, sl])).cuda()
            kb.kvc_append(gpu, layer, kd, vd)
            ref.append(layer, k[layer, :, :, sl], v[layer, :, :, sl])
            got = kb.gqa_cached_attn(gpu, qd, layer).cpu().numpy()
            want = gqa_cached_attention(ref, layer, q[layer, :, :, sl])
            check_outputs(got, want, "f32", f"s={s} T={T} layer {layer}")
            assert np.abs(got - full[layer, :, :, sl]).max() <= 1e-5
        kb.kvc_commit(gpu)
        ref.commit()
        s += T
    assert kb.kvc_seq_len(gpu) == [n]
    gpu.close()


CASES = [
    # dtype, d_h, H_q, H_kv, T, lengths
    ("bf16", 128, 32, 8, 1, [0, 1, 63, 64, 65, 700, 1500]),
    ("f16", 64, 9, 3, 1, [2048, 5, 129]),
    ("f32", 32, 4, 2, 1, [47, 300]),
    ("bf16", 128, 8, 8, 1, [257, 3]),          # G = 1
    ("f16", 128, 16, 2, 1, [513, 31]),         # G = 8
    ("f32", 128, 8, 2, 1, [100, 33]),
    ("f32", 64, 6, 2, 1, [260, 1]),
    ("f16", 32, 8, 2, 1, [600, 17]),
    ("bf16", 64, 12, 4, 2, [90, 0]),
    ("f16", 128, 32, 8, 3, [777, 64]),
    ("bf16", 128, 32, 8, 5, [128, 1000]),
    ("f16", 128, 32, 8, 8, [2048, 333]),       # speculative verify chunk
    ("f32", 32, 4, 2, 17, [0, 40]),
    ("bf16", 32, 4, 1, 64, [0, 100]),
    ("f16", 64, 4, 4, 129, [1, 200]),
    # chunks of more than 32 query rows per K/V head on the tensor-core chunk kernel
    ("bf16", 128, 32, 8, 9, [0, 300]),         # 36 rows: one partial row tile
    ("bf16", 128, 32, 8, 7, [129, 1]),         # 28 rows: four copies of the rows, 32 keys each
    ("f16", 128, 24, 8, 11, [500, 7]),         # G = 3, 33 rows: two copies of the rows
    ("bf16", 128, 32, 8, 16, [2047, 64]),      # 64 rows: two copies, every MMA row used
    ("f16", 128, 32, 8, 64, [5, 700]),         # 256 rows: two full row tiles
    ("bf16", 128, 16, 2, 17, [130, 0, 3]),     # G = 8, 136 rows: a ragged last tile
    ("f16", 128, 8, 8, 200, [0, 129]),         # G = 1, 200 rows, diagonal masking over many tiles
    ("f16", 128, 32, 8, 64, [90, 1000]),       # the first 128 rows of a CTA end a key tile earlier
    ("bf16", 128, 32, 8, 96, [10, 400]),       # 384 rows: the second CTA has one 128-row tile
    ("f16", 128, 16, 4, 75, [0, 333]),         # 300 rows: the second CTA has one ragged tile
]


@pytest.mark.parametrize("dtype,d,Hq,Hkv,T,lengths", CASES)
def test_attention_matches_oracle(dtype, d, Hq, Hkv, T, lengths):
    B = len(lengths)
    max_len = max(lengths) + T + 8
    m = Mirror(L=2, B=B, H_kv=Hkv, d_h=d, max_len=max_len, dtype=dtype, seed=len(CASES) + T)
    s0 = max(lengths)
    if s0:
        for layer in range(2):
            m.append(layer, s0)
        m.commit()
        m.truncate(np.array(lengths))
    m.forward(T, Hq, what=f"{dtype} d={d} G={Hq // Hkv} T={T}")
    m.check_state()
    m.close()


@pytest.mark.parametrize("dtype,T", [("f16", 64), ("bf16", 96), ("bf16", 1), ("f16", 8)])
def test_scores_growing_along_the_keys(dtype, T):
    """Keys aligned with the queries and growing with position: every key tile's largest score passes
    the previous tiles' by far, so a running softmax must rescale its partial output on every tile."""
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    B, H, Hq, d = 2, 2, 8, 128
    lengths = [700, 301]
    n = max(lengths)
    m = Mirror(L=1, B=B, H_kv=H, d_h=d, max_len=n + T + 8, dtype=dtype, seed=77)
    pos = np.arange(n + T, dtype=np.float32)
    k_all = (pos[None, None, :, None] / 32.0 + 0.3 * kvc_synth.normal_f32((B, H, n + T, d), 77, 1)).astype(np.float32)
    v_all = kvc_synth.normal_f32((B, H, n + T, d), 77, 2)

    def append(k, v):
        m.ref.append(0, k, v)
        kb.kvc_append(m.gpu, 0, m.dev(k), m.dev(v))

    append(k_all[:, :, :n], v_all[:, :, :n])
    m.commit()
    m.truncate(np.array(lengths))
    append(np.stack([k_all[b, :, s:s + T] for b, s in enumerate(lengths)]),
           np.stack([v_all[b, :, s:s + T] for b, s in enumerate(lengths)]))
    q = (1.0 + 0.3 * kvc_synth.normal_f32((B, Hq, T, d), 77, 3)).astype(np.float32)
    want = gqa_cached_attention(m.ref, 0, q)
    got = kb.gqa_cached_attn(m.gpu, m.dev(q), 0).cpu().numpy()
    check_outputs(got, want, dtype, f"growing scores {dtype} T={T}")
    torch.cuda.synchronize()
    m.close()


@pytest.mark.parametrize("split", [64, 128, 512, 1024])
def test_split_size_does_not_change_results(split):
    m = Mirror(L=1, B=3, H_kv=2, d_h=128, max_len=1100, dtype="bf16", seed=3)
    m.append(0, 1000)
    m.commit()
    m.truncate(np.array([999, 500, 64]))
    m.append(0, 1)
    got, want = m.attend(0, 8, 1, split_keys=split)
    check_outputs(got, want, "bf16", f"split {split}")
    m.close()


@pytest.mark.parametrize("dtype,d,Hq,Hkv,T,split", [
    ("f16", 64, 9, 3, 1, 0),          # the planner's own splits (9 per unit on this shape)
    ("f16", 64, 9, 3, 1, 1024),       # 3 splits per unit
    ("bf16", 128, 32, 8, 1, 0),
    ("bf16", 128, 32, 8, 1, 256),     # 9 splits: a cluster past the portable size of 8
    ("bf16", 128, 16, 4, 4, 128),     # 17 splits: more than a cluster holds, the L2 merge instead
    ("f16", 128, 8, 2, 2, 384),
])
def test_uniform_splits_merge_in_a_cluster(dtype, d, Hq, Hkv, T, split):
    """Every sequence as long as the others and one wave of CTAs: the splits of each (sequence, K/V
    head) run as one thread-block cluster and merge through distributed shared memory."""
    B, s0 = 4, 2048
    m = Mirror(L=2, B=B, H_kv=Hkv, d_h=d, max_len=s0 + 2 * T + 4, dtype=dtype, seed=17 + split)
    for layer in range(2):
        m.append(layer, s0)
    m.commit()
    for step in range(2):
        for layer in range(2):
            m.append(layer, T)
            got, want = m.attend(layer, Hq, T, split_keys=split)
            check_outputs(got, want, dtype, f"cluster merge split={split} step {step} layer {layer}")
        m.commit()
    m.check_state()
    m.close()


def test_query_in_cache_dtype_equals_rounded_f32_query():
    m = Mirror(L=1, B=2, H_kv=2, d_h=64, max_len=300, dtype="f16", seed=4)
    m.append(0, 250)
    got_f32, want = m.attend(0, 4, 250)
    check_outputs(got_f32, want, "f16")
    m.n_draws -= 1                               # draw the same queries again
    got_16, want2 = m.attend(0, 4, 250, q_in="f16")
    np.testing.assert_array_equal(want, want2)
    np.testing.assert_array_equal(got_f32, got_16)
    m.close()


def test_speculative_verify_rollback_reappend():
    """Verify chunk T=8 at s, truncate back 5, re-append the same rows: the store is bit-identical
    to before the truncate and the attention outputs repeat exactly."""
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    L, B, Hq, Hkv, d, s = 2, 3, 16, 4, 128, 300
    m = Mirror(L=L, B=B, H_kv=Hkv, d_h=d, max_len=s + 16, dtype="f16", seed=6)
    for layer in range(L):
        m.append(layer, s)
    m.commit()
    drafts = [(kvc_synth.normal_f32((B, Hkv, 8, d), 6, 50 + l), kvc_synth.normal_f32((B, Hkv, 8, d), 6, 60 + l))
              for l in range(L)]
    q = kvc_synth.normal_f32((B, Hq, 5, d), 6, 70)
    for layer in range(L):
        kb.kvc_append(m.gpu, layer, m.dev(drafts[layer][0]), m.dev(drafts[layer][1]))
    kb.kvc_commit(m.gpu)
    before = (m.gpu.k.clone(), m.gpu.v.clone())
    kb.kvc_truncate(m.gpu, s + 3)
    assert kb.kvc_seq_len(m.gpu) == [s + 3] * B
    outs = []
    for layer in range(L):
        kb.kvc_append(m.gpu, layer, m.dev(drafts[layer][0][:, :, 3:]), m.dev(drafts[layer][1][:, :, 3:]))
        outs.append(kb.gqa_cached_attn(m.gpu, m.dev(q), layer).cpu().numpy())
    kb.kvc_commit(m.gpu)
    assert torch.equal(before[0], m.gpu.k) and torch.equal(before[1], m.gpu.v)
    kb.kvc_truncate(m.gpu, s + 3)
    for layer in range(L):
        kb.kvc_append(m.gpu, layer, m.dev(drafts[layer][0][:, :, 3:]), m.dev(drafts[layer][1][:, :, 3:]))
        np.testing.assert_array_equal(kb.gqa_cached_attn(m.gpu, m.dev(q), layer).cpu().numpy(), outs[layer])
    # and the oracle agrees with the outputs
    ref = OracleKVCache(L, B, Hkv, d, s + 16, "f16")
    ref.k[...] = m.ref.k
    ref.v[...] = m.ref.v
    ref.fill[:] = s
    ref.lens[:] = s
    from oracle.kvc_oracle import gqa_cached_attention
    for layer in range(L):
        ref.append(layer, drafts[layer][0][:, :, :3], drafts[layer][1][:, :, :3])
    ref.commit()
    for layer in range(L):
        ref.append(layer, drafts[layer][0][:, :, 3:], drafts[layer][1][:, :, 3:])
        check_outputs(outs[layer], gqa_cached_attention(ref, layer, q), "f16", f"layer {layer}")
    m.close()


def test_errors_leave_state_unchanged():
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    m = Mirror(L=2, B=2, H_kv=2, d_h=64, max_len=10, dtype="bf16", seed=8)
    for layer in range(2):
        m.append(layer, 6)
    m.commit()
    m.append(0, 1)
    snap = (m.gpu.k.clone(), m.gpu.v.clone(), kb.kvc_seq_len(m.gpu, 0), kb.kvc_seq_len(m.gpu, 1),
            kb.kvc_seq_len(m.gpu))
    big = torch.zeros((2, 2, 4, 64), device="cuda")
    q = torch.zeros((2, 4, 1, 64), device="cuda")
    bad = [
        (-2, lambda: kb.kvc_append(m.gpu, 0, big, big)),                 # past max_len
        (-1, lambda: kb.kvc_append(m.gpu, 2, big, big)),                 # layer out of range
        (-3, lambda: kb.kvc_commit(m.gpu)),                                # layer 1 not appended
        (-3, lambda: kb.kvc_truncate(m.gpu, 7)),                           # beyond committed length
        (-1, lambda: kb.kvc_truncate(m.gpu, -1)),
        (-3, lambda: kb.gqa_cached_attn(m.gpu, q, 1)),                     # layer 1 lacks the chunk
        (-3, lambda: kb.gqa_cached_attn(m.gpu, q, 0, s=5)),                # wrong explicit s
        (-1, lambda: kb.gqa_cached_attn(m.gpu, torch.zeros((2, 3, 1, 64), device="cuda"), 0)),  # H_q % H_kv
        (-1, lambda: kb.kvc_append(m.gpu, 1, big.half(), big.half())),     # f16 into a bf16 cache
    ]
    for code, fn in bad:
        with pytest.raises(kb.KvcError) as ei:
            fn()
        assert ei.value.code == code, str(ei.value)
    torch.cuda.synchronize()
    assert torch.equal(snap[0], m.gpu.k) and torch.equal(snap[1], m.gpu.v)
    assert (kb.kvc_seq_len(m.gpu, 0), kb.kvc_seq_len(m.gpu, 1), kb.kvc_seq_len(m.gpu)) == snap[2:]
    kb.kvc_status(m.gpu)
    m.close()


def test_tiny_decoder_cached_vs_uncached_logits():
    """Tiny decoder, fp32, N(0, 0.02) weights: vocab 96, d_model 128, 4 heads (MHA), 4 layers,
    learned positions, max_len 256; prompt of 48 ids, 20 greedy tokens. The dense layers run in
    torch float32 (the harness); the cache and attention run in the library. Logits match the
    float64 oracle within 1e-5 at every step; greedy ids match unless the oracle's top-1/top-2
    margin is below 1e-4 ("Generation and the KV Cache", verify_cache's margin gate)."""
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    from oracle.tiny_decoder import DecoderShape, build_tiny_decoder, decoder_logits, greedy
    w = kvc_synth.WORKLOADS["tiny-decoder-fp32"]
    shape = DecoderShape(w["vocab"], w["d_model"], w["n_heads"], w["n_layers"], w["max_len"])
    model = build_tiny_decoder(shape, seed=w["seed"], init="baseline", cache_dtype="f32")
    prompt = kvc_synth.prompt_ids(w["prompt"], w["vocab"], w["seed"])
    n_new, P = w["new_tokens"], len(prompt)
    ids_ref, logits_ref, _ = greedy(model, prompt, n_new, use_cache=True)
    uncached = np.stack([decoder_logits(shape, model.weights, ids_ref[:P + i])[-1] for i in range(n_new)])
    assert np.abs(uncached - logits_ref).max() < 1e-5          # the oracle's own two paths agree

    wt = {k: torch.from_numpy(np.asarray(v, dtype=np.float32)).cuda() for k, v in vars(model.weights).items()}
    H, dh, dm = shape.n_heads, shape.d_head, shape.d_model
    cache = kb.Cache(shape.n_layers, 1, H, dh, shape.max_len, 0)
    norm = lambda x, g, b: torch.nn.functional.layer_norm(x, (dm,), g, b, eps=1e-5)
    as_heads = lambda y: y.view(-1, H, dh).permute(1, 0, 2).unsqueeze(0).contiguous()   # [1, H, m, dh]

    def run(ids):
        t = kb.kvc_seq_len(cache)[0]
        x = wt["token_table"][torch.tensor(ids, device="cuda")] + wt["position_table"][t:t + len(ids)]
        for layer in range(shape.n_layers):
            a = norm(x, wt["norm_gain"][layer, 0], wt["norm_bias"][layer, 0])
            q, k, v = (as_heads(a @ wt["w_qkv"][layer, n]) for n in range(3))
            kb.kvc_append(cache, layer, k, v)
            o = kb.gqa_cached_attn(cache, q, layer)                        # [1, H, m, dh]
            x = x + o[0].permute(1, 0, 2).reshape(-1, dm) @ wt["w_mix"][layer]
            b = norm(x, wt["norm_gain"][layer, 1], wt["norm_bias"][layer, 1])
            x = x + torch.relu(b @ wt["w_up"][layer]) @ wt["w_down"][layer]
        kb.kvc_commit(cache)
        return (norm(x, wt["final_gain"], wt["final_bias"]) @ wt["w_vocab"]).double().cpu().numpy()

    feed = list(prompt)
    for step in range(n_new):                            # teacher-forced on the oracle's ids
        got = run(feed)[-1]
        assert np.abs(got - logits_ref[step]).max() <= 1e-5, step
        top2 = np.sort(logits_ref[step])[-2:]
        if top2[1] - top2[0] >= 1e-4:
            assert int(np.argmax(got)) == ids_ref[P + step]
        feed = [ids_ref[P + step]]
    assert kb.kvc_seq_len(cache) == [P + n_new - 1]
    cache.close()


def test_bounded_wait_gives_up_and_reports_without_fault():
    """A kernel wait that runs out sets the status word; kvc_status reports it once, and the handle
    (and the CUDA context) keep working."""
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    m = Mirror(L=1, B=2, H_kv=2, d_h=128, max_len=64, dtype="bf16", seed=9)
    m.append(0, 40)
    kb.kvc_selftest_wait_timeout(m.gpu, 2000)                 # 2 ms
    with pytest.raises(kb.KvcError) as ei:
        kb.kvc_status(m.gpu)
    assert ei.value.code == -5
    kb.kvc_status(m.gpu)                                       # the flag was cleared
    got, want = m.attend(0, 8, 40)
    check_outputs(got, want, "bf16", "after a reported timeout")
    kb.kvc_status(m.gpu)
    m.close()
