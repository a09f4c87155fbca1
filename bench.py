"""Benchmark of the KV-cached GQA decode step on one or more GB300s.

A step is one decode forward of the Llama-3-8B-shaped batch (32 layers; H_q=32, H_kv=8, d_h=128,
B=64, bf16 cache, ragged s_b ~ U[512, 4096], T=1): for every layer, append the new K/V row and
attend; then commit; then truncate back to s_b so every timed step does the same work. Inputs are
synthetic (seeded Philox draws) and already resident in HBM when timing starts; the K/V read per
layer (~580 MB) is far larger than L2, so no flush is needed between iterations.

Prints one JSON line (rank 0). `value` is algorithmic HBM GB/s of the whole job; `steps_per_s` and
the roofline fraction of the attention kernel come with it. `--impl reference` times the CPU oracle
instead, on a bounded sample of the same workload.

Multi-GPU: the workload has no exchange step, so each rank runs an independent replica (weak
scaling); timing is bracketed by barriers and the maximum over ranks is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "cached GQA decode-attention HBM GB/s (% of peak) and decode steps/sec"
DEFAULT_WORKLOAD = "llama3-8b-decode-bf16"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TFLOPS = 1900.0             # dense bf16, burst (fallback only)
FALLBACK_TFLOPS_SUSTAINED = 1700.0   # dense bf16, sustained (fallback only)


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--split-keys", type=int, default=0)
    p.add_argument("--layers", type=int, default=0,
                   help="profiling only: fewer layers of the same per-layer shape (not a bench line)")
    p.add_argument("--graph", action="store_true",
                   help="replay the whole step from one CUDA graph (for launch-bound small workloads)")
    p.add_argument("--fused", action="store_true",
                   help="one gqa_cached_attn_append call per layer instead of kvc_append + the attention call "
                        "(decode workloads)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample-seconds", type=float, default=12.0)
    p.add_argument("--cpu-sample-child", default=None, help=argparse.SUPPRESS)
    return p.parse_args(argv)


# ------------------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense 16-bit tensor TFLOP/s (bf16 and f16 run at the same rate): the sustained cuBLAS figure,
    since the attention kernel is timed inside a step of many back-to-back layers."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_TFLOPS_SUSTAINED, FALLBACK_TFLOPS, "fallback"


# The attention call of every TIMED_EVERY-th layer is bracketed by CUDA events (the roofline's kernel
# time); an event between two launches ends their programmatic overlap, so not every layer is timed.
TIMED_EVERY = 4

# The sources that define each attention kernel and its launch plan: a stored DRAM traffic figure
# stands only while these are unchanged since its ncu capture.
_SHARED_SOURCES = ("kvc_device.cuh", "kvc_host.cpp", "kvc_internal.h")
KERNEL_SOURCES = {
    "decode_tc_kernel": ("kvc_decode_tc.cu", "kvc_splitk.cu", "kvc_append.cuh") + _SHARED_SOURCES,
    "prefill_tc_kernel": ("kvc_prefill_tc.cu",) + _SHARED_SOURCES,
    "mla_tc_kernel": ("kvc_mla_tc.cu",) + _SHARED_SOURCES,
    "mla_kernel": ("kvc_mla.cu",) + _SHARED_SOURCES,
    "splitk_kernel": ("kvc_splitk.cu",) + _SHARED_SOURCES,
}


def kernel_of(sp):
    """The attention kernel's name, as `attention_kernel_name` states it."""
    return attention_kernel_name(sp).split("(")[1].split(":")[0]


def kernel_source_hash(kernel):
    """Hash of the sources that define `kernel` and its launch plan."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "kv_cached_gqa_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_per_launch(sp):
    """DRAM bytes per attention launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[sp.name]
        if e.get("kernel_sha") == kernel_source_hash(kernel_of(sp)):
            return e["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.device_index = device_index

    def __enter__(self):
        try:
            import torch
            ident = str(self.device_index)
            uuid = getattr(torch.cuda.get_device_properties(self.device_index), "uuid", None)
            if uuid is not None:
                ident = "GPU-" + str(uuid) if not str(uuid).startswith("GPU-") else str(uuid)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", ident], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, RuntimeError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# the CPU oracle on a bounded sample, on every host core: a child process (no GPU visible) spawns one
# worker process per core, each with one BLAS thread and a share of the sample's sequences
# ------------------------------------------------------------------------------------------------

def _oracle_sample(sp, b):
    """The oracle's layer-0 attention of sequence b, ready to run: (callable, algorithmic bytes)."""
    import numpy as np

    from oracle.kvc_oracle import OracleKVCache, OraclePagedKVCache, gqa_cached_attention, rope_chunk
    s_b = int(sp.lengths[b])
    if sp.mla:
        from oracle.kvc_oracle import OracleLatentCache, mla_cached_attention
        c = OracleLatentCache(1, 1, sp.d_h, sp.d_rope, s_b + sp.T, sp.dtype)
        if s_b:
            c.append(0, *(x[None] for x in sp.host_prefill_latent(0, b, s_b)))
            c.commit()
        c.append(0, *(x[None] for x in sp.host_step_latent(0, 0, b)))
        ql, qr = (x[None] for x in sp.host_queries_mla(0, 0, b, range(sp.H_q)))
        return (lambda: mla_cached_attention(c, 0, ql, qr, sp.mla_scale)), sp.attn_bytes([b])

    def rot(x, start):                 # the workload's rotary positions, if it has them
        return rope_chunk(x, [start], sp.rope_base, sp.rope_style) if sp.rope_base else x

    if sp.block:
        c = OraclePagedKVCache(1, 1, sp.H_kv, sp.d_h, s_b + sp.T, sp.block, -(-(s_b + sp.T) // sp.block), sp.dtype)
    else:
        c = OracleKVCache(1, 1, sp.H_kv, sp.d_h, s_b + sp.T, sp.dtype)
    if s_b:
        rows = [sp.host_prefill_rows(0, b, h, s_b) for h in range(sp.H_kv)]
        c.append(0, rot(np.stack([r[0] for r in rows])[None], 0), np.stack([r[1] for r in rows])[None])
        c.commit()
    new = [sp.host_step_rows(0, 0, b, h) for h in range(sp.H_kv)]
    c.append(0, rot(np.stack([r[0] for r in new])[None], s_b), np.stack([r[1] for r in new])[None])
    q = rot(sp.host_queries(0, 0, b, range(sp.H_q))[None], s_b)
    return (lambda: gqa_cached_attention(c, 0, q)), sp.attn_bytes([b])


def _oracle_worker(cfg, seqs, barrier, results):
    """One core's share: build its sequences' caches, meet the others at the barrier, then run
    passes over them (a fixed count in lockstep, one barrier per pass, or free-running for a time)."""
    import kvc_workloads
    sp = kvc_workloads.spec(cfg["workload"])
    jobs = [_oracle_sample(sp, b) for b in seqs]
    nbytes = sum(n for _, n in jobs)
    barrier.wait()
    times = []
    t_end = time.perf_counter() + cfg["seconds"]
    while (len(times) < cfg["passes"]) if cfg["passes"] else (time.perf_counter() < t_end or not times):
        if cfg["passes"]:
            barrier.wait()
        t0 = time.perf_counter()
        for run, _ in jobs:
            run()
        times.append(time.perf_counter() - t0)
    results.put({"seqs": list(seqs), "bytes": nbytes, "times": times})


def cpu_sample_child(arg):
    """Spread a sample of the batch's sequences (layer 0) over one worker per core; print a JSON result."""
    import multiprocessing as mp

    import kvc_workloads
    cfg = json.loads(arg)
    sp = kvc_workloads.spec(cfg["workload"])
    n_seq = min(cfg["n_seq"], sp.B)
    workers = max(1, min(cfg["workers"], n_seq))
    order = sorted(range(n_seq), key=lambda b: -int(sp.lengths[b]))     # longest first, dealt round-robin
    shares = [order[w::workers] for w in range(workers)]
    ctx = mp.get_context("spawn")
    barrier, results = ctx.Barrier(workers), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(cfg, share, barrier, results)) for share in shares]
    for p in procs:
        p.start()
    outs = [results.get(timeout=1200) for _ in procs]
    for p in procs:
        p.join()
    print(json.dumps({"workers": outs, "n_seq": n_seq, "n_workers": workers, "cores": os.cpu_count(),
                      "sample_bytes": sp.attn_bytes(range(n_seq)), "layer_bytes": sp.attn_bytes(),
                      "step_bytes": sp.step_bytes(), "B": sp.B, "L": sp.L}))


def run_cpu_sample(workload, n_seq, seconds=0.0, passes=0):
    """The oracle child: every host core (one BLAS thread per worker process), no GPU visible."""
    cores = os.cpu_count() or 1
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    arg = json.dumps({"workload": workload, "n_seq": n_seq, "workers": cores, "seconds": seconds,
                      "passes": passes})
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample-child", arg],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"oracle sample failed:\n{r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def _sample_text(res, how):
    return (f"layer 0 attention of {res['n_seq']} of the batch's {res['B']} sequences (all their heads), "
            f"float64 NumPy oracle on {res['n_workers']} worker processes of one BLAS thread each "
            f"({res['cores']} host cores), {how}; GB/s over the same algorithmic bytes as the GPU line; "
            f"a whole step ({res['L']} layers, {res['B']} sequences) scaled linearly from it")


def cpu_baseline_entry(workload, seconds, n_seq=None):
    """Throughput of the oracle with every core busy: the sum of the workers' rates over one window."""
    cores = os.cpu_count() or 1
    res = run_cpu_sample(workload, n_seq or cores, seconds=seconds)
    gbs = sum(w["bytes"] * len(w["times"]) / sum(w["times"]) for w in res["workers"]) / 1e9
    passes = sum(len(w["times"]) for w in res["workers"])
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": res["n_workers"], "kind": "oracle",
            "sample": _sample_text(res, f"{passes} passes over about {seconds:.0f} s"),
            "steps_per_s_equiv": round(gbs * 1e9 / res["step_bytes"], 6)}


# ------------------------------------------------------------------------------------------------
# arms
# ------------------------------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(values, device):
    """Each value's maximum over the job's ranks (the slowest rank's time), in one all_reduce; the
    values themselves when the job has one rank or no process group."""
    import torch
    import torch.distributed as dist
    values = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return values
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rate(units_per_rank, ms, world):
    """Whole-job rate: the units every rank processed (each runs its own replica of the workload)
    per second of the slowest rank's time."""
    return world * units_per_rank / (ms * 1e-3)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import kvc_workloads
    sp = kvc_workloads.spec(args.workload)
    res = run_cpu_sample(args.workload, os.cpu_count() or 1, passes=args.warmup + args.steps)
    # a step is one lockstep pass of every worker (they start together at a barrier): its time is the
    # slowest worker's
    step_s = [max(w["times"][i] for w in res["workers"]) for i in range(args.warmup, args.warmup + args.steps)]
    t = sum(step_s)
    gbs = res["sample_bytes"] * len(step_s) / t / 1e9
    sample = _sample_text(res, f"each step one lockstep pass of every worker ({args.steps} timed after "
                               f"{args.warmup} warm-up)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t / len(step_s), 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": sp.dtype, "data": "synthetic (seeded Philox draws)",
        "config": workload_config(sp, f"each step is the oracle over a bounded sample: layer 0 of "
                                      f"{res['n_seq']} sequences"),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": res["n_workers"], "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def attention_kernel_name(sp):
    """The kernel that serves the workload's attention calls (the library's own choice, restated)."""
    if sp.mla:
        if sp.dtype in ("f16", "bf16") and sp.d_h in (256, 512) and sp.d_rope == 64:
            return "mla_cached_attn (mla_tc_kernel: tcgen05 latent attention, online softmax, fused merge)"
        return "mla_cached_attn (mla_kernel: CUDA-core latent attention, split keys, fused merge)"
    rows = sp.T * (sp.H_q // sp.H_kv)
    tc_decode = rows <= 16 and ((sp.dtype in ("f16", "bf16") and sp.d_h in (64, 128)) or
                                (sp.dtype == "e4m3" and sp.d_h == 128))
    if tc_decode:
        return "gqa_cached_attn (decode_tc_kernel: tcgen05 split-K attention with fused merge)"
    if sp.dtype in ("f16", "bf16") and sp.d_h == 128:
        if rows <= 128:
            return "gqa_cached_attn (prefill_tc_kernel: tcgen05 chunk attention, wide form, one CTA per SM)"
        return "gqa_cached_attn (prefill_tc_kernel: tcgen05 chunk attention, narrow form, two CTAs per SM, split keys)"
    return "gqa_cached_attn (splitk_kernel: CUDA-core split-K attention)"


def workload_config(sp, note=None):
    import numpy as np
    if sp.mla:
        c = {"workload": sp.name, "L": sp.L, "B": sp.B, "heads": sp.H_q, "r": sp.d_h, "d_rope": sp.d_rope,
             "scale": sp.mla_scale, "T": sp.T, "cache_dtype": sp.dtype, "max_len": sp.max_len,
             "s_b": {"min": int(np.min(sp.lengths)), "mean": float(np.mean(sp.lengths)), "max": int(np.max(sp.lengths))},
             "l2": "no flush: the latent rows read per layer are larger than the 129 MB L2"}
        return c
    c = {"workload": sp.name, "L": sp.L, "B": sp.B, "H_q": sp.H_q, "H_kv": sp.H_kv, "d_h": sp.d_h,
         "T": sp.T, "cache_dtype": sp.dtype, "max_len": sp.max_len,
         "s_b": {"min": int(np.min(sp.lengths)), "mean": float(np.mean(sp.lengths)),
                 "max": int(np.max(sp.lengths))},
         "l2": "no flush: K/V read per layer is larger than the 129 MB L2"}
    if sp.rope_base:
        c["rope"] = {"base": sp.rope_base, "style": sp.rope_style,
                     "fused": "keys rotated in the append kernel, queries in the attention prologue"}
    if sp.block:
        c["paged"] = {"block": sp.block, "n_blocks": sp.B * (-(-sp.max_len // sp.block)),
                      "layout": "prefilled one block per sequence in turn: a sequence's blocks lie B apart"}
    if note:
        c["note"] = note
    return c


def run_ours(args):
    import torch
    import torch.distributed as dist

    import kvc_workloads
    from kv_cached_gqa_gb300 import _binding as kb

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    kb.load()
    sp = kvc_workloads.spec(args.workload)
    if args.layers:
        sp.L = args.layers
    wl = kvc_workloads.GpuWorkload(sp, device=f"cuda:{local}")
    if args.split_keys:
        kb.kvc_set_split_keys(wl.cache, args.split_keys)
    wl.prefill()
    inputs = wl.step_inputs(0)
    outs = [torch.empty((sp.B, sp.H_q, sp.T, sp.d_h), dtype=torch.float32, device=f"cuda:{local}")
            for _ in range(sp.L)]
    lengths = [int(x) for x in sp.lengths]
    stream = torch.cuda.current_stream()

    # --fused: one call per layer where the decode kernel stores the chunk itself (a single launch); the
    # other kernels would take the append kernel as a second launch, so they keep the two calls
    fused = args.fused and "decode_tc_kernel" in attention_kernel_name(sp)

    def layer_step(layer, qs, k, v, out, ev=None):
        """One layer: the chunk's append and its attention (one call with --fused); events, when
        given, bracket the attention call (the fused call, which includes the append)."""
        if not fused:
            wl.append(layer, k, v)
        if ev is not None:
            ev[0].record(stream)
        if fused:
            wl.append_attend(layer, k, v, qs, out=out)
        else:
            wl.attend(qs, layer, out=out)
        if ev is not None:
            ev[1].record(stream)

    def step(ev=None):
        for layer, (*qs, k, v) in enumerate(inputs):
            timed = ev is not None and layer % TIMED_EVERY == 0
            layer_step(layer, qs, k, v, outs[layer], ev[layer] if timed else None)
        kb.kvc_commit(wl.cache)
        kb.kvc_truncate_ragged(wl.cache, lengths)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        step()
    kb.kvc_status(wl.cache)
    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(sp.L)]
              for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph, graph_launches = None, 0
    if args.graph:
        # the step ends where it started (truncate back to s_b), so every replay does the same work
        graph = torch.cuda.CUDAGraph()
        before = kb.kvc_launch_count(wl.cache)
        with torch.cuda.graph(graph):
            step()
        graph_launches = kb.kvc_launch_count(wl.cache) - before
        graph.replay()
        torch.cuda.synchronize()
    launches0 = kb.kvc_launch_count(wl.cache)
    barrier()
    with ClockSampler(local) as clocks:
        t0.record(stream)
        for i in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                step(events[i])
        t1.record(stream)
        barrier()
    launches = kb.kvc_launch_count(wl.cache) - launches0 + graph_launches * args.steps
    kb.kvc_status(wl.cache)
    ms = t0.elapsed_time(t1) / args.steps
    if graph is not None:                  # kernel durations from a pass without the graph
        for i in range(args.steps):
            step(events[i])
        torch.cuda.synchronize()
        graph_ms = ms
    else:                                  # the same step replayed from one CUDA graph, for reference
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2):
            step()
        g2.replay()
        barrier()
        t0.record(stream)
        for i in range(args.steps):
            g2.replay()
        t1.record(stream)
        barrier()
        graph_ms = t0.elapsed_time(t1) / args.steps
        del g2
    attn_ms = [ev[l][0].elapsed_time(ev[l][1]) for ev in events for l in range(0, sp.L, TIMED_EVERY)]
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    ms, attn_avg_ms, graph_ms = max_over_ranks([ms, attn_avg_ms, graph_ms], f"cuda:{local}")

    # end to end through the public API with host buffers: every step copies every layer's inputs in
    # from pinned host memory and reads every layer's output back, inside the timed region. The copies
    # run on their own stream, as a serving loop would issue them: layer l + 1's inputs arrive while
    # layer l computes, and layer l's output leaves while layer l + 1 computes. Device buffers are
    # double-buffered across steps; events order every copy against the kernels that use its data.
    e2e = None
    if not args.no_e2e:
        host_in = [tuple(x.cpu().pin_memory() for x in trio) for trio in inputs]
        host_out = [[torch.empty_like(o, device="cpu").pin_memory() for o in outs] for _ in range(2)]
        dev_in = [[tuple(torch.empty_like(x) for x in trio) for trio in inputs] for _ in range(2)]
        dev_out = [[torch.empty_like(o) for o in outs] for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for trio in host_in for x in trio)
        d2h = sum(o.numel() * o.element_size() for o in host_out[0])
        copy_stream = torch.cuda.Stream()
        ev_in = [[torch.cuda.Event() for _ in range(sp.L)] for _ in range(2)]
        ev_done = [[torch.cuda.Event() for _ in range(sp.L)] for _ in range(2)]
        ev_set_free = [torch.cuda.Event() for _ in range(2)]
        n_step = [0]

        def e2e_step():
            st = n_step[0] % 2
            n_step[0] += 1
            copy_stream.wait_event(ev_set_free[st])          # the step that last used this set is done
            with torch.cuda.stream(copy_stream):
                for layer in range(sp.L):
                    for d_, h_ in zip(dev_in[st][layer], host_in[layer]):
                        d_.copy_(h_, non_blocking=True)
                    ev_in[st][layer].record(copy_stream)
            for layer in range(sp.L):
                stream.wait_event(ev_in[st][layer])
                *qs, k, v = dev_in[st][layer]
                layer_step(layer, qs, k, v, dev_out[st][layer])
                ev_done[st][layer].record(stream)
                copy_stream.wait_event(ev_done[st][layer])
                with torch.cuda.stream(copy_stream):
                    host_out[st][layer].copy_(dev_out[st][layer], non_blocking=True)
            kb.kvc_commit(wl.cache)
            kb.kvc_truncate_ragged(wl.cache, lengths)
            ev_set_free[st].record(copy_stream)              # after the step's last read-back
            stream.wait_event(ev_set_free[st])               # the step ends when its outputs are home

        for _ in range(max(3, args.warmup)):
            e2e_step()
        barrier()
        t0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        t1.record(stream)
        barrier()
        e2e_ms, = max_over_ranks([t0.elapsed_time(t1) / args.steps], f"cuda:{local}")
        e2e = {"value": round(job_rate(sp.step_bytes(), e2e_ms, world) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps_per_s": round(job_rate(1, e2e_ms, world), 3)}
    kb.kvc_status(wl.cache)

    if rank != 0:
        wl.close()
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0
    peak, peak_kind = measured_peaks()
    # the timed call's algorithmic bytes: the attention's, plus the chunk's append when it is fused in
    call_bytes = sp.attn_bytes() + (sp.append_bytes() if fused else 0)
    attn_gbs = call_bytes / (attn_avg_ms * 1e-3) / 1e9
    value = job_rate(sp.step_bytes(), ms, world) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline_entry(args.workload, args.cpu_sample_seconds)
    clk = clocks.summary()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": sp.dtype,
        "data": "synthetic (seeded Philox draws; approximately N(0,1))",
        "config": dict(workload_config(sp, None if not args.layers else "PROFILING CASE: fewer layers, not a bench line"),
                       graph=bool(args.graph),
                       layer_calls="gqa_cached_attn_append" if fused else "kvc_append + attention call"),
        "steps_per_s": round(job_rate(1, ms, world), 3),
        "graph_replay": {"value": round(job_rate(sp.step_bytes(), graph_ms, world) / 1e9, 2), "unit": "GB/s",
                         "ms_per_step": round(graph_ms, 4), "steps_per_s": round(job_rate(1, graph_ms, world), 3),
                         "note": "the same step captured once in a CUDA graph and replayed (no host launches)"},
        "pct_of_peak": {"measured_hbm": round(100 * value / world / peak, 2),
                        "nominal_8tbs": round(100 * value / world / 8000.0, 2)},
        "roofline": roofline_entry(sp, attn_avg_ms, attn_gbs, peak, peak_kind, args, fused, call_bytes),
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
    }
    print(json.dumps(line), flush=True)
    wl.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def roofline_entry(sp, attn_avg_ms, attn_gbs, peak, peak_kind, args, fused=False, call_bytes=None):
    """The attention kernel against its roofline: HBM GB/s, or dense tensor TFLOP/s when the call's
    arithmetic intensity (causal-counted flops per algorithmic byte) is above the ridge point."""
    t_sus, t_burst, t_kind = measured_tensor_peak()
    flops = sp.attn_flops()
    ridge = t_sus * 1e12 / (peak * 1e9)
    call = "gqa_cached_attn_append call (the chunk's append fused into the kernel)" if fused else "attention call"
    timing = f"CUDA events around the {call} of every {TIMED_EVERY}th layer" + (
        " (in a pass without the graph)" if args.graph else " inside the timed region")
    e = {"kernel": attention_kernel_name(sp)}
    call_bytes = call_bytes or sp.attn_bytes()
    if flops / call_bytes > ridge:
        tflops = flops / (attn_avg_ms * 1e-3) / 1e12
        e.update({"bound": "tensor", "achieved": round(tflops, 2), "peak": t_sus, "unit": "TFLOP/s",
                  "frac": round(tflops / t_sus, 4), "peak_source": f"{t_kind} bf16_tflops_sustained",
                  "frac_of_burst_peak": round(tflops / t_burst, 4),
                  "flops_per_launch": flops, "flops_counted": "causal: unmasked (query, key) pairs only",
                  "hbm_gbs": round(attn_gbs, 2)})
    else:
        e.update({"bound": "hbm", "achieved": round(attn_gbs, 2), "peak": peak, "unit": "GB/s",
                  "frac": round(attn_gbs / peak, 4), "peak_source": f"{peak_kind} hbm_gbs"})
    e.update({"bytes_per_launch": call_bytes, "launch_ms": round(attn_avg_ms, 5), "timing": timing,
              "traffic": traffic_per_launch(sp)})
    return e


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_sample_child is not None:
        cpu_sample_child(args.cpu_sample_child)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
