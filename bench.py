#!/usr/bin/env python
"""Benchmark of the KV-cache GQA attention step on the Qwen3-0.6B-shaped workload.

One benchmark step = one whole generation job through the C ABI:
  * prefill: fused QK-Norm+RoPE+cache append of 512 tokens into 28 layer caches, then causal
    flash prefill attention of all 28 layers, then the lm_head argmax;
  * 256 decode steps, each: one launch that appends the new token to the 28 layer caches and
    runs split-KV decode attention of the 28 layers over the valid prefix of the 1024-slot
    window, then the lm_head argmax (151936 x 1024 bf16).
Inputs are synthetic (seeded), resident in HBM; the job is captured once as a CUDA graph.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle instead (the only
reference implementation for this path) on a bounded sample of the same job.
"""
import os

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")     # the CPU oracle baseline runs single-threaded

import argparse
import hashlib
import json
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn KV GB/s + tokens/s; prefill-attn TFLOPS; % of GB300 roofline"
UNIT = "tokens/s"
LAYERS, PROMPT, STEPS, WINDOW = 28, 512, 256, 1024
HQ, HKV, D, HIDDEN, VOCAB = 16, 8, 128, 1024, 151936
TOKENS_PER_JOB = STEPS + 1          # one greedy token after prefill + one per decode step
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The part's nominal figures (HBM3e bandwidth, dense bf16 tensor rate), quoted beside the
# measured ones: every fraction is reported against both.
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}


# ----------------------------------------------------------------------------
# algorithmic work of one job
# ----------------------------------------------------------------------------
def append_bytes(tokens):
    # fp32 q, k, v in; bf16 q_out, k, v out
    return tokens * ((HQ + 2 * HKV) * D * 4 + (HQ + 2 * HKV) * D * 2)


def prefill_flops():
    return LAYERS * HQ * 4 * D * (PROMPT * (PROMPT + 1) // 2)


def decode_bytes(L):
    """One fused decode step over L valid slots (the new token's included): bf16 K and V rows
    read, fp32 q/k/v of the new token in, its bf16 K/V row written, fp32 attention out."""
    kv = LAYERS * HKV * L * D * 2 * 2
    return kv + LAYERS * ((HQ + 2 * HKV) * D * 4 + 2 * HKV * D * 2 + HQ * D * 4)


def prefill_min_bytes():
    """Bytes the prefill must move at least: bf16 q and the prompt's bf16 K/V rows in, fp32 out."""
    return LAYERS * PROMPT * (HQ * D * 2 + 2 * HKV * D * 2 + HQ * D * 4)


def lmhead_bytes(B=1):
    return VOCAB * HIDDEN * 2 + B * (HIDDEN * 4 + 4)


# ----------------------------------------------------------------------------
# distributed plumbing (one process per GPU, independent replicas: weak scaling)
# ----------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(value, world, device=None):
    """Max of a float over ranks (identity when world == 1)."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank, world, max_seconds):
    """Whole-job throughput: units processed by all ranks / the slowest rank's time."""
    return units_per_rank * world / max_seconds


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def gpu_smi_id(local_rank):
    """nvidia-smi identifier of CUDA device `local_rank` (its UUID: device indices differ from
    nvidia-smi's when CUDA_VISIBLE_DEVICES remaps them)."""
    try:
        import torch
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x for x in vis.split(",") if x.strip()]
        return ids[local_rank] if local_rank < len(ids) else str(local_rank)


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu, self.proc, self.file = gpu_index, None, None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush(); self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.count(",") >= 7]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0])); mx.append(float(r[1]))
            except ValueError:
                continue
            for name, val in zip(names, r[4:8]):
                if val.strip() == "Active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# the GPU job
# ----------------------------------------------------------------------------
class Qwen3Job:
    """Resident inputs, caches and workspaces of one generation job; `record(stream)` enqueues
    the job's 515 kernel launches (optionally bracketing each with timing events)."""

    def __init__(self, seed=0):
        import torch
        import kv_cache_gqa_gb300 as K
        self.K, self.torch = K, torch
        dev = "cuda"
        g = torch.Generator(device=dev); g.manual_seed(seed)
        rn = lambda *s: torch.randn(s, device=dev, generator=g)
        self.q, self.k, self.v = rn(LAYERS, PROMPT, HQ, D), rn(LAYERS, PROMPT, HKV, D), rn(LAYERS, PROMPT, HKV, D)
        self.dq, self.dk, self.dv = rn(STEPS, LAYERS, 1, HQ, D), rn(STEPS, LAYERS, 1, HKV, D), rn(STEPS, LAYERS, 1, HKV, D)
        self.qw = 1 + 0.1 * rn(LAYERS, D)
        self.kw = 1 + 0.1 * rn(LAYERS, D)
        self.h = rn(TOKENS_PER_JOB, 1, HIDDEN)
        self.W = (0.02 * rn(VOCAB, HIDDEN)).to(torch.bfloat16)
        self.kc = torch.zeros((LAYERS, HKV, WINDOW, D), device=dev, dtype=torch.bfloat16)
        self.vc = torch.zeros_like(self.kc)
        self.cache = K.KVCache(self.kc, self.vc)
        self.rope = K.Rope("1d", 1e6)
        self.q_pre = torch.empty((LAYERS, PROMPT, HQ, D), device=dev, dtype=torch.bfloat16)
        self.out_pre = torch.empty((LAYERS, PROMPT, HQ, D), device=dev)
        self.out_dec = torch.empty((STEPS, LAYERS, HQ, D), device=dev)
        self.pre_slot = np.arange(PROMPT, dtype=np.int32)[None]
        self.pre_slot_d = torch.from_numpy(self.pre_slot).to(dev)
        self.pre_pos_d = torch.arange(PROMPT, dtype=torch.int32, device=dev)[None, :, None].contiguous()
        self.step_slot_d = torch.arange(PROMPT, PROMPT + STEPS, dtype=torch.int32, device=dev).view(STEPS, 1, 1)
        self.len_host = [np.full(LAYERS, PROMPT + s + 1, np.int32) for s in range(STEPS)]
        self.len_d = torch.from_numpy(np.stack(self.len_host)).to(dev)
        self.ids = torch.empty((TOKENS_PER_JOB,), dtype=torch.int32, device=dev)
        self.dec_ws = torch.zeros(K.decode_workspace_bytes(LAYERS, HKV, HQ, WINDOW, D), dtype=torch.uint8, device=dev)
        self.lm_ws = torch.zeros(K.lmhead_workspace_bytes(1, HIDDEN), dtype=torch.uint8, device=dev)
        self.events = None
        self._calls = {}

    def step_calls(self):
        """The decode loop's C-ABI calls with their arguments marshalled once per input set
        (PreparedCall: each call still runs the library's validation, planning and launch; a
        serving loop holds its buffers, so converting tensors per call would only add host time).
        Made on the stream current at the first call of record()."""
        key = (id(self.dq), id(self.dk), id(self.dv), id(self.h))
        calls = self._calls.get(key)
        if calls is None:
            K, c = self.K, self.cache
            calls = [K.prepare_lmhead_argmax(self.h[0], self.W, self.ids[0:1], self.lm_ws)]
            for s in range(STEPS):
                calls.append(K.prepare_decode_step(
                    self.dq[s, :, 0], self.dk[s, :, 0], self.dv[s, :, 0], self.step_slot_d[s], c, self.len_d[s],
                    self.len_host[s], self.out_dec[s], self.dec_ws, self.rope, q_norm_w=self.qw, k_norm_w=self.kw,
                    eps=1e-6, norm_inst_stride=D))
                calls.append(K.prepare_lmhead_argmax(self.h[s + 1], self.W, self.ids[s + 1:s + 2], self.lm_ws))
            self._calls[key] = calls
        return calls

    def _ev(self, key):
        if self.events is not None:
            e = timing_event(self.torch, self.external_events)
            e.record()
            self.events.setdefault(key, []).append(e)

    external_events = True

    def record(self, with_events=False):
        K = self.K
        self.events = {} if with_events else None
        c = self.cache
        self._ev("t0")
        K.kv_cache_append_rope_qknorm(self.q, self.k, self.v, self.pre_pos_d, self.pre_slot_d, self.pre_slot, c,
                                      self.q_pre, self.rope, q_norm_w=self.qw, k_norm_w=self.kw, eps=1e-6,
                                      norm_inst_stride=D)
        self._ev("append_pre")
        K.kv_attn_prefill(self.q_pre, c, self.out_pre, mask="causal")
        self._ev("prefill")
        calls = self.step_calls()
        calls[0]()                                  # lmhead_argmax after the prompt
        self._ev("lm_head")
        for s in range(STEPS):
            calls[1 + 2 * s]()                      # kv_attn_decode_step
            self._ev("decode")
            calls[2 + 2 * s]()                      # lmhead_argmax
            self._ev("lm_head")

    def kernel_times_ms(self):
        """Per-kind launch durations (ms) of the last replay, from consecutive events."""
        order = ["t0", "append_pre", "prefill", "lm_head"] + ["decode", "lm_head"] * STEPS
        seq, idx = [], {}
        for key in order:
            i = idx.get(key, 0); idx[key] = i + 1
            seq.append((key, self.events[key][i]))
        out = {}
        for (k0, e0), (k1, e1) in zip(seq[:-1], seq[1:]):
            out.setdefault(k1, []).append(e0.elapsed_time(e1))
        return out


def events_in_graphs_supported(torch):
    """Timing events recorded inside a captured graph must be external event-record nodes."""
    import inspect
    try:
        return "external" in inspect.signature(torch.cuda.Event.__new__).parameters
    except (TypeError, ValueError):
        return False


def timing_event(torch, external):
    if external:
        return torch.cuda.Event(enable_timing=True, external=True)
    return torch.cuda.Event(enable_timing=True)


def graph_avg_ms(torch, stream, launch, n, reps=4):
    """Average duration of one launch: n launches captured in one graph, replayed `reps` times
    between two events on the launching stream (after one warm replay)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n):
            launch()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (n * reps)


def graph_seq_ms(torch, stream, fns, reps=4):
    """Average duration of one launch of the sequence `fns` (callables, each one launch),
    captured back to back in one graph and replayed `reps` times between two events on the
    launching stream (after one warm replay).  Launches that rotate over copies of their data
    whose total exceeds L2 read cold data, as inside a long job."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for f in fns:
            f()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (len(fns) * reps)


# FP32 FFMA peak of the SIMT (fp32-cache) paths: 152 SMs x 128 FMA lanes x 2 flop x 2.07 GHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def prefill_long_bench(torch, K, stream, bf16):
    """The tcgen05 prefill on long prompts: 2 instances x 4096 tokens, 16/8 heads, D = 128, bf16
    cache, causal and full masks (units of 32 key tiles, where the 512-token prompt's units hold
    1 to 4).  Graphs of launches alternating over two buffer sets (2 x 134 MB, larger than L2).
    Flops count visible pairs only: 4 D Hq per pair, S (S + 1) / 2 pairs per head when causal."""
    N, S = 2, 4096
    g = torch.Generator(device="cuda"); g.manual_seed(11)
    sets = []
    for _ in range(2):
        kc = torch.randn((N, HKV, S, D), device="cuda", generator=g).to(torch.bfloat16)
        vc = torch.randn_like(kc)
        q = torch.randn((N, S, HQ, D), device="cuda", generator=g).to(torch.bfloat16)
        sets.append((q, K.KVCache(kc, vc), torch.empty((N, S, HQ, D), device="cuda")))
    res = {"config": f"{N} instances x {S} tokens, {HQ}/{HKV} heads, D={D}, bf16 cache, fp32 out",
           "timing": "graphs of 8 launches alternating over 2 buffer sets (larger than L2)"}
    for mask in ("causal", "full"):
        fns = [(lambda st: (lambda: K.kv_attn_prefill(st[0], st[1], st[2], mask=mask)))(st) for st in sets]
        with torch.cuda.stream(stream):
            fns[0]()
        torch.cuda.synchronize()
        ms = graph_seq_ms(torch, stream, fns * 4, reps=4)
        pairs = S * (S + 1) // 2 if mask == "causal" else S * S
        flops = 4 * D * HQ * N * pairs
        tf = flops / (ms / 1e3) / 1e12
        res[mask] = {"us": round(ms * 1e3, 1), "flops": flops, "TFLOP/s": round(tf, 1),
                     "frac_bf16": round(tf / bf16, 4)}
    del sets
    return res


def decode_step_bench(torch, K, stream, job, copies=4):
    """kv_attn_decode_step alone as the job runs it (28 layer caches, 256 steps at L = 513..768,
    the job's inputs and per-layer norm weights), timed directly: one graph of the 256 launches,
    step s on cache copy s % copies (each copy 117 MB, so every launch reads its K/V from HBM as
    in the job, where the lm_head's 311 MB stream sits between two decode steps)."""
    g = torch.Generator(device="cuda"); g.manual_seed(21)
    caches = []
    for _ in range(copies):
        kc = torch.randn((LAYERS, HKV, WINDOW, D), device="cuda", generator=g).to(torch.bfloat16)
        vc = torch.randn((LAYERS, HKV, WINDOW, D), device="cuda", generator=g).to(torch.bfloat16)
        caches.append(K.KVCache(kc, vc))

    def step(s):
        return lambda: K.kv_attn_decode_step(job.dq[s, :, 0], job.dk[s, :, 0], job.dv[s, :, 0], job.step_slot_d[s],
                                             caches[s % copies], job.len_d[s], job.len_host[s], job.out_dec[s],
                                             job.dec_ws, job.rope, q_norm_w=job.qw, k_norm_w=job.kw, eps=1e-6,
                                             norm_inst_stride=D)
    fns = [step(s) for s in range(STEPS)]
    ms = graph_seq_ms(torch, stream, fns, reps=4)
    dec_bytes = [decode_bytes(PROMPT + s + 1) for s in range(STEPS)]
    del caches
    return {"avg_launch_us": round(ms * 1e3, 2), "algorithmic_bytes_per_launch": int(np.mean(dec_bytes)),
            "GB/s": round(np.mean(dec_bytes) / (ms / 1e3) / 1e9, 1),
            "timing": f"graph of the 256 launches of the job's decode loop (L = 513..768), step s on cache "
                      f"copy s % {copies} ({copies} x 117 MB, larger than L2), CUDA events around 4 replays"}


def configs_bench(torch, K, stream, hbm, bf16):
    """The other workloads' hot paths, each timed as a CUDA graph on the launching stream:
      tiny fp32 layer (latency: 64-token append + prefill, then 16 steps of append + decode);
      image-span prefill (xdRoPE, norm after RoPE, causal, 512 tokens) and its 64 decode steps;
      vision windowed attention (1288 patches, 16 heads, D = 72): window pass and full pass,
      bf16 and fp32 caches.
    Prefill and vision launches rotate over copies of their buffers larger than L2 in total."""
    import workloads as WL
    res = {}
    dv = lambda a, dt=None: (torch.from_numpy(np.ascontiguousarray(a)).cuda() if dt is None
                             else torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dt))

    # ---- 1. tiny fp32 single layer: prefill 64, 16 decode steps ----
    w = WL.tiny_fp32(0)
    W_, P_ = w["capacity"], w["n_prefill"]
    kc = torch.zeros((1, HKV, W_, D), device="cuda"); vc = torch.zeros_like(kc)
    cache = K.KVCache(kc, vc)
    rope = K.Rope("1d", w["base"])
    qw, kw = dv(w["q_norm_w"]), dv(w["k_norm_w"])
    q_all, k_all, v_all, pos_all = dv(w["q"][None]), dv(w["k"][None]), dv(w["v"][None]), dv(w["pos"][None])
    slot_h = np.arange(W_, dtype=np.int32)[None]
    slot_d = dv(slot_h)
    q_pre = torch.empty((1, P_, HQ, D), device="cuda"); o_pre = torch.empty_like(q_pre)
    q_dec = torch.empty((1, 1, HQ, D), device="cuda"); o_dec = torch.empty((W_ - P_, HQ, D), device="cuda")
    lens_h = [np.array([t + 1], np.int32) for t in range(W_)]
    lens_d = [dv(x) for x in lens_h]                 # one small tensor per step (aligned)
    pos_t = [dv(w["pos"][None, t:t + 1]) for t in range(W_)]
    slot_t = [dv(slot_h[:, t:t + 1]) for t in range(W_)]
    ws = torch.zeros(K.decode_workspace_bytes(1, HKV, HQ, W_, D), dtype=torch.uint8, device="cuda")

    def tiny_prefill():
        K.kv_cache_append_rope_qknorm(q_all[:, :P_], k_all[:, :P_], v_all[:, :P_], pos_all[:, :P_], slot_d[:, :P_],
                                      slot_h[:, :P_], cache, q_pre, rope, q_norm_w=qw, k_norm_w=kw, eps=w["eps"])
        K.kv_attn_prefill(q_pre, cache, o_pre, mask="causal")

    def tiny_run():
        tiny_prefill()
        for t in range(P_, W_):                      # fused append + decode, one launch per step
            K.kv_attn_decode_step(q_all[0, t:t + 1], k_all[0, t:t + 1], v_all[0, t:t + 1], pos_t[t][0], cache,
                                  lens_d[t], lens_h[t], o_dec[t - P_:t - P_ + 1], ws, rope, q_norm_w=qw, k_norm_w=kw,
                                  eps=w["eps"])
    with torch.cuda.stream(stream):
        tiny_run()
    torch.cuda.synchronize()
    run_ms = graph_seq_ms(torch, stream, [tiny_run], reps=20)
    pre_ms = graph_seq_ms(torch, stream, [tiny_prefill], reps=20)
    res["tiny_fp32"] = {
        "config": "1 layer, 16/8 heads, D=128, fp32 cache of 80 slots: 64-token append + causal prefill, then "
                  "16 fused append + decode steps (18 launches)",
        "run_us": round(run_ms * 1e3, 1), "prefill_phase_us": round(pre_ms * 1e3, 1),
        "decode_step_us": round((run_ms - pre_ms) * 1e3 / (W_ - P_), 2),
        "note": "latency-bound (17 MFLOP, ~3 MB): no roofline; the data stays in L2"}
    del kc, vc

    # ---- 3. image-span prefill and its 64 decode steps ----
    w = WL.image_span_prefill(0)
    S3, W3, steps3 = w["pos"].shape[0], w["capacity"], w["dq"].shape[0]
    rope3 = K.Rope("sections", w["base"], w["sections"])
    qw3, kw3 = dv(w["q_norm_w"]), dv(w["k_norm_w"])
    n3 = 16                                          # 16 copies x 10 MB (q, window K/V, output)
    kc3 = torch.zeros((n3, HKV, W3, D), device="cuda", dtype=torch.bfloat16); vc3 = torch.zeros_like(kc3)
    q3 = torch.empty((n3, S3, HQ, D), device="cuda", dtype=torch.bfloat16)
    o3 = torch.empty((n3, S3, HQ, D), device="cuda")
    c3 = [K.KVCache(kc3[i:i + 1], vc3[i:i + 1]) for i in range(n3)]
    sl3_h = np.arange(S3, dtype=np.int32)[None]
    sl3, pos3 = dv(sl3_h), dv(w["pos"][None])
    qi, ki, vi = dv(w["q"][None]), dv(w["k"][None]), dv(w["v"][None])
    app3 = lambda i: K.kv_cache_append_rope_qknorm(qi, ki, vi, pos3, sl3, sl3_h, c3[i], q3[i:i + 1], rope3,
                                                   q_norm_w=qw3, k_norm_w=kw3, eps=w["eps"], norm_after_rope=True)
    with torch.cuda.stream(stream):
        for i in range(n3):
            app3(i)
    torch.cuda.synchronize()
    pre3 = [(lambda i: (lambda: K.kv_attn_prefill(q3[i:i + 1], c3[i], o3[i:i + 1], mask="causal")))(i)
            for i in range(n3)]
    with torch.cuda.stream(stream):
        pre3[0]()
    torch.cuda.synchronize()
    pre3_ms = graph_seq_ms(torch, stream, pre3, reps=4)
    app3_ms = graph_seq_ms(torch, stream, [(lambda i: (lambda: app3(i)))(i) for i in range(n3)], reps=4)
    flops3 = 4 * D * HQ * (S3 * (S3 + 1) // 2)
    dq3, dk3, dv3, dpos3 = dv(w["dq"]), dv(w["dk"]), dv(w["dv"]), dv(w["dpos"])
    lens3_h = [np.array([S3 + s + 1], np.int32) for s in range(steps3)]
    lens3_d = [dv(x) for x in lens3_h]
    o3d = torch.empty((steps3, HQ, D), device="cuda")
    ws3 = torch.zeros(K.decode_workspace_bytes(1, HKV, HQ, W3, D), dtype=torch.uint8, device="cuda")
    dec3 = [(lambda s: (lambda: K.kv_attn_decode_step(
        dq3[s:s + 1], dk3[s:s + 1], dv3[s:s + 1], dpos3[s:s + 1], c3[0], lens3_d[s], lens3_h[s], o3d[s:s + 1],
        ws3, rope3, q_norm_w=qw3, k_norm_w=kw3, eps=w["eps"], norm_after_rope=True)))(s) for s in range(steps3)]
    with torch.cuda.stream(stream):
        dec3[0]()
    torch.cuda.synchronize()
    dec3_ms = graph_seq_ms(torch, stream, dec3, reps=4)
    dec3_bytes = sum(HKV * (S3 + s + 1) * D * 2 * 2 + (HQ + 2 * HKV) * D * 4 + 2 * HKV * D * 2 + HQ * D * 4
                     for s in range(steps3)) / steps3
    pre3_tf = flops3 / (pre3_ms / 1e3) / 1e12
    res["image_span"] = {
        "config": f"1 layer, {S3} tokens (20 text + 274 image rows + 218 text), 4-axis xdRoPE [16,16,16,16] base "
                  f"1.11588e7, norm after RoPE, causal, 16/8 heads, D=128, bf16 window of {W3}; then {steps3} fused "
                  f"decode steps (L = {S3 + 1}..{S3 + steps3})",
        "prefill_us": round(pre3_ms * 1e3, 2), "prefill_TFLOP/s": round(pre3_tf, 1),
        "prefill_frac_bf16": round(pre3_tf / bf16, 4), "prefill_flops": flops3,
        "append_us": round(app3_ms * 1e3, 2),
        "append_GB/s": round(append_bytes(S3) / (app3_ms / 1e3) / 1e9, 1),
        "decode_step_us": round(dec3_ms * 1e3, 2),
        "decode_GB/s": round(dec3_bytes / (dec3_ms / 1e3) / 1e9, 1),
        "decode_frac_hbm": round(dec3_bytes / (dec3_ms / 1e3) / 1e9 / hbm, 4),
        "timing": "prefill and append: graphs of 16 launches over 16 buffer copies (160 MB); decode: graph of "
                  "the 64 steps (one layer, ~2.3 MB per step: launch-latency bound, read from L2)"}
    del kc3, vc3, q3, o3

    # ---- 4. vision windowed attention: window pass and full pass, bf16 and fp32 ----
    w = WL.vision_windowed(0)
    lay = w["layout"]
    S4, H4, D4 = lay.pos_rc.shape[0], WL.VISION_HEADS, WL.VISION_HEAD_DIM
    seg_sizes = np.bincount(lay.segment)
    flops_win = int(4 * D4 * H4 * int(np.sum(seg_sizes.astype(np.int64) ** 2)))
    flops_full = 4 * D4 * H4 * S4 * S4
    seg_d, ros_d = dv(lay.segment), dv(lay.row_of_slot)
    sl4_h = lay.slot[None]
    sl4, pos4 = dv(sl4_h), dv(lay.pos_rc[None])
    qi4, ki4, vi4 = dv(w["q"][None]), dv(w["k"][None]), dv(w["v"][None])
    rope4 = K.Rope("2d", w["base"])
    vis = {}
    for name, tdt in (("bf16", torch.bfloat16), ("f32", torch.float32)):
        n4 = 10                                      # 10 copies: 148 MB (bf16) / 237 MB (fp32)
        kc4 = torch.zeros((n4, H4, S4, D4), device="cuda", dtype=tdt); vc4 = torch.zeros_like(kc4)
        q4 = torch.empty((n4, S4, H4, D4), device="cuda", dtype=tdt)
        o4 = torch.empty((n4, S4, H4, D4), device="cuda")
        c4 = [K.KVCache(kc4[i:i + 1], vc4[i:i + 1]) for i in range(n4)]
        with torch.cuda.stream(stream):
            for i in range(n4):
                K.kv_cache_append_rope_qknorm(qi4, ki4, vi4, pos4, sl4, sl4_h, c4[i], q4[i:i + 1], rope4)
        torch.cuda.synchronize()
        win = [(lambda i: (lambda: K.kv_attn_prefill(q4[i:i + 1], c4[i], o4[i:i + 1], mask="segment", segment=seg_d,
                                                     segment_host=lay.segment, row_of_slot=ros_d)))(i)
               for i in range(n4)]
        full = [(lambda i: (lambda: K.kv_attn_prefill(q4[i:i + 1], c4[i], o4[i:i + 1], mask="full",
                                                      row_of_slot=ros_d)))(i) for i in range(n4)]
        with torch.cuda.stream(stream):
            win[0](); full[0]()
        torch.cuda.synchronize()
        win_ms = graph_seq_ms(torch, stream, win, reps=4)
        full_ms = graph_seq_ms(torch, stream, full, reps=4)
        peak = bf16 if name == "bf16" else FP32_ALU_TFLOPS
        tw, tf = flops_win / (win_ms / 1e3) / 1e12, flops_full / (full_ms / 1e3) / 1e12
        vis[name] = {"window_us": round(win_ms * 1e3, 2), "window_TFLOP/s": round(tw, 2),
                     "window_frac": round(tw / peak, 4), "full_us": round(full_ms * 1e3, 2),
                     "full_TFLOP/s": round(tf, 2), "full_frac": round(tf / peak, 4),
                     "peak_TFLOP/s": round(peak, 1),
                     "peak": "measured bf16 dense (tensor cores)" if name == "bf16" else
                             "FP32 FFMA: 152 SMs x 128 lanes x 2 flop x 2.07 GHz (derived)"}
        del kc4, vc4, q4, o4
    res["vision"] = dict(vis, config=f"{S4} patches (14x92 grid, windows of 8x8 merged 2x2 groups: "
                                     f"{'/'.join(str(int(x)) for x in seg_sizes)} patches), {H4} heads = KV heads, "
                                     f"D={D4}, 2D RoPE, bidirectional; window pass (block-diagonal) and full pass",
                         window_flops=flops_win, full_flops=flops_full,
                         timing="graphs of 10 launches over 10 buffer copies (larger than L2)")
    return res


VERIFY_B, VERIFY_L, VERIFY_K = 64, 2048, 16


def verify_bench(torch, K, stream):
    """Average duration of kv_attn_verify on VERIFY_B sequences of VERIFY_L valid slots with
    VERIFY_K-token blocks (Qwen3 heads), as a graph of 8 back-to-back launches."""
    B, L, k = VERIFY_B, VERIFY_L, VERIFY_K
    g = torch.Generator(device="cuda"); g.manual_seed(7)
    kc = torch.randn((B, HKV, L, D), device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn((B, HKV, L, D), device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn((B, k, HQ, D), device="cuda", generator=g).to(torch.bfloat16)
    out = torch.empty((B, k, HQ, D), device="cuda")
    lengths = np.full(B, L, np.int32)
    ld = torch.from_numpy(lengths).cuda()
    ws = torch.zeros(K.verify_workspace_bytes(B, HKV, HQ, k, L, D), dtype=torch.uint8, device="cuda")
    cache = K.KVCache(kc, vc)
    with torch.cuda.stream(stream):
        K.kv_attn_verify(q, cache, ld, lengths, out, ws)          # configures the kernel before capture
    torch.cuda.synchronize()
    ms = graph_avg_ms(torch, stream, lambda: K.kv_attn_verify(q, cache, ld, lengths, out, ws), 8, reps=2)
    kv_bytes = B * HKV * L * D * 2 * 2
    io_bytes = B * k * HQ * D * (2 + 4)
    del kc, vc
    return {"config": f"{B} sequences x {L} slots, {k}-token blocks, {HQ}/{HKV} heads, D={D}, bf16 cache",
            "avg_launch_us": round(ms * 1e3, 2), "algorithmic_bytes_per_launch": kv_bytes + io_bytes,
            "GB/s": round((kv_bytes + io_bytes) / (ms / 1e3) / 1e9, 1),
            "block_tokens_per_s": round(B * k / (ms / 1e3), 1)}


def serving_bench(torch, K, stream, W, lm_ws_bytes, batch=None):
    """The batched serving step: 64 sequences with contexts uniform in [1024, 32768] (the same
    seeded draw as the parity tests), capacity ctx + 128; one step = the fused append + decode
    over all 64 caches and the batched lm_head argmax.  Caches are random bf16 (contents do not
    change the work).  Timed as a graph of 8 back-to-back steps at the first step's lengths.
    `batch` keeps only the first sequences of the draw (a smaller case for counter captures)."""
    import workloads as WL
    ctx = WL.serving_contexts(0)
    if batch is not None:
        ctx = ctx[:batch]
    B, cap = ctx.size, int(ctx.max()) + 128
    g = torch.Generator(device="cuda"); g.manual_seed(11)
    kc = torch.randn((B, HKV, cap, D), device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn((B, HKV, cap, D), device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn((B, HQ, D), device="cuda", generator=g)
    k = torch.randn((B, HKV, D), device="cuda", generator=g)
    v = torch.randn((B, HKV, D), device="cuda", generator=g)
    h = torch.randn((B, HIDDEN), device="cuda", generator=g)
    qw = 1 + 0.1 * torch.randn((D,), device="cuda", generator=g)
    kw = 1 + 0.1 * torch.randn((D,), device="cuda", generator=g)
    lengths = (ctx + 1).astype(np.int32)
    ld = torch.from_numpy(lengths).cuda()
    pos = torch.from_numpy(ctx.reshape(B, 1).astype(np.int32)).cuda()
    out = torch.empty((B, HQ, D), device="cuda")
    ids = torch.empty((B,), dtype=torch.int32, device="cuda")
    dws = torch.zeros(K.decode_workspace_bytes(B, HKV, HQ, cap, D), dtype=torch.uint8, device="cuda")
    lws = torch.zeros(K.lmhead_workspace_bytes(B, HIDDEN), dtype=torch.uint8, device="cuda")
    cache, rope = K.KVCache(kc, vc), K.Rope("1d", 1e6)
    dec = lambda: K.kv_attn_decode_step(q, k, v, pos, cache, ld, lengths, out, dws, rope, q_norm_w=qw, k_norm_w=kw)
    lmh = lambda: K.lmhead_argmax(h, W, ids, lws)
    with torch.cuda.stream(stream):
        dec(); lmh()                                   # configure the kernels before capture
    torch.cuda.synchronize()
    dec_ms = graph_avg_ms(torch, stream, dec, 8, reps=2)
    lm_ms = graph_avg_ms(torch, stream, lmh, 8, reps=2)
    step_ms = graph_avg_ms(torch, stream, lambda: (dec(), lmh()), 8, reps=2)
    kv_bytes = int(lengths.sum()) * HKV * D * 2 * 2
    dec_bytes = kv_bytes + B * ((HQ + 2 * HKV) * D * 4 + 2 * HKV * D * 2 + HQ * D * 4)
    del kc, vc
    return {"config": f"{B} sequences, contexts {int(ctx.min())}..{int(ctx.max())} (sum {int(ctx.sum())}), "
                      f"{HQ}/{HKV} heads, D={D}, bf16 caches; step = fused append+decode + lm_head (B={B})",
            "step_us": round(step_ms * 1e3, 1), "tokens_per_s": round(B / (step_ms / 1e3), 1),
            "decode_step_us": round(dec_ms * 1e3, 1), "decode_GB/s": round(dec_bytes / (dec_ms / 1e3) / 1e9, 1),
            "decode_algorithmic_bytes": dec_bytes,
            "lm_head_us": round(lm_ms * 1e3, 1),
            "lm_head_GB/s": round((VOCAB * HIDDEN * 2) / (lm_ms / 1e3) / 1e9, 1)}


MLA_LAYERS, MLA_H, MLA_W, MLA_DK, MLA_DV = 40, 32, 512, 192, 128


def mla_bench(torch, K, stream):
    """The asymmetric MLA-expanded cache of a 40-layer model (K rows 192 wide, V rows 128, 32 heads,
    a 512-slot window, interleaved RoPE on the last 64 K dims): the prompt phase (per layer: append
    512 bf16 tokens, causal prefill over them) and one decode token (per layer: append, decode over
    the full 512-slot window), each as a graph of all 40 layers back to back; plus the decode kernel
    alone on 16 sequences x 32 heads x 4096 slots, a cache larger than L2, for its bandwidth."""
    Lr, H, W, DKm, DVm = MLA_LAYERS, MLA_H, MLA_W, MLA_DK, MLA_DV
    g = torch.Generator(device="cuda"); g.manual_seed(13)
    bf = torch.bfloat16
    kc = torch.zeros((Lr, H, W, DKm), device="cuda", dtype=bf)
    vc = torch.zeros((Lr, H, W, DVm), device="cuda", dtype=bf)
    caches = [K.KVCache(kc[l:l + 1], vc[l:l + 1]) for l in range(Lr)]
    rope = K.Rope("interleaved", 1e6, rot_offset=128, rot_dim=64)
    q = torch.randn((1, W, H, DKm), device="cuda", generator=g).to(bf)
    k = torch.randn((1, W, H, DKm), device="cuda", generator=g).to(bf)
    v = torch.randn((1, W, H, DVm), device="cuda", generator=g).to(bf)
    pos = torch.arange(W, dtype=torch.int32, device="cuda").view(1, W, 1)
    slot_h = np.arange(W, dtype=np.int32).reshape(1, W)
    slot = torch.from_numpy(slot_h).cuda()
    q_out = torch.empty((1, W, H, DKm), device="cuda", dtype=bf)
    out = torch.empty((1, W, H, DVm), device="cuda")

    def prompt():
        for c in caches:
            K.kv_cache_append_rope_qknorm(q, k, v, pos, slot, slot_h, c, q_out, rope)
            K.kv_attn_prefill(q_out, c, out, mask="causal")

    qn, kn, vn = q[:, :1].contiguous(), k[:, :1].contiguous(), v[:, :1].contiguous()
    pn = torch.full((1, 1, 1), W - 1, dtype=torch.int32, device="cuda")
    sn_h = np.full((1, 1), W - 1, np.int32)
    sn = torch.from_numpy(sn_h).cuda()
    lens_h = np.array([W], np.int32)
    lens = torch.from_numpy(lens_h).cuda()
    qo = torch.empty((1, 1, H, DKm), device="cuda", dtype=bf)
    o = torch.empty((1, H, DVm), device="cuda")
    ws = torch.zeros(K.decode_workspace_bytes(1, H, H, W, DVm), dtype=torch.uint8, device="cuda")

    def token():                                     # fused append + decode per layer
        for c in caches:
            K.kv_attn_decode_step(qn[0], kn[0], vn[0], pn[0], c, lens, lens_h, o, ws, rope)

    B2, L2 = 16, 4096
    kb = torch.randn((B2, H, L2, DKm), device="cuda", generator=g).to(bf)
    vb = torch.randn((B2, H, L2, DVm), device="cuda", generator=g).to(bf)
    qb = torch.randn((B2, H, DKm), device="cuda", generator=g).to(bf)
    ob = torch.empty((B2, H, DVm), device="cuda")
    lb_h = np.full(B2, L2, np.int32)
    lb = torch.from_numpy(lb_h).cuda()
    wsb = torch.zeros(K.decode_workspace_bytes(B2, H, H, L2, DVm), dtype=torch.uint8, device="cuda")
    cb = K.KVCache(kb, vb)
    big = lambda: K.kv_attn_decode(qb, cb, lb, lb_h, ob, wsb)
    with torch.cuda.stream(stream):
        prompt(); token(); big()                       # configure the kernels before capture
    torch.cuda.synchronize()
    prompt_ms = graph_avg_ms(torch, stream, prompt, 1, reps=4)
    token_ms = graph_avg_ms(torch, stream, token, 2, reps=4)
    big_ms = graph_avg_ms(torch, stream, big, 8, reps=2)
    big_bytes = B2 * H * L2 * (DKm + DVm) * 2 + B2 * H * (DKm * 2 + DVm * 4)
    tok_bytes = Lr * H * W * (DKm + DVm) * 2
    del kb, vb, kc, vc
    return {"config": f"{Lr} layers, {H}/{H} heads, K {DKm} / V {DVm}, {W}-slot bf16 window, interleaved RoPE "
                      f"on dims 128..191; prompt = {W} tokens (append + causal prefill per layer), token = one "
                      f"decode step at the full window (one fused append + decode launch per layer)",
            "prompt_ms": round(prompt_ms, 3), "prompt_tokens_per_s": round(W / (prompt_ms / 1e3), 1),
            "token_us": round(token_ms * 1e3, 1), "token_per_layer_us": round(token_ms * 1e3 / Lr, 2),
            "token_cache_GB/s": round(tok_bytes / (token_ms / 1e3) / 1e9, 1),
            "decode_16x4096_us": round(big_ms * 1e3, 1),
            "decode_16x4096_GB/s": round(big_bytes / (big_ms / 1e3) / 1e9, 1),
            "decode_16x4096_algorithmic_bytes": big_bytes}


def run_only(args, torch, K):
    """One sub-benchmark alone (for counter captures of its kernels); prints its own JSON line."""
    stream = torch.cuda.Stream()
    if args.only == "verify":
        res = verify_bench(torch, K, stream)
    elif args.only == "mla":
        res = mla_bench(torch, K, stream)
    elif args.only == "lm64":                        # the batched lm_head alone, 64 hidden rows
        g = torch.Generator(device="cuda"); g.manual_seed(3)
        W = (torch.randn((VOCAB, HIDDEN), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        h = torch.randn((64, HIDDEN), device="cuda", generator=g)
        ids = torch.empty((64,), dtype=torch.int32, device="cuda")
        lws = torch.zeros(K.lmhead_workspace_bytes(64, HIDDEN), dtype=torch.uint8, device="cuda")
        with torch.cuda.stream(stream):
            K.lmhead_argmax(h, W, ids, lws)          # configures the kernel before capture
        torch.cuda.synchronize()
        ms = graph_avg_ms(torch, stream, lambda: K.lmhead_argmax(h, W, ids, lws), 8, reps=2)
        res = {"lm_head_b64_us": round(ms * 1e3, 2), "GB/s": round(VOCAB * HIDDEN * 2 / (ms / 1e3) / 1e9, 1)}
    elif args.only == "configs":                     # tiny fp32, image span and vision workloads
        peaks, _ = load_peaks()
        res = configs_bench(torch, K, stream, float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                            float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])))
    elif args.only == "prefill_long":
        peaks, _ = load_peaks()
        res = prefill_long_bench(torch, K, stream, float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])))
    elif args.only == "topk":                        # final RMSNorm + lm_head, top 1 and top 8, batch 1
        g = torch.Generator(device="cuda"); g.manual_seed(3)
        W = (torch.randn((VOCAB, HIDDEN), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        h = torch.randn((1, HIDDEN), device="cuda", generator=g)
        fn_w = 1 + 0.1 * torch.randn(HIDDEN, device="cuda", generator=g)
        ws = torch.zeros(K.lmhead_topk_workspace_bytes(1, HIDDEN, VOCAB, 8), dtype=torch.uint8, device="cuda")
        ids1 = torch.empty((1, 1), dtype=torch.int32, device="cuda")
        ids8 = torch.empty((1, 8), dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            K.lmhead_topk(h, W, ids8, ws, norm_w=fn_w)   # configures the kernels before capture
        torch.cuda.synchronize()
        ms1 = graph_avg_ms(torch, stream, lambda: K.lmhead_topk(h, W, ids1, ws, norm_w=fn_w), 8, reps=2)
        ms8 = graph_avg_ms(torch, stream, lambda: K.lmhead_topk(h, W, ids8, ws, norm_w=fn_w), 8, reps=2)
        res = {"top1_us": round(ms1 * 1e3, 2), "top8_us": round(ms8 * 1e3, 2)}
    else:                                            # serving16: the first 16 sequences of the draw
        g = torch.Generator(device="cuda"); g.manual_seed(3)
        W = (torch.randn((VOCAB, HIDDEN), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        res = serving_bench(torch, K, stream, W, None, batch=16)
    print(json.dumps({"case": args.only, "result": res}), flush=True)


def run_gpu(args, rank, world, local_rank):
    import torch
    import kv_cache_gqa_gb300 as K
    torch.cuda.set_device(local_rank)
    if args.only:
        if rank == 0:
            run_only(args, torch, K)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    job = Qwen3Job(seed=rank)
    stream = torch.cuda.Stream()
    # eager warm-up (also initialises every kernel's attributes before capture)
    with torch.cuda.stream(stream):
        job.record()
    torch.cuda.synchronize()
    in_graph_events = events_in_graphs_supported(torch)
    n0 = K.launch_count()
    graph = torch.cuda.CUDAGraph()              # the timed job: kernels only
    with torch.cuda.graph(graph, stream=stream):
        job.record()
    launches_per_job = K.launch_count() - n0
    graph_ev = None                             # the same job with an event node after every launch
    if in_graph_events:
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev, stream=stream):
            job.record(with_events=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(gpu_smi_id(local_rank))
    clocks.start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(args.steps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = start.elapsed_time(end)
    max_ms = reduce_max(ms, world, device=torch.device("cuda", local_rank))
    value = aggregate_throughput(TOKENS_PER_JOB * args.steps, world, max_ms / 1e3)
    if args.job_only:                       # counter captures: the timed job and nothing else
        if rank == 0:
            print(json.dumps({"case": "job_only", "ms_per_step": round(max_ms / args.steps, 4),
                              "value": round(value, 1), "unit": UNIT}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    if in_graph_events:                     # per-kernel times: one replay of the instrumented graph
        with torch.cuda.stream(stream):
            graph_ev.replay()
        torch.cuda.synchronize()
        kt = job.kernel_times_ms()
        kt_source = ("CUDA event nodes between the launches of one replay of the job graph, right after the "
                     "timed region (the timed replays carry no event nodes)")
    else:                                   # this torch cannot time inside a graph: one eager job
        job.external_events = False
        with torch.cuda.stream(stream):
            job.record(with_events=True)
        torch.cuda.synchronize()
        kt = job.kernel_times_ms()
        kt_source = "CUDA events around an eager replay of one job right after the timed region"

    # the dominant kernel alone: 32 back-to-back launches in one graph (its 311 MB table is larger
    # than L2, so every launch streams it from HBM as inside the job)
    lm_iso_ms = graph_avg_ms(torch, stream, lambda: K.lmhead_argmax(job.h[1], job.W, job.ids[1:2], job.lm_ws), 32)
    # the same with the final RMSNorm fused in front (top 1), and the 8 best ids (logits + ranking)
    fn_w = 1 + 0.1 * torch.randn(HIDDEN, device="cuda")
    tk_ws = torch.zeros(K.lmhead_topk_workspace_bytes(1, HIDDEN, VOCAB, 8), dtype=torch.uint8, device="cuda")
    tk_ids1 = torch.empty((1, 1), dtype=torch.int32, device="cuda")
    tk_ids8 = torch.empty((1, 8), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        K.lmhead_topk(job.h[1], job.W, tk_ids8, tk_ws, norm_w=fn_w)   # configures the kernels before capture
    torch.cuda.synchronize()
    lm_norm_ms = graph_avg_ms(torch, stream, lambda: K.lmhead_topk(job.h[1], job.W, tk_ids1, tk_ws, norm_w=fn_w), 32)
    # the prompt's append and prefill alone, each as a graph of back-to-back launches (inputs
    # and outputs larger than L2); the in-job figures above also carry an event node's latency
    app_iso_ms = graph_avg_ms(torch, stream, lambda: K.kv_cache_append_rope_qknorm(
        job.q, job.k, job.v, job.pre_pos_d, job.pre_slot_d, job.pre_slot, job.cache, job.q_pre, job.rope,
        q_norm_w=job.qw, k_norm_w=job.kw, eps=1e-6, norm_inst_stride=D), 8)
    pre_iso_ms = graph_avg_ms(torch, stream, lambda: K.kv_attn_prefill(job.q_pre, job.cache, job.out_pre,
                                                                        mask="causal"), 8)
    lm_top8_ms = graph_avg_ms(torch, stream, lambda: K.lmhead_topk(job.h[1], job.W, tk_ids8, tk_ws, norm_w=fn_w), 32)

    # speculative-decoding verify block on a cache larger than L2: 64 sequences x 2048 slots,
    # 16-token blocks (each launch streams 537 MB of K/V once for all 16 block rows)
    vb = verify_bench(torch, K, stream)
    sv = serving_bench(torch, K, stream, job.W, None)
    mla = mla_bench(torch, K, stream)
    ds = decode_step_bench(torch, K, stream, job)
    peaks0, _ = load_peaks()
    pl = prefill_long_bench(torch, K, stream, float(peaks0.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])))
    cfg = configs_bench(torch, K, stream, float(peaks0.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                        float(peaks0.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])))

    # ---- end to end: inputs from pinned host memory, ids back to the host, every step ----
    # Two device input sets, each with its own graph of the job: step i copies its inputs into
    # set i % 2 on a copy stream (once the graph that last read that set is done) while the
    # previous step's graph runs, then replays the graph reading that set and reads the ids back.
    names = ("q", "k", "v", "dq", "dk", "dv", "h")
    host_in = {n: getattr(job, n).cpu().pin_memory() for n in names}
    ids_host = torch.empty_like(job.ids, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = ids_host.numel() * ids_host.element_size()
    dev_sets = [{n: getattr(job, n) for n in names}, {n: torch.empty_like(getattr(job, n)) for n in names}]
    for n in names:
        setattr(job, n, dev_sets[1][n])
    graph_b = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_b, stream=stream):
        job.record()
    for n in names:
        setattr(job, n, dev_sets[0][n])
    graphs = [graph, graph_b]
    copy_stream = torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_step(i):
        j = i % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(done[j])             # the graph that last read set j has finished
            for n in names:
                dev_sets[j][n].copy_(host_in[n], non_blocking=True)
            ready[j].record(copy_stream)
        stream.wait_event(ready[j])
        graphs[j].replay()
        done[j].record(stream)
        ids_host.copy_(job.ids, non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(max(2, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_event(e0)                      # the timed copies start after e0
        for i in range(args.steps):
            e2e_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), world, device=torch.device("cuda", local_rank))
    e2e_value = aggregate_throughput(TOKENS_PER_JOB * args.steps, world, e2e_ms / 1e3)

    # ---- end to end, eager: the same copies, and every step calls the four entry points through the
    # C ABI (515 calls: host validation, planning and launch each time; the Python-side argument
    # marshalling of the decode loop is done once per input set), no graph ----
    def e2e_eager_step(i):
        j = i % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(done[j])
            for n in names:
                dev_sets[j][n].copy_(host_in[n], non_blocking=True)
            ready[j].record(copy_stream)
        stream.wait_event(ready[j])
        for n in names:
            setattr(job, n, dev_sets[j][n])
        job.record()
        done[j].record(stream)
        ids_host.copy_(job.ids, non_blocking=True)

    n_eager0 = K.launch_count()
    with torch.cuda.stream(stream):
        for i in range(max(2, args.warmup)):
            e2e_eager_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0.record(stream)
        copy_stream.wait_event(e0)
        n_eager0 = K.launch_count()
        t_host0 = time.perf_counter()
        for i in range(args.steps):
            e2e_eager_step(i)
        t_host = time.perf_counter() - t_host0
        e1.record(stream)
        torch.cuda.synchronize()
    eager_launches = K.launch_count() - n_eager0
    for n in names:
        setattr(job, n, dev_sets[0][n])
    eager_ms = reduce_max(e0.elapsed_time(e1), world, device=torch.device("cuda", local_rank))
    eager_value = aggregate_throughput(TOKENS_PER_JOB * args.steps, world, eager_ms / 1e3)

    if rank == 0:
        peaks, peak_src = load_peaks()
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        bf16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        # The decode step is timed directly (a graph of the job's 256 launches over rotating cache
        # copies); the difference of the job and its other kernels is kept beside it as a check.
        totals = {k: sum(v) for k, v in kt.items()}
        job_ms = max_ms / args.steps
        in_job = {"lm_head": lm_iso_ms, "prefill": kt["prefill"][0], "append_pre": kt["append_pre"][0],
                  "decode": ds["avg_launch_us"] / 1e3}
        dec_by_diff_ms = (job_ms - in_job["prefill"] - in_job["append_pre"] - TOKENS_PER_JOB * lm_iso_ms) / STEPS
        dec_bytes = [decode_bytes(PROMPT + s + 1) for s in range(STEPS)]
        dec_gbs = np.mean(dec_bytes) / (in_job["decode"] / 1e3) / 1e9
        lm_gbs = lmhead_bytes() / (lm_iso_ms / 1e3) / 1e9
        pre_tf = prefill_flops() / (in_job["prefill"] / 1e3) / 1e12
        app_gbs = append_bytes(LAYERS * PROMPT) / (in_job["append_pre"] / 1e3) / 1e9
        job_bytes = (append_bytes(LAYERS * PROMPT) + prefill_min_bytes() + float(np.sum(dec_bytes))
                     + TOKENS_PER_JOB * lmhead_bytes())
        dominant = max(totals, key=totals.get)
        roof = {"kernel": "lmhead_argmax", "bound": "hbm", "achieved": round(lm_gbs, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(lm_gbs / hbm, 4), "traffic": lm_traffic(),
                "algorithmic_bytes_per_launch": lmhead_bytes(), "avg_launch_us": round(lm_iso_ms * 1e3, 2),
                "timing": "CUDA events around a graph of 32 back-to-back launches on the launching stream",
                "peak_source": f"{peak_src} hbm_gbs"}
        if dominant == "decode":
            roof.update({"kernel": "kv_attn_decode_step", "achieved": round(dec_gbs, 1),
                         "frac": round(dec_gbs / hbm, 4), "traffic": None,
                         "algorithmic_bytes_per_launch": int(np.mean(dec_bytes)),
                         "avg_launch_us": round(in_job["decode"] * 1e3, 2), "timing": ds["timing"]})
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": job_config(),
            "e2e": {"value": round(eager_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h),
                    "leg": "eager C-ABI calls",
                    "copies": "each step's inputs copied from pinned host memory on a copy stream while "
                              "the previous step runs (two device input sets); ids read back after every step",
                    "legs": {
                        "eager_c_abi": {"value": round(eager_value, 1), "ms_per_step": round(eager_ms / args.steps, 3),
                                        "host_ms_per_step": round(t_host * 1e3 / args.steps, 3),
                                        "launches_per_step": int(eager_launches // args.steps),
                                        "what": "every step calls the four entry points through the C ABI "
                                                "(515 calls, host validation, planning and launch each time; "
                                                "the decode loop's Python marshalling done once per input set), "
                                                "no graph"},
                        "graph_replay": {"value": round(e2e_value, 1), "ms_per_step": round(e2e_ms / args.steps, 3),
                                         "what": "the job captured once through the same calls, replayed as one "
                                                 "CUDA graph per step"}}},
            "gpu_launches": int(launches_per_job * args.steps),
            "roofline": roof,
            "kernels": {
                "decode_step": {"GB/s": round(dec_gbs, 1), "frac_hbm": round(dec_gbs / hbm, 4),
                                "avg_launch_us": round(in_job["decode"] * 1e3, 2),
                                "algorithmic_bytes_per_launch": int(np.mean(dec_bytes)), "timing": ds["timing"],
                                "by_difference_us": round(dec_by_diff_ms * 1e3, 2)},
                "prefill_attn": {"TFLOP/s": round(pre_tf, 2), "frac_bf16": round(pre_tf / bf16, 4),
                                 "launch_us": round(in_job["prefill"] * 1e3, 1), "flops": prefill_flops(),
                                 "alone_us": round(pre_iso_ms * 1e3, 1),
                                 "alone_frac_bf16": round(prefill_flops() / (pre_iso_ms / 1e3) / 1e12 / bf16, 4),
                                 "min_bytes": prefill_min_bytes(),
                                 "byte_floor_us": round(prefill_min_bytes() / (hbm * 1e9) * 1e6, 1),
                                 "flop_floor_us": round(prefill_flops() / (bf16 * 1e12) * 1e6, 1),
                                 "alone_frac_of_roofline": round(max(prefill_min_bytes() / (hbm * 1e9),
                                                                     prefill_flops() / (bf16 * 1e12))
                                                                 / (pre_iso_ms / 1e3), 4)},
                "prefill_attn_long": pl,
                "tiny_fp32": cfg["tiny_fp32"],
                "image_span": cfg["image_span"],
                "vision": cfg["vision"],
                "append_prefill": {"GB/s": round(app_gbs, 1), "frac_hbm": round(app_gbs / hbm, 4),
                                   "launch_us": round(in_job["append_pre"] * 1e3, 1),
                                   "alone_us": round(app_iso_ms * 1e3, 1),
                                   "alone_frac_hbm": round(append_bytes(LAYERS * PROMPT) / (app_iso_ms / 1e3) / 1e9 / hbm, 4)},
                "lm_head": {"GB/s": round(lm_gbs, 1), "frac_hbm": round(lm_gbs / hbm, 4),
                            "avg_launch_us": round(lm_iso_ms * 1e3, 2)},
                "verify_block": dict(vb, frac_hbm=round(vb["GB/s"] / hbm, 4)),
                "batched_serving": dict(sv, decode_frac_hbm=round(sv["decode_GB/s"] / hbm, 4),
                                        lm_head_frac_hbm=round(sv["lm_head_GB/s"] / hbm, 4)),
                "mla_asymmetric_cache": dict(mla, decode_16x4096_frac_hbm=round(mla["decode_16x4096_GB/s"] / hbm, 4)),
                "lm_head_final_norm_top1_us": round(lm_norm_ms * 1e3, 2),
                "lm_head_final_norm_top8_us": round(lm_top8_ms * 1e3, 2),
                # the whole job against the byte floor: every kernel's algorithmic bytes over the
                # timed job (the prefill at its minimum bytes; all of it is HBM-bound but the prefill)
                "job_hbm": {"algorithmic_bytes": int(job_bytes), "GB/s": round(job_bytes / (job_ms / 1e3) / 1e9, 1),
                            "frac_hbm": round(job_bytes / (job_ms / 1e3) / 1e9 / hbm, 4),
                            "floor_ms": round(job_bytes / (hbm * 1e9) * 1e3, 3)},
                "time_share": {k: round(v / sum(totals.values()), 4) for k, v in totals.items()},
                "peaks": {"hbm_gbs": hbm, "bf16_tflops": bf16, "source": peak_src},
                "frac_of_nominal": {
                    "peaks": NOMINAL_PEAKS,
                    "lm_head": round(lm_gbs / NOMINAL_PEAKS["hbm_gbs"], 4),
                    "decode_step": round(dec_gbs / NOMINAL_PEAKS["hbm_gbs"], 4),
                    "append_prefill_alone": round(append_bytes(LAYERS * PROMPT) / (app_iso_ms / 1e3) / 1e9
                                                  / NOMINAL_PEAKS["hbm_gbs"], 4),
                    "prefill_alone": round(prefill_flops() / (pre_iso_ms / 1e3) / 1e12
                                           / NOMINAL_PEAKS["bf16_tflops"], 4),
                    "prefill_in_job": round(pre_tf / NOMINAL_PEAKS["bf16_tflops"], 4),
                    "prefill_long_causal": round(pl["causal"]["TFLOP/s"] / NOMINAL_PEAKS["bf16_tflops"], 4),
                    "prefill_long_full": round(pl["full"]["TFLOP/s"] / NOMINAL_PEAKS["bf16_tflops"], 4),
                    "serving_decode": round(sv["decode_GB/s"] / NOMINAL_PEAKS["hbm_gbs"], 4),
                    "serving_lm_head": round(sv["lm_head_GB/s"] / NOMINAL_PEAKS["hbm_gbs"], 4),
                    "verify_block": round(vb["GB/s"] / NOMINAL_PEAKS["hbm_gbs"], 4),
                    "mla_decode_16x4096": round(mla["decode_16x4096_GB/s"] / NOMINAL_PEAKS["hbm_gbs"], 4),
                    "vision_bf16_full": round(cfg["vision"]["bf16"]["full_TFLOP/s"] / NOMINAL_PEAKS["bf16_tflops"], 4),
                    "image_span_prefill": round(cfg["image_span"]["prefill_TFLOP/s"] / NOMINAL_PEAKS["bf16_tflops"], 4)},
                "timing": ("lm_head: graph of 32 back-to-back launches; prefill, append: " + kt_source +
                           "; decode step: graph of the job's 256 decode launches over 4 rotating cache copies; "
                           "verify block: graph of 8 back-to-back launches (outside the job)"),
                "event_node_us": {k: round(statistics.mean(v) * 1e3, 2) for k, v in kt.items()},
            },
            "clocks": clk,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(target_s=args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def lm_traffic():
    """DRAM bytes per lm_head launch from the committed ncu summary, if it was taken on the
    current sources of the kernel (its .cu file and the headers it includes; else null)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)["lmhead_argmax"]
        h = hashlib.sha256()
        for rel in d["sources"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        if d.get("source_sha256") == h.hexdigest():
            return d["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------
# CPU oracle on a bounded sample of the job
# ----------------------------------------------------------------------------
def oracle_sample_times(rows_pf=32, dec_layers=1, lm_rows=8192, seed=0):
    """Time the oracle on one sample of each part of the job; return seconds per part and the
    factor that scales each part to the whole job."""
    import oracle as O
    import workloads as WL
    rng = np.random.default_rng(seed)
    rope = O.Rope("1d", 1e6)
    qw = 1 + 0.1 * rng.standard_normal(D); kw = 1 + 0.1 * rng.standard_normal(D)
    q = rng.standard_normal((PROMPT, HQ, D)).astype(np.float32)
    k = rng.standard_normal((PROMPT, HKV, D)).astype(np.float32)
    v = rng.standard_normal((PROMPT, HKV, D)).astype(np.float32)
    t = {}
    ck = np.zeros((HKV, WINDOW, D)); cv = np.zeros((HKV, WINDOW, D))
    t0 = time.perf_counter()
    qr = O.cache_append(q, k, v, np.arange(PROMPT)[:, None], np.arange(PROMPT), qw, kw, 1e-6, rope, False, ck, cv, "bf16")
    t["append_pre"] = time.perf_counter() - t0
    rows = np.linspace(0, PROMPT - 1, rows_pf).astype(int)
    allowed = np.zeros((rows.size, WINDOW), bool)
    for i, r in enumerate(rows):
        allowed[i, :r + 1] = True
    t0 = time.perf_counter()
    O.attend(qr[rows], ck, cv, allowed)
    t["prefill"] = time.perf_counter() - t0
    dq = rng.standard_normal((1, HQ, D)); dk = rng.standard_normal((1, HKV, D)); dv = rng.standard_normal((1, HKV, D))
    t0 = time.perf_counter()
    for _ in range(dec_layers):
        qd = O.cache_append(dq, dk, dv, [[PROMPT + 128]], [PROMPT + 128], qw, kw, 1e-6, rope, False, ck, cv, "bf16")
        O.decode(qd[0], ck, cv, PROMPT + 129)
    t["decode_step"] = time.perf_counter() - t0
    W = WL.f32_to_bf16_bits((0.02 * rng.standard_normal((lm_rows, HIDDEN))).astype(np.float32))
    h = rng.standard_normal(HIDDEN)
    t0 = time.perf_counter()
    O.lmhead_argmax(h, W, lm_rows)
    t["lm_head"] = time.perf_counter() - t0
    scale = {"append_pre": LAYERS, "prefill": LAYERS * PROMPT / rows_pf,
             "decode_step": STEPS * LAYERS / dec_layers, "lm_head": TOKENS_PER_JOB * VOCAB / lm_rows}
    job_s = sum(t[p] * scale[p] for p in t)
    sample = (f"per sample: 1 layer's 512-token append, {rows_pf} of 512 causal prefill rows x 16 heads, "
              f"{dec_layers} layer decode step (append + attention at L=641), lm_head over {lm_rows} of "
              f"{VOCAB} vocab rows; each part scaled to the full job (28 layers, 256 steps, 257 lm_head calls)")
    return job_s, sample


ORACLE_SAMPLE = dict(rows_pf=64, dec_layers=2, lm_rows=16384)   # the one sample recipe of both oracle legs


def host_info():
    """Host cores available to this process and the CPU model (lscpu, else /proc/cpuinfo)."""
    try:
        nproc = len(os.sched_getaffinity(0))
    except Exception:
        nproc = os.cpu_count()
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Vendor ID") and ":" in line:
                model = (model + " / " if model else "") + line.split(":", 1)[1].strip()
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            model = "unknown"
    return {"nproc": nproc, "cpu_model": model, "machine": os.uname().machine}


def oracle_full_configs():
    """The oracle on the small workloads in full, no sampling: seconds for the tiny fp32 layer
    (64-token prefill + 16 decode steps), the image-span layer (512-token append + prefill + 64
    decode steps) and the vision pass (append, window pass and full pass) in fp32 and bf16."""
    import oracle as O
    import workloads as WL
    out = {}
    w = WL.tiny_fp32(0)
    W_, P_ = w["capacity"], w["n_prefill"]
    rope = O.Rope("1d", w["base"])
    t0 = time.perf_counter()
    ck = np.zeros((HKV, W_, D)); cv = np.zeros((HKV, W_, D))
    qr = O.cache_append(w["q"][:P_], w["k"][:P_], w["v"][:P_], w["pos"][:P_], np.arange(P_), w["q_norm_w"],
                        w["k_norm_w"], w["eps"], rope, False, ck, cv, "f32")
    O.prefill(qr, ck, cv, P_, "causal")
    for t in range(P_, W_):
        qd = O.cache_append(w["q"][t:t + 1], w["k"][t:t + 1], w["v"][t:t + 1], w["pos"][t:t + 1], [t], w["q_norm_w"],
                            w["k_norm_w"], w["eps"], rope, False, ck, cv, "f32")
        O.decode(qd[0], ck, cv, t + 1)
    out["tiny_fp32_s"] = round(time.perf_counter() - t0, 4)
    w = WL.image_span_prefill(0)
    S3, W3, steps3 = w["pos"].shape[0], w["capacity"], w["dq"].shape[0]
    rope = O.Rope("sections", w["base"], w["sections"])
    t0 = time.perf_counter()
    ck = np.zeros((HKV, W3, D)); cv = np.zeros((HKV, W3, D))
    qr = O.cache_append(w["q"], w["k"], w["v"], w["pos"], np.arange(S3), w["q_norm_w"], w["k_norm_w"], w["eps"],
                        rope, True, ck, cv, "bf16")
    t1 = time.perf_counter()
    O.prefill(qr, ck, cv, S3, "causal")
    out["image_span_prefill_s"] = round(time.perf_counter() - t1, 4)
    for st in range(steps3):
        qd = O.cache_append(w["dq"][st:st + 1], w["dk"][st:st + 1], w["dv"][st:st + 1], w["dpos"][st:st + 1], [S3 + st],
                            w["q_norm_w"], w["k_norm_w"], w["eps"], rope, True, ck, cv, "bf16")
        O.decode(qd[0], ck, cv, S3 + st + 1)
    out["image_span_s"] = round(time.perf_counter() - t0, 4)
    w = WL.vision_windowed(0)
    lay = w["layout"]
    S4 = lay.pos_rc.shape[0]
    for dt in ("f32", "bf16"):
        t0 = time.perf_counter()
        ck = np.zeros((WL.VISION_HEADS, S4, WL.VISION_HEAD_DIM)); cv = np.zeros_like(ck)
        qr = O.cache_append(w["q"], w["k"], w["v"], lay.pos_rc, lay.slot, None, None, 0.0, O.Rope("2d", w["base"]),
                            False, ck, cv, dt)
        qs = O.store(qr, dt)[lay.row_of_slot]
        t1 = time.perf_counter()
        O.prefill(qs, ck, cv, S4, "segment", lay.segment)
        t2 = time.perf_counter()
        O.prefill(qs, ck, cv, S4, "full")
        t3 = time.perf_counter()
        out[f"vision_{dt}_window_s"] = round(t2 - t1, 4)
        out[f"vision_{dt}_full_s"] = round(t3 - t2, 4)
        out[f"vision_{dt}_s"] = round(t3 - t0, 4)
    return out


def oracle_job_samples(target_s=None, n=None, warmup=0):
    """Repeated samples of the job with ORACLE_SAMPLE: either for about target_s seconds or
    exactly warmup + n samples (the first warmup not kept).  Returns the per-sample seconds, the
    extrapolated job seconds of each kept sample, and the sample's description."""
    t_start = time.perf_counter()
    wall, jobs, sample, i = [], [], "", 0
    while True:
        t0 = time.perf_counter()
        js, sample = oracle_sample_times(seed=i, **ORACLE_SAMPLE)
        if i >= warmup:
            wall.append(time.perf_counter() - t0)
            jobs.append(js)
        i += 1
        if n is not None and len(jobs) >= n:
            break
        if n is None and jobs and time.perf_counter() - t_start >= target_s:
            break
    return wall, jobs, sample


def oracle_serving_step_sample(n_seq=2, lm_rows=8192):
    """One step of the 64-sequence serving workload on the oracle, sampled: the append and
    decode of n_seq of the 64 sequences (evenly spaced, each at its own context) and the
    lm_head of one hidden row over lm_rows vocab rows.  The attention part is scaled by the
    keys read (all 64 sequences' lengths over the sample's), the lm_head part by rows x vocab
    (64 x 151936 over 1 x lm_rows).  Returns the extrapolated seconds of one step and the
    sample's description."""
    import oracle as O
    import workloads as WL
    ctx = WL.serving_contexts(0)
    B = ctx.size
    qw, kw = WL.serving_norm_weights(0)
    inp = WL.serving_step_inputs(0, 0, batch=B)
    rope = O.Rope("1d", 1e6)
    picks = [i * (B // n_seq) for i in range(n_seq)]
    t_att = 0.0
    for b in picks:
        c = int(ctx[b])
        kb, vb = WL.serving_prefix(0, b, c)
        ck = np.zeros((HKV, c + 128, D)); cv = np.zeros((HKV, c + 128, D))
        ck[:, :c] = WL.bf16_bits_to_f32(kb); cv[:, :c] = WL.bf16_bits_to_f32(vb)
        t0 = time.perf_counter()
        qd = O.cache_append(inp["q"][b:b + 1], inp["k"][b:b + 1], inp["v"][b:b + 1], [[c]], [c], qw, kw, 1e-6,
                            rope, False, ck, cv, "bf16")
        O.decode(qd[0], ck, cv, c + 1)
        t_att += time.perf_counter() - t0
    keys_all = float(np.sum(ctx.astype(np.int64) + 1))
    keys_pick = float(sum(int(ctx[b]) + 1 for b in picks))
    rng = np.random.default_rng(5)
    W = WL.f32_to_bf16_bits((0.02 * rng.standard_normal((lm_rows, HIDDEN))).astype(np.float32))
    t0 = time.perf_counter()
    O.lmhead_argmax(inp["h"][0], W, lm_rows)
    t_lm = time.perf_counter() - t0
    step_s = t_att * keys_all / keys_pick + t_lm * B * VOCAB / lm_rows
    sample = (f"append + decode of sequences {picks} (contexts {[int(ctx[b]) for b in picks]}) scaled by keys "
              f"read to all {B}; lm_head of 1 hidden row over {lm_rows} of {VOCAB} vocab rows scaled to {B} rows "
              f"x {VOCAB}")
    return step_s, sample


def cpu_baseline(target_s=12.0):
    """Oracle (single thread, float64) on repeated bounded samples of the job for ~target_s
    seconds, the small workloads timed in full, and one sampled step of the serving workload
    (extrapolated)."""
    t_start = time.perf_counter()
    wall, jobs, sample = oracle_job_samples(target_s=target_s, warmup=1)
    job_s = statistics.median(jobs)
    full = oracle_full_configs()
    serving_s, serving_sample = oracle_serving_step_sample()
    return {"value": round(TOKENS_PER_JOB / job_s, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "host": host_info(),
            "sample": f"{len(jobs)} samples of {statistics.median(wall):.2f} s each (after one warm-up sample); "
                      f"{sample}", "job_seconds_extrapolated": round(job_s, 2),
            "full_configs_seconds": full,
            "serving_step": {"seconds_extrapolated": round(serving_s, 2),
                             "tokens_per_s_extrapolated": round(64 / serving_s, 4), "sample": serving_sample},
            "cpu_seconds": round(time.perf_counter() - t_start, 1)}


def job_config():
    return {"workload": "Qwen3-0.6B-shaped attention step: 28 layers x (512-token causal prefill + "
                        "256 decode steps), 1024-slot bf16 window, tied lm_head 151936x1024 bf16 argmax",
            "layers": LAYERS, "prompt": PROMPT, "decode_steps": STEPS, "window": WINDOW,
            "q_heads": HQ, "kv_heads": HKV, "head_dim": D, "vocab": VOCAB, "batch": 1,
            "step": "one whole job (prefill + 256 decode steps) as one CUDA graph replay",
            "l2": "inputs larger than L2: the 311 MB lm_head table streams through the 129 MB L2 "
                  "between decode steps"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one bounded sample of the job (the same
    recipe as the cpu_baseline block of the main line); the value is the job's tokens/s that the
    sample's time extrapolates to, and ms_per_step the sample's own wall time."""
    if rank != 0:
        return
    wall, jobs, sample = oracle_job_samples(n=args.steps, warmup=args.warmup)
    job_s = statistics.median(jobs)
    value = TOKENS_PER_JOB / job_s
    cfg = job_config()                      # the same workload and keys as the GPU arm's line
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.median(wall) * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "host": host_info(), "sample": sample,
                             "step": "one bounded sample of the job per step; ms_per_step is the sample's "
                                     "wall time, value the job throughput it extrapolates to",
                             "job_seconds_extrapolated": round(job_s, 2)},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kv_attn", choices=["kv_attn", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--job-only", action="store_true",
                    help="time the job only and print a short line (for counter captures); not the benchmark line")
    ap.add_argument("--only", choices=["verify", "mla", "serving16", "lm64", "configs", "topk", "prefill_long"],
                    default=None,
                    help="run one sub-benchmark alone and print its figures (for counter captures); "
                         "not the benchmark line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    from kv_cache_gqa_gb300 import build
    build.build_library(verbose=False)
    run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
