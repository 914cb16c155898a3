#!/usr/bin/env python
"""Benchmark of the attention hot path on one GB300 (or N replicas).

One *step* is one pass of the whole hot path over one batch of synthetic
input:
  1. packed causal GQA prefill attention of the Prefill-Only request batch
     (16 requests x 15 samples = 240 sequences, L ~ U{64..500}, 16/8 heads,
     d 128) through all 28 layers, each layer with its own Q/K/V;
  2. a complete short-prompt beam search (32 requests, 128-token prompts,
     beam 100, 4 decode steps, 14/2 heads, d 64) through 28 layers: per step
     and layer the suffix reorder + append, then decode attention (one
     bg_beam_decode_step call);
  3. the same for the long-prompt beam search (16 requests, prompts
     U{400..500}, beam 400, 5 steps).
The headline ``value`` is prefill TFLOP/s (causal FLOPs of valid tokens
only); decode is reported as microseconds per decode step per layer.

Inputs are resident in HBM before the timed region (drawn on the device with
a seeded generator); every layer has its own inputs, so each step streams
far more than the 129 MB L2 and nothing is reused from cache across steps.

``--impl reference`` times the fp64 CPU oracle (the only reference that
exists for this path) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_packed_varlen_causal_gb300 import workloads as wl  # noqa: E402

METRIC = "packed-prefill attn TFLOP/s (% bf16 peak); beam-decode attn µs/step (% roofline)"
LAYERS = 28
SPEC_HBM_GBS = 8000.0   # nominal GB300 HBM3e bandwidth (~8 TB/s), reported beside the measured copy peak

# DRAM bytes of one attn_kernel<Prefill,128> launch on one layer of the Prefill-Only batch
# (dram__bytes_read.sum + dram__bytes_write.sum from one ncu capture of that launch).  It holds
# only for the sources that launch is built from, identified by `sources`
# (kernel_sources_hash); otherwise the bench reports null.
PREFILL_TRAFFIC = {"sources": "13fe91063a561eee", "bytes": 649549824 + 243861504}
# the files a bg_packed_prefill_attn launch is built from
PREFILL_SOURCES = ["abi.cu", "prefill.cu", "bg_attn_kernel.cuh", "bg_ptx.cuh", "bg_internal.h"]


def kernel_sources_hash(names=PREFILL_SOURCES):
    import hashlib
    pkg = os.path.join(ROOT, "attention_packed_varlen_causal_gb300")
    files = [os.path.join(pkg, "csrc", n) for n in names] + [os.path.join(ROOT, "include", "bg_attn.h")]
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------- work accounting
def prefill_flops(lengths, Hq, d):
    """Causal attention FLOPs over valid tokens: QK^T and PV each 2*d per
    (query, key) pair with key <= query, so 2*d*Hq*sum L(L+1)."""
    L = np.asarray(lengths, dtype=np.float64)
    return float(2.0 * d * Hq * np.sum(L * (L + 1)))


def prefill_bytes(T, Hq, Hkv, d):
    """Algorithmic HBM bytes of one call: Q, K, V read once, O written once (bf16)."""
    return float(T * (2 * Hq + 2 * Hkv) * d * 2)


def decode_step_work(cfg, prompt_lengths, t):
    """FLOPs and algorithmic bytes of decode step t (1-based) for one layer:
    reorder reads+writes t-1 suffix slots, the append reads the new token's
    K/V and writes it to slot t-1, the attention reads Q, the prompt K/V once
    per request and t suffix slots per beam, and writes O."""
    R, W, Hq, Hkv, d = cfg.R, cfg.W, cfg.Hq, cfg.Hkv, cfg.head_dim
    P = float(np.sum(prompt_lengths))
    rows = R * W * Hq
    flops = 4.0 * d * rows * (np.mean(prompt_lengths) + t)
    slot = R * W * Hkv * d * 2.0                     # one suffix slot of K (or V), all beams
    reorder = 2 * 2 * slot * (t - 1) + 2 * 2 * slot  # K and V read + write, plus the append's read + write
    attn = 2 * rows * d * 2.0 + 2 * P * Hkv * d * 2.0 + 2 * slot * t
    return flops, reorder + attn


# --------------------------------------------------------------------------- helpers
def decode_item_spread(cfg, n_sm: int, tiles_per_item: int = 2):
    """How the decode attention's work items fall on the persistent CTAs (one per SM): an
    item is a request x kv head x `tiles_per_item` query tiles of floor(128 / g) beams each,
    and the CTAs take items round-robin.  Returns (items, CTAs, most items on one CTA)."""
    g = cfg.Hq // cfg.Hkv
    beams_per_tile = 128 // g
    tiles = -(-cfg.W // beams_per_tile)
    items = cfg.R * cfg.Hkv * (-(-tiles // tiles_per_item))
    ctas = min(items, n_sm)
    return items, ctas, -(-items // ctas) if ctas else 0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, directory=None):
        import tempfile
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(directory or tempfile.gettempdir(), f"bg_bench_clocks_gpu{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0=None, t1=None):
        """Stops sampling; keeps the samples taken between wall times t0 and t1
        (the timed region) when there are any."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            return summarize_clock_samples(f, t0, t1)


def summarize_clock_samples(lines, t0=None, t1=None):
    """Median SM clock, maximum SM clock and the throttle reasons seen, from nvidia-smi rows
    (timestamp, index, clocks.sm, clocks.max.sm, power, active mask, hw_slowdown,
    hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap).  Only rows inside the wall-clock
    window [t0, t1] (50 ms of slack) count when there are any; otherwise all rows do."""
    import datetime
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            rows.append((ts, float(parts[2]), float(parts[3]),
                         [n for n, v in zip(names, parts[6:10]) if v.lower() == "active"]))
        except ValueError:
            continue
    inside = [r for r in rows if t0 is not None and t0 - 0.05 <= r[0] <= t1 + 0.05]
    use = inside if inside else rows
    sm = [r[1] for r in use]
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(r[2] for r in use) if use else None,
            "reasons": sorted({n for r in use for n in r[3]}), "samples": len(use),
            "samples_in_timed_region": len(inside)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (a timing scalar, not a data-path
    collective)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- our arm
class PrefillStack:
    def __init__(self, cfg, layers, device, seed_base=1000):
        import torch
        from attention_packed_varlen_causal_gb300 import binding as bg
        self.bg = bg
        self.lengths = wl.prefill_lengths(cfg)
        self.cu_np = wl.cu_from_lengths(self.lengths)
        self.T = int(self.cu_np[-1])
        self.Hq, self.Hkv, self.d = cfg.Hq, cfg.Hkv, cfg.head_dim
        self.maxlen = max(self.lengths)
        self.cu = torch.from_numpy(self.cu_np).to(device)
        g = torch.Generator(device=device)
        self.q, self.k, self.v, self.o = [], [], [], []
        for l in range(layers):
            g.manual_seed(seed_base + l)
            self.q.append(torch.randn((self.T, self.Hq, self.d), generator=g, device=device).to(torch.bfloat16))
            self.k.append(torch.randn((self.T, self.Hkv, self.d), generator=g, device=device).to(torch.bfloat16))
            self.v.append(torch.randn((self.T, self.Hkv, self.d), generator=g, device=device).to(torch.bfloat16))
            self.o.append(torch.empty((self.T, self.Hq, self.d), dtype=torch.bfloat16, device=device))
        self.ws = torch.empty(bg.bg_packed_prefill_workspace_size(len(self.lengths), self.T, self.maxlen, self.Hq,
                                                                  self.Hkv, self.d), dtype=torch.uint8, device=device)
        self.flops = prefill_flops(self.lengths, self.Hq, self.d)
        self.bytes = prefill_bytes(self.T, self.Hq, self.Hkv, self.d)

    def plan(self, stream):
        """The batch's work list, once per step: every layer shares the packing."""
        self.bg.bg_packed_prefill_plan(self.cu, self.T, self.maxlen, workspace=self.ws, stream=stream)

    def run_layer(self, l, stream):
        self.bg.bg_packed_prefill_attn_planned(self.q[l], self.k[l], self.v[l], self.cu, self.maxlen, self.o[l],
                                               workspace=self.ws, stream=stream)


class DecodeStack:
    """One full beam search (steps x layers) with per-layer prompt K/V and
    per-step inputs, replayed from a CUDA graph."""

    def __init__(self, cfg, layers, device, seed_base):
        import torch
        from attention_packed_varlen_causal_gb300 import binding as bg
        self.bg = bg
        self.cfg = cfg
        self.plen = wl.decode_prompt_lengths(cfg)
        cu = wl.cu_from_lengths(self.plen)
        self.cu = torch.from_numpy(cu).to(device)
        self.P = int(cu[-1])
        R, W, Hq, Hkv, d, S = cfg.R, cfg.W, cfg.Hq, cfg.Hkv, cfg.head_dim, cfg.steps
        g = torch.Generator(device=device)
        bf = torch.bfloat16
        self.pk, self.pv, self.q, self.nk, self.nv, self.sk, self.sv, self.out = [], [], [], [], [], [], [], []
        for l in range(layers):
            g.manual_seed(seed_base + l)
            self.pk.append(torch.randn((self.P, Hkv, d), generator=g, device=device).to(bf))
            self.pv.append(torch.randn((self.P, Hkv, d), generator=g, device=device).to(bf))
            self.q.append([torch.randn((R, W, Hq, d), generator=g, device=device).to(bf) for _ in range(S)])
            self.nk.append([torch.randn((R, W, Hkv, d), generator=g, device=device).to(bf) for _ in range(S)])
            self.nv.append([torch.randn((R, W, Hkv, d), generator=g, device=device).to(bf) for _ in range(S)])
            self.sk.append([torch.zeros((R, W, S, Hkv, d), dtype=bf, device=device) for _ in range(2)])
            self.sv.append([torch.zeros((R, W, S, Hkv, d), dtype=bf, device=device) for _ in range(2)])
            self.out.append(torch.empty((R, W, Hq, d), dtype=bf, device=device))
        self.parent = [torch.from_numpy(np.random.default_rng(wl.SEED_PARENT + s).integers(0, W, size=(R, W))
                                        .astype(np.int32)).to(device) for s in range(S)]
        self.layers = layers
        self.graph = None
        fl, by = 0.0, 0.0
        for t in range(1, S + 1):
            f, b = decode_step_work(cfg, self.plen, t)
            fl += f
            by += b
        self.flops_per_search = fl * layers
        self.bytes_per_search = by * layers
        self.launches = 2 * S * layers            # reorder + attention per step and layer

    def enqueue(self, stream):
        bg = self.bg
        for s in range(self.cfg.steps):
            src, dst = s % 2, 1 - s % 2
            for l in range(self.layers):
                # reorder + append into dst, then attention over it
                bg.bg_beam_decode_step(self.q[l][s], self.pk[l], self.pv[l], self.cu, max(self.plen),
                                       self.sk[l][src], self.sv[l][src], self.parent[s], self.nk[l][s],
                                       self.nv[l][s], self.sk[l][dst], self.sv[l][dst], s + 1, self.out[l],
                                       stream=stream)

    def capture(self, stream):
        import torch
        self.enqueue(stream)                      # warm (also sets kernel attributes outside capture)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            self.enqueue(torch.cuda.current_stream())
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()


def time_oracle_sample(layer_seqs: int = 240, seed_layer: int = 0):
    """The fp64 oracle, as it stands, on a bounded sample of the Prefill-Only
    batch: the first `layer_seqs` sequences of one layer.  Returns
    (TFLOP/s, seconds, threads, description)."""
    import oracle
    n = layer_seqs
    x = wl.make_prefill_config_prefix(wl.PREFILL_CONFIGS["prefill_only"], n, layer=seed_layer)
    cu = x["cu_seqlens"]
    T = int(cu[n])
    lengths = x["lengths"]
    scale = 1.0 / math.sqrt(x["head_dim"])
    t0 = time.perf_counter()
    oracle.prefill(x["q"], x["k"], x["v"], cu, scale)
    dt = time.perf_counter() - t0
    fl = prefill_flops(lengths, x["Hq"], x["head_dim"])
    desc = f"oracle fp64 prefill of {n} of 240 sequences of one layer ({T} tokens, {fl / 1e9:.1f} GFLOP)"
    return fl / dt / 1e12, dt, oracle.num_threads(), desc


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def time_oracle_configs(skewed_seqs: int = 160):
    """The fp64 oracle, as it stands, on every workload (one layer each), timed on the host
    cores: the tiny prefill, a stated sample of the skewed layer (its first ``skewed_seqs``
    sequences), and for both beam searches one decode step (the last, longest one) and one
    complete search of one layer (per step the history reorder through the parent index, the
    append and the attention).  The Prefill-Only layer is timed by time_oracle_sample."""
    import oracle
    res = {}
    # tiny
    cfg = wl.PREFILL_CONFIGS["tiny"]
    x = wl.make_prefill_config_inputs(cfg)
    fl = prefill_flops(x["lengths"], x["Hq"], x["head_dim"])
    t0 = time.perf_counter()
    oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], 1.0 / math.sqrt(x["head_dim"]))
    dt = time.perf_counter() - t0
    res["tiny"] = {"seconds": round(dt, 4), "gflop": round(fl / 1e9, 3), "tflops": round(fl / dt / 1e12, 6),
                   "sample": "the whole tiny layer (4 sequences, T = 392)"}
    # skewed: the first sequences of the layer, with the layer's 1 % outlier K rows drawn over them
    cfg = wl.PREFILL_CONFIGS["skewed"]
    lengths = wl.prefill_lengths(cfg)[:skewed_seqs]
    x = wl.make_prefill_inputs(lengths, cfg.Hq, cfg.Hkv, cfg.head_dim, outlier_frac=cfg.outlier_frac,
                               outlier_scale=cfg.outlier_scale)
    fl = prefill_flops(lengths, cfg.Hq, cfg.head_dim)
    full = prefill_flops(wl.prefill_lengths(cfg), cfg.Hq, cfg.head_dim)
    t0 = time.perf_counter()
    oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], 1.0 / math.sqrt(cfg.head_dim))
    dt = time.perf_counter() - t0
    res["skewed"] = {"seconds": round(dt, 3), "gflop": round(fl / 1e9, 2), "tflops": round(fl / dt / 1e12, 6),
                     "sample": f"first {skewed_seqs} of 4096 sequences of one layer ({int(sum(lengths))} tokens, "
                               f"{fl / 1e9:.1f} of the layer's {full / 1e9:.0f} GFLOP)",
                     "full_layer_seconds_extrapolated": round(dt * full / fl, 1)}
    # beam searches
    for name in ("beam_short", "beam_long"):
        cfg = wl.DECODE_CONFIGS[name]
        pb = wl.make_decode_config_problem(cfg)
        scale = 1.0 / math.sqrt(cfg.head_dim)
        plen = pb["prompt_lengths"]
        hist = oracle.BeamHistory(cfg.R, cfg.W)
        step_s, step_fl = [], []
        t_all = time.perf_counter()
        for s in range(cfg.steps):
            t0 = time.perf_counter()
            hist.step(pb["parent"][s], pb["new_k"][s], pb["new_v"][s])
            hk, hv = hist.materialise(cfg.Hkv, cfg.head_dim)
            oracle.decode(pb["q"][s], pb["prompt_k"], pb["prompt_v"], pb["cu_prompt"], hk, hv, scale)
            step_s.append(time.perf_counter() - t0)
            step_fl.append(decode_step_work(cfg, plen, s + 1)[0])
        dt_all = time.perf_counter() - t_all
        res[name] = {"step_seconds": round(step_s[-1], 4), "step": cfg.steps,
                     "step_tflops": round(step_fl[-1] / step_s[-1] / 1e12, 6),
                     "search_seconds": round(dt_all, 3), "search_tflops": round(sum(step_fl) / dt_all / 1e12, 6),
                     "us_per_step_avg": round(dt_all * 1e6 / cfg.steps, 1),
                     "sample": f"one layer: the last decode step (suffix length {cfg.steps}), and the complete "
                               f"{cfg.steps}-step search (history reorder + append + attention per step)"}
    return res


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from attention_packed_varlen_causal_gb300 import binding as bg
    from attention_packed_varlen_causal_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    bg.load()
    peaks = load_peaks()
    layers = args.layers
    stream = torch.cuda.Stream(device=device)

    pre = PrefillStack(wl.PREFILL_CONFIGS["prefill_only"], layers, device)
    dec_s = DecodeStack(wl.DECODE_CONFIGS["beam_short"], layers, device, seed_base=2000)
    dec_l = DecodeStack(wl.DECODE_CONFIGS["beam_long"], layers, device, seed_base=3000)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        dec_s.capture(stream)
        dec_l.capture(stream)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    n_ev = args.steps * layers
    pre_start = [ev() for _ in range(n_ev)]
    pre_end = [ev() for _ in range(n_ev)]
    step_marks = [[ev() for _ in range(4)] for _ in range(args.steps)]

    def one_step(i=None):
        with torch.cuda.stream(stream):
            if i is not None:
                step_marks[i][0].record(stream)
            pre.plan(stream)
            for l in range(layers):
                if i is not None:
                    pre_start[i * layers + l].record(stream)
                pre.run_layer(l, stream)
                if i is not None:
                    pre_end[i * layers + l].record(stream)
            if i is not None:
                step_marks[i][1].record(stream)
            dec_s.replay()
            if i is not None:
                step_marks[i][2].record(stream)
            dec_l.replay()
            if i is not None:
                step_marks[i][3].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, args.clocks_dir)
    clocks.start()
    time.sleep(0.5)                      # let nvidia-smi start sampling
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start = ev()
    t_end = ev()
    t_start.record(stream)
    for i in range(args.steps):
        one_step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop(wall0, wall1)

    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world, device)
    prefill_ms = sum(step_marks[i][0].elapsed_time(step_marks[i][1]) for i in range(args.steps))
    short_ms = sum(step_marks[i][1].elapsed_time(step_marks[i][2]) for i in range(args.steps))
    long_ms = sum(step_marks[i][2].elapsed_time(step_marks[i][3]) for i in range(args.steps))
    prefill_ms = max_over_ranks(prefill_ms, world, device)
    call_ms = [pre_start[j].elapsed_time(pre_end[j]) for j in range(n_ev)]
    avg_call_s = statistics.mean(call_ms) / 1e3
    med_call_s = statistics.median(call_ms) / 1e3
    pre_flops_step = pre.flops * layers
    tflops = world * pre_flops_step * args.steps / (prefill_ms / 1e3) / 1e12
    per_gpu_tflops = pre_flops_step * args.steps / (prefill_ms / 1e3) / 1e12

    n_sm = torch.cuda.get_device_properties(device).multi_processor_count

    def replay_median_ms(dec, reps):
        """Median over ``reps`` individually timed replays of the whole search."""
        evs = [(ev(), ev()) for _ in range(reps)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                a.record(stream)
                dec.replay()
                b.record(stream)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    def dec_report(dec, ms):
        cfg = dec.cfg
        n_step = cfg.steps * layers
        mean_us = ms * 1e3 / args.steps / n_step
        med_ms = replay_median_ms(dec, args.reps)
        us_per_step = med_ms * 1e3 / n_step
        t_flops = dec.flops_per_search / (peaks["bf16_tflops"] * 1e12)
        t_bytes = dec.bytes_per_search / (peaks["hbm_gbs"] * 1e9)
        roof_us = max(t_flops, t_bytes) * 1e6 / n_step
        items, ctas, most = decode_item_spread(cfg, n_sm)
        return {"workload": f"{cfg.name}: R{cfg.R} W{cfg.W} {cfg.steps} steps Hq{cfg.Hq}/Hkv{cfg.Hkv} d{cfg.head_dim}, "
                            f"{layers} layers, CUDA-graph replay",
                "attention_items": items, "attention_ctas": ctas, "max_items_per_cta": most,
                "us_per_step": round(us_per_step, 3), "us_per_step_mean_in_step": round(mean_us, 3),
                "replays_timed": args.reps, "roofline_us_per_step": round(roof_us, 3),
                "roofline_frac": round(roof_us / us_per_step, 4),
                "bound": "tensor" if t_flops > t_bytes else "hbm",
                "tokens_per_s": round(cfg.R * cfg.W * cfg.steps / (med_ms / 1e3), 1),
                "tokens_per_s_definition": f"R*W*steps new tokens per search / time of the search's decode "
                                           f"attention steps through all {layers} layers (attention only)",
                "us_per_step_definition": "one decode step of one layer (bg_beam_decode_step: suffix reorder + "
                                          "append and attention), median over the timed replays of the whole "
                                          "search / (steps x layers)",
                "launches_per_step": round(dec.launches / n_step, 3)}

    decode = {"beam_short": dec_report(dec_s, short_ms), "beam_long": dec_report(dec_l, long_ms)}
    tiny = run_tiny(device, stream, args.reps)

    # e2e: one layer per step through the C ABI with host buffers (pinned),
    # H2D of q, k, v, cu_seqlens and D2H of the output inside the timed region
    e2e = run_e2e(pre, device, stream, args)
    last = run_last_token(pre, stream, peaks)
    fp8 = run_fp8_prefill(pre, stream, peaks)
    select = run_beam_select(device, stream, peaks, args.reps)
    skewed = run_skewed(device, stream, peaks, args.reps)

    # oracle CPU baseline (rank 0, N = 1 only)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        v, dt, thr, desc = time_oracle_sample(args.cpu_sample_seqs)
        cpu = {"value": round(v, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle", "sample": desc,
               "seconds": round(dt, 2), "cpu_model": cpu_model(),
               "per_config": {"prefill_only": {"seconds": round(dt, 3), "tflops": round(v, 6), "sample": desc}}}
        cpu["per_config"].update(time_oracle_configs())

    achieved = pre.bytes / med_call_s / 1e9
    traffic = args.traffic
    src_hash = kernel_sources_hash()
    traffic_source = "--traffic argument" if traffic is not None else None
    if traffic is None and src_hash == PREFILL_TRAFFIC["sources"]:
        traffic = PREFILL_TRAFFIC["bytes"]
        traffic_source = f"stored ncu capture of this launch, prefill sources hash {src_hash}"
    if traffic is None:
        traffic_source = f"none: prefill sources (hash {src_hash}) changed since the stored capture"
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic, "traffic_source": traffic_source,
                "algorithmic_bytes_per_launch": pre.bytes,
                "launch_us_median": round(med_call_s * 1e6, 2), "launch_us_mean": round(avg_call_s * 1e6, 2),
                "launches_timed": n_ev,
                "kernel": "bg_packed_prefill_attn_planned (attn_kernel<Prefill,128>; the step plans the batch's "
                          "work list once, bg_packed_prefill_plan, inside the timed prefill phase)",
                "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)",
                "spec_hbm_gbs": SPEC_HBM_GBS, "frac_of_spec_hbm": round(achieved / SPEC_HBM_GBS, 4),
                "tensor_frac_of_bf16_peak": round(pre.flops / med_call_s / 1e12 / peaks["bf16_tflops"], 4),
                "tensor_frac_of_bf16_sustained": round(pre.flops / med_call_s / 1e12 /
                                                       peaks["bf16_tflops_sustained"], 4)}
    launches = args.steps * (1 + layers + dec_s.launches + dec_l.launches)   # plan + one attention per layer
    line = {
        "metric": METRIC, "value": round(tflops, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "pct_bf16_peak": round(per_gpu_tflops / peaks["bf16_tflops"], 4),
        "config": {"workload": f"Prefill-Only batch: 240 seqs (16 req x 15 samples), L~U{{64..500}} seed 0, "
                               f"T={pre.T}, Hq16/Hkv8 d128, causal, {layers} layers; plus one short- and one "
                               f"long-prompt beam search per step", "layers": layers, "tokens_per_layer": pre.T,
                   "l2": "inputs larger than L2: every layer has its own Q/K/V (per-layer working set "
                         f"{pre.bytes / 1e6:.0f} MB > 129 MB L2), no flush needed", "parallelism": f"replicas x{world}"},
        "prefill": {"ms_per_step": round(prefill_ms / args.steps, 3), "tflops_per_gpu": round(per_gpu_tflops, 3),
                    "avg_call_us": round(avg_call_s * 1e6, 2), "tokens_per_s": round(world * pre.T * layers * args.steps / (prefill_ms / 1e3), 1),
                    "calls": f"per step one bg_packed_prefill_plan (the batch's work list) and {layers} "
                             "bg_packed_prefill_attn_planned, all inside the prefill phase; avg_call_us is one "
                             "planned call"},
        "decode": decode,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "gpu_launches": launches,
        "last_token": last, "beam_select": select, "skewed": skewed, "tiny": tiny, "fp8_prefill": fp8,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def median_us_of_calls(stream, fns, reps):
    """Median, in microseconds, over ``reps`` individually timed calls; call i runs fns[i % len(fns)]
    (CUDA events on the launching stream around every call)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for i, (a, b) in enumerate(evs):
            a.record(stream)
            fns[i % len(fns)]()
            b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3


def run_tiny(device, stream, reps: int = 50):
    """The tiny packed prefill (4 sequences {17, 64, 100, 211}, 16/8 heads, d 128), median over
    ``reps`` individually timed calls.  The inputs (4.8 MB) would sit in L2, so the calls rotate
    over enough copies in distinct buffers to cover four times the L2 size."""
    import torch
    from attention_packed_varlen_causal_gb300 import binding as bg
    cfg = wl.PREFILL_CONFIGS["tiny"]
    x = wl.make_prefill_config_inputs(cfg)
    T, Hq, Hkv, d = x["q"].shape[0], x["Hq"], x["Hkv"], x["head_dim"]
    by = prefill_bytes(T, Hq, Hkv, d)
    l2 = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 129 << 20))
    n_sets = max(2, int(math.ceil(4 * l2 / by)))

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    q0, k0, v0 = dev(x["q"]), dev(x["k"]), dev(x["v"])
    cu = torch.from_numpy(x["cu_seqlens"]).to(device)
    sets = [(q0.clone(), k0.clone(), v0.clone(), torch.empty_like(q0)) for _ in range(n_sets)]
    ws = torch.empty(bg.bg_packed_prefill_workspace_size(len(x["lengths"]), T, x["max_seqlen"], Hq, Hkv, d),
                     dtype=torch.uint8, device=device)
    fns = [lambda st=st: bg.bg_packed_prefill_attn(st[0], st[1], st[2], cu, x["max_seqlen"], st[3], workspace=ws,
                                                    stream=stream) for st in sets]
    for f in fns[:10]:
        with torch.cuda.stream(stream):
            f()
    us = median_us_of_calls(stream, fns, max(reps, n_sets))
    fl = prefill_flops(x["lengths"], Hq, d)
    del sets
    return {"workload": "tiny packed prefill: lengths {17, 64, 100, 211}, Hq16/Hkv8 d128, causal",
            "us_per_call": round(us, 2), "tflops": round(fl / us / 1e6, 3), "gflop": round(fl / 1e9, 4),
            "bytes": by, "l2": f"calls rotate over {n_sets} input copies ({n_sets * by / 1e6:.0f} MB >= 4x L2)",
            "definition": f"median over {max(reps, n_sets)} individually timed bg_packed_prefill_attn calls "
                          "(work-list pre-pass + attention)"}


def fp8_codes_on_device(x):
    """E4M3 codes (uint8) and the per-tensor power-of-two scale of a bf16 CUDA tensor: the
    smallest 2^k with max|x| / 2^k <= 448, then torch's round-to-nearest cast (input
    preparation for the FP8 leg, outside any timed region)."""
    import torch
    amax = float(x.abs().max().float().item())
    s = 1.0 if amax == 0.0 else 2.0 ** math.ceil(math.log2(amax / 448.0))
    if amax / s > 448.0:
        s *= 2.0
    codes = (x.float() / s).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, s


def fp8_prefill_bytes(T, Hq, Hkv, d):
    """Algorithmic HBM bytes of one FP8 call: E4M3 Q and K (1 byte), bf16 V read once, bf16 O
    written once: 9,216 bytes per token for 16/8 heads at d 128."""
    return float(T * (Hq * d + Hkv * d + Hkv * d * 2 + Hq * d * 2))


def run_fp8_prefill(pre, stream, peaks, reps: int = 56):
    """bg_packed_prefill_attn_fp8 on every layer of the Prefill-Only batch (each layer's Q and K
    quantised to E4M3 codes with per-tensor power-of-two scales, bf16 V), median over
    individually timed calls, apart from the step."""
    import torch
    bg = pre.bg
    layers = len(pre.q)
    qc, kc = [], []
    for l in range(layers):
        qc.append(fp8_codes_on_device(pre.q[l]))
        kc.append(fp8_codes_on_device(pre.k[l]))
    out = torch.empty_like(pre.o[0])
    fns = [lambda l=l: bg.bg_packed_prefill_attn_fp8(qc[l][0], qc[l][1], kc[l][0], kc[l][1], pre.v[l], pre.cu,
                                                      pre.maxlen, out, workspace=pre.ws, stream=stream)
           for l in range(layers)]
    with torch.cuda.stream(stream):
        for f in fns:
            f()
    torch.cuda.synchronize()
    us = median_us_of_calls(stream, fns, max(reps, 50))
    by = fp8_prefill_bytes(pre.T, pre.Hq, pre.Hkv, pre.d)
    del qc, kc
    return {"workload": f"Prefill-Only batch (240 seqs, T={pre.T}), E4M3 Q and K with per-tensor power-of-two "
                        f"scales, bf16 V, {layers} layers",
            "us_per_layer": round(us, 2), "tflops": round(pre.flops / us / 1e6, 2),
            "pct_bf16_peak": round(pre.flops / us / 1e6 / peaks["bf16_tflops"], 4),
            "bytes_per_layer": by, "achieved_gbs": round(by / us / 1e3, 1),
            "hbm_frac": round(by / us / 1e3 / peaks["hbm_gbs"], 4),
            "roofline_us": round(max(pre.flops / (peaks["bf16_tflops"] * 1e6), by / (peaks["hbm_gbs"] * 1e3)), 1),
            "definition": "bg_packed_prefill_attn_fp8 per layer (work-list pre-pass + attn_kernel<Prefill,128,E4M3 "
                          f"Q/K>), median over {max(reps, 50)} individually timed calls, apart from the step "
                          "(not in value); Q.K^T runs as kind::f8f6f4, P.V in bf16"}


def run_last_token(pre, stream, peaks, reps: int = 56):
    """The Prefill-Only last-layer variant, timed apart from the step: attention of each
    sequence's last valid token over the layer's K/V (bg_packed_last_token_attn), on every
    layer's own K/V, CUDA events on the launching stream."""
    import torch
    bg = pre.bg
    rows = torch.from_numpy(pre.cu_np[1:] - 1).to(pre.q[0].device).long()
    B = len(pre.lengths)
    qs = [pre.q[l].index_select(0, rows).contiguous() for l in range(len(pre.q))]
    out = torch.empty((B, pre.Hq, pre.d), dtype=torch.bfloat16, device=pre.q[0].device)
    fns = [lambda l=l: bg.bg_packed_last_token_attn(qs[l], pre.k[l], pre.v[l], pre.cu, pre.maxlen, out,
                                                     stream=stream) for l in range(len(qs))]
    with torch.cuda.stream(stream):
        for f in fns:
            f()
    torch.cuda.synchronize()
    us = median_us_of_calls(stream, fns, max(reps, 50))
    by = float(pre.T * pre.Hkv * pre.d * 2 * 2 + 2 * B * pre.Hq * pre.d * 2)   # K, V once; q in, out
    gbs = by / us / 1e3
    return {"workload": f"Prefill-Only batch, last valid token of each of {B} sequences, {len(qs)} layers",
            "us_per_layer": round(us, 2), "bytes_per_layer": by, "achieved_gbs": round(gbs, 1),
            "hbm_frac": round(gbs / peaks["hbm_gbs"], 4), "bound": "hbm",
            "definition": "bg_packed_last_token_attn per layer (each layer's own K/V in turn), median over "
                          f"{max(reps, 50)} individually timed calls, apart from the step (not in value)"}


def run_skewed(device, stream, peaks, reps: int = 50):
    """The skewed packed-prefill stress workload, timed apart from the step: 4096 sequences,
    L = clip(round(lognormal(5.5, 0.8)), 1, 2048), 16 Q / 8 KV heads, head_dim 128, 1 % of the
    (token, kv head) K rows scaled by 8 (outlier logits).  One layer stays resident (16.7 GB,
    far above L2); bg_packed_prefill_attn is called ``reps`` times after two warm-up calls,
    CUDA events on the launching stream."""
    import numpy as np
    import torch
    from attention_packed_varlen_causal_gb300 import binding as bg
    cfg = wl.PREFILL_CONFIGS["skewed"]
    lengths = wl.prefill_lengths(cfg)
    cu_np = wl.cu_from_lengths(lengths)
    T, Hq, Hkv, d = int(cu_np[-1]), cfg.Hq, cfg.Hkv, cfg.head_dim
    g = torch.Generator(device=device)
    g.manual_seed(5000)
    q = torch.randn((T, Hq, d), generator=g, device=device).to(torch.bfloat16)
    k = torch.randn((T, Hkv, d), generator=g, device=device).to(torch.bfloat16)
    v = torch.randn((T, Hkv, d), generator=g, device=device).to(torch.bfloat16)
    rows = T * Hkv
    pick = np.random.default_rng(wl.SEED_OUTLIER).choice(rows, size=int(round(cfg.outlier_frac * rows)),
                                                         replace=False)
    pick = torch.from_numpy(pick.astype(np.int64)).to(device)
    k2 = k.view(rows, d)
    k2[pick] = k2[pick] * cfg.outlier_scale          # x8 is exact in bf16
    out = torch.empty_like(q)
    cu = torch.from_numpy(cu_np).to(device)
    maxlen = max(lengths)
    ws = torch.empty(bg.bg_packed_prefill_workspace_size(len(lengths), T, maxlen, Hq, Hkv, d), dtype=torch.uint8,
                     device=device)
    call = lambda: bg.bg_packed_prefill_attn(q, k, v, cu, maxlen, out, workspace=ws, stream=stream)  # noqa: E731
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    torch.cuda.synchronize()
    us = median_us_of_calls(stream, [call], reps)
    flops = prefill_flops(lengths, Hq, d)
    by = prefill_bytes(T, Hq, Hkv, d)
    res = {"workload": f"skewed stress: {len(lengths)} seqs, L=clip(round(lognormal(5.5, 0.8)), 1, 2048) seed 0, "
                       f"T={T}, Hq{Hq}/Hkv{Hkv} d{d}, causal, 1% of K rows x8, one layer (inputs > L2)",
           "us_per_call": round(us, 1), "tflops": round(flops / us / 1e6, 2),
           "pct_bf16_peak": round(flops / us / 1e6 / peaks["bf16_tflops"], 4),
           "achieved_gbs": round(by / us / 1e3, 1), "hbm_frac": round(by / us / 1e3 / peaks["hbm_gbs"], 4),
           "roofline_us": round(max(flops / (peaks["bf16_tflops"] * 1e6), by / (peaks["hbm_gbs"] * 1e3)), 1),
           "flops": flops, "bytes": by,
           "definition": f"bg_packed_prefill_attn on one layer of the skewed workload, median over {reps} "
                         "individually timed calls, apart from the step (not in value)"}
    del q, k, v, out, ws, k2, pick
    torch.cuda.empty_cache()
    return res


SELECT_VOCAB = 65536   # the pages give no vocabulary size; selection cost is linear in it


def run_beam_select(device, stream, peaks, reps: int = 50):
    """Beam candidate selection of one decode step (bg_beam_select) on the two beam
    configurations' shapes, timed apart from the step: fp32 logits N(0, 3) of every beam
    over SELECT_VOCAB tokens (0.84 / 1.68 GB, larger than L2), accumulated scores N(-3, 1)."""
    import torch
    from attention_packed_varlen_causal_gb300 import binding as bg
    res = {}
    g = torch.Generator(device=device)
    for name in ("beam_short", "beam_long"):
        cfg = wl.DECODE_CONFIGS[name]
        R, W, V = cfg.R, cfg.W, SELECT_VOCAB
        g.manual_seed(4000 + R)
        logits = torch.randn((R, W, V), generator=g, device=device) * 3.0
        cum = torch.randn((R, W), generator=g, device=device) - 3.0
        tok = torch.empty((R, W), dtype=torch.int32, device=device)
        par = torch.empty((R, W), dtype=torch.int32, device=device)
        sc = torch.empty((R, W), dtype=torch.float32, device=device)
        ws = torch.empty(bg.bg_beam_select_workspace_size(R, W, V), dtype=torch.uint8, device=device)
        call = lambda: bg.bg_beam_select(logits, cum, tok, par, sc, workspace=ws, stream=stream)  # noqa: E731
        with torch.cuda.stream(stream):
            for _ in range(3):
                call()
        torch.cuda.synchronize()
        us = median_us_of_calls(stream, [call], reps)
        by = float(R * W * V * 4 + R * W * 4 * 4)      # logits once; cum in; token, parent, score out
        gbs = by / us / 1e3
        res[name] = {"workload": f"R{R} W{W} V{V} fp32 logits", "us_per_call": round(us, 2), "bytes": by,
                     "achieved_gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4)}
        del logits
    res["definition"] = ("bg_beam_select per decode step (per-beam logsumexp + top-W, merged by accumulated score), "
                         f"median over {reps} individually timed calls, apart from the step (not in value); "
                         "bound: HBM, logits read from HBM once (the second pass over a row hits L2)")
    return res


def run_e2e(pre, device, stream, args):
    """End to end through the C ABI, one layer per step, from pinned host memory: every step
    copies its Q/K/V/cu_seqlens host -> device, runs bg_packed_prefill_attn and copies the
    output device -> host, all inside the timed region.  Consecutive steps overlap as a
    serving loop would: step i+1's inputs copy in (own stream, own copy direction) while
    step i computes and copies out; two device buffer sets keep them apart."""
    import torch
    bg = pre.bg
    T, Hq, Hkv, d = pre.T, pre.Hq, pre.Hkv, pre.d
    h_q = pre.q[0].cpu().pin_memory()
    h_k = pre.k[0].cpu().pin_memory()
    h_v = pre.v[0].cpu().pin_memory()
    h_cu = pre.cu.cpu().pin_memory()
    h_o = torch.empty((T, Hq, d), dtype=torch.bfloat16).pin_memory()
    bufs = [dict(q=torch.empty_like(pre.q[0]), k=torch.empty_like(pre.k[0]), v=torch.empty_like(pre.v[0]),
                 cu=torch.empty_like(pre.cu), o=torch.empty_like(pre.o[0])) for _ in range(2)]
    s_in = torch.cuda.Stream(device=device)
    s_out = torch.cuda.Stream(device=device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    recorded = set()

    def wait(strm, e, key):
        if key in recorded:
            strm.wait_event(e)

    def step(i):
        j = i % 2
        b = bufs[j]
        with torch.cuda.stream(s_in):
            wait(s_in, comp_done[j], ("c", j))            # step i-2 no longer reads buffer set j
            b["q"].copy_(h_q, non_blocking=True)
            b["k"].copy_(h_k, non_blocking=True)
            b["v"].copy_(h_v, non_blocking=True)
            b["cu"].copy_(h_cu, non_blocking=True)
            in_done[j].record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(in_done[j])
            wait(stream, out_done[j], ("o", j))           # step i-2's output has left buffer set j
            bg.bg_packed_prefill_attn(b["q"], b["k"], b["v"], b["cu"], pre.maxlen, b["o"], workspace=pre.ws,
                                      stream=stream)
            comp_done[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[j])
            h_o.copy_(b["o"], non_blocking=True)
            out_done[j].record(s_out)
        recorded.update({("c", j), ("o", j)})

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(3, args.steps)
    a.record(s_in)
    for i in range(n):
        step(i)
    e.record(s_out)                                       # after the last step's output copy
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / n
    h2d = h_q.numel() * 2 + h_k.numel() * 2 + h_v.numel() * 2 + h_cu.numel() * 4
    d2h = h_o.numel() * 2
    return {"value": round(pre.flops / (ms / 1e3) / 1e12, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 3),
            "definition": "one layer per step via bg_packed_prefill_attn with pinned host Q/K/V/cu_seqlens copied "
                          "in and the output copied out inside the timed region; consecutive steps overlap (inputs "
                          "of step i+1 copy in while step i computes and copies out)"}


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return
    vals, secs = [], []
    thr, desc = 0, ""
    for _ in range(min(args.warmup, 1)):
        time_oracle_sample(args.ref_sample_seqs)
    for _ in range(args.steps):
        v, dt, thr, desc = time_oracle_sample(args.ref_sample_seqs)
        vals.append(v)
        secs.append(dt)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.mean(secs), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "Prefill-Only batch (240 seqs, L~U{64..500}, Hq16/Hkv8 d128, causal); each step "
                                   "a bounded sample: " + desc},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--cpu-sample-seqs", type=int, default=240)
    ap.add_argument("--ref-sample-seqs", type=int, default=24)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reps", type=int, default=50,
                    help="individually timed repetitions behind every median (kernel legs)")
    ap.add_argument("--clocks-dir", default=None,
                    help="where the raw nvidia-smi samples of the timed region go (default: the temp directory)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the prefill kernel from the committed ncu summary")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
