#!/usr/bin/env python
"""Wave-index decode benchmark (one JSON line on rank 0).

Main line: the Llama-3-8B-shaped single-layer decode -- 131072 tokens, 32
query heads over 8 kv heads, head size 128, bf16 KV, 16 segments x 512
clusters per kv head, retrieval budget 148 clusters (1.8%), steady zone 4 + 64
tokens -- on seeded synthetic data (kvsynth).  A step is one decode step of the
whole batch: centroid scoring, top-k with the estimation over all clusters,
exact attention over steady + retrieved rows, LSE merge.

Timing: the decode steps are captured in CUDA graphs and replayed (every graph
is replayed once untimed first); each step runs on one of R independent index +
KV replicas in turn (4.7 GB of replicas in total, far above the 129 MB L2),
with a different query per step.  Each decode kernel is also timed alone: a
graph of launches of that kernel only (wi_decode_kernel), over the same
rotating replicas, gives its average launch duration without events between
kernels; the roofline of the line is the longest of those kernels.

`configs` adds the other workloads at full size, generated on the device
(kvsynth_cuda): batch 16 at 120K tokens, one million tokens across 32 layers,
and the Qwen2.5-7B-shaped batch 8 at 262K tokens (its index build and 64
decode steps that each append a token).  Each gets steps/s, its step's
algorithmic bytes and HBM rate, its kernels alone, its build, and the dense
comparator.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import kvsynth  # noqa: E402

METRIC = "wave-index decode steps/s (batch×layer) at 128K–1M; HBM GB/s vs peak"
UNIT = "steps/s"
WORKLOAD = "llama3-8b-131k"
INDEX_BYTES_PER_CLUSTER = 128 * 2 + 128 * 4 + 4   # mu bf16 + valsum fp32 + count (bf16 variant: 128 * 2)
ROW_BYTES = 128 * 2 * 2                           # one K row + one V row (bf16)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps") or d.get("hbm")
            tf = d.get("bf16_tflops")
            tfs = d.get("bf16_tflops_sustained", tf)
            if hbm:
                return float(hbm), float(tf or FALLBACK_BF16_TFLOPS), float(tfs or FALLBACK_BF16_TFLOPS), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_setup(w, k, v, seed_units=None):
    """Oracle index (one k-means round, setup only) and float64 caches for the CPU baseline."""
    import oracle
    K = oracle.bf16_from_bits(k).reshape(w.units, w.n_ctx, 128)
    V = oracle.bf16_from_bits(v).reshape(w.units, w.n_ctx, 128)
    p = oracle.IndexParams(seg_len=w.seg_len, clusters_per_seg=w.clusters_per_seg, iters=1, n_sink=w.n_sink,
                           local_window=w.local_window, budget_frac=w.budget_frac, budget_k=w.budget_k)
    units = range(w.units) if seed_units is None else seed_units
    idx = {u: oracle.build_unit_index(K[u], V[u], p) for u in units}
    return K, V, idx, p


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        n = [i.get("num_threads", 1) for i in info if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(w, k, v, budget_s=15.0):
    """Time the float64 oracle's decode on a bounded sample of the same workload."""
    import oracle
    K, V, idx, p = oracle_setup(w, k, v)
    p10 = oracle.IndexParams(seg_len=w.seg_len, clusters_per_seg=w.clusters_per_seg, iters=w.iters,
                             n_sink=w.n_sink, local_window=w.local_window, budget_frac=w.budget_frac,
                             budget_k=w.budget_k)
    heads = 0
    t0 = time.perf_counter()
    step = 0
    while time.perf_counter() - t0 < budget_s:
        q = kvsynth.queries(w, step=step)
        Q = oracle.bf16_from_bits(q).reshape(w.units, w.group, 128)
        for u in range(w.units):
            oracle.decode_unit(Q[u], K[u], V[u], idx[u], p10)
            heads += w.group
        step += 1
    dt = time.perf_counter() - t0
    steps_equiv = heads / (w.units * w.group)
    # the build, for context: one segment-unit (one segment of one kv head, every round), timed once
    t0 = time.perf_counter()
    oracle.build_unit_index(K[0][:w.seg_len], V[0][:w.seg_len], p10)
    tb = time.perf_counter() - t0
    return {"value": steps_equiv / dt * w.batch * w.layers, "unit": UNIT, "cores": blas_threads(),
            "kind": "oracle",
            "build": {"segment_units_per_s": 1.0 / tb, "seconds": tb,
                      "sample": f"one segment-unit ({w.seg_len} tokens, {w.clusters_per_seg} clusters, "
                                f"{w.iters} rounds)",
                      "extrapolated_build_s": {n: kvsynth.get_workload(n).units * kvsynth.get_workload(n).n_segments
                                               * tb for n in [w.name] + EXTRA_CONFIGS}},
            "sample": f"{step} full decode steps ({heads} query heads) of {w.name} in {dt:.1f} s; the oracle index "
                      f"is a one-round k-means index built before timing"}


def run_reference(args, w, rank, world):
    """Reference arm: the float64 CPU oracle, timed on the host cores."""
    if rank != 0:
        return
    k, v = kvsynth.kv_cache(w)
    import oracle
    K, V, idx, p0 = oracle_setup(w, k, v)
    p = oracle.IndexParams(seg_len=w.seg_len, clusters_per_seg=w.clusters_per_seg, iters=w.iters, n_sink=w.n_sink,
                           local_window=w.local_window, budget_frac=w.budget_frac, budget_k=w.budget_k)
    # one step of this arm = one unit's decode (its G query heads in one oracle call, 1/U of a decode
    # step), as in the CPU baseline of the main arm; bounded to ~2 min in total
    t_one = time.perf_counter()
    Q = oracle.bf16_from_bits(kvsynth.queries(w, step=0)).reshape(w.units, w.group, 128)
    oracle.decode_unit(Q[0], K[0], V[0], idx[0], p)
    t_one = time.perf_counter() - t_one
    steps = min(args.steps, max(1, int(120.0 / max(t_one, 1e-4))))
    for s in range(args.warmup):
        oracle.decode_unit(Q[s % w.units], K[s % w.units], V[s % w.units], idx[s % w.units], p)
    t0 = time.perf_counter()
    for s in range(steps):
        u = s % w.units
        if u == 0:
            Q = oracle.bf16_from_bits(kvsynth.queries(w, step=s // w.units)).reshape(w.units, w.group, 128)
        oracle.decode_unit(Q[u], K[u], V[u], idx[u], p)
    dt = time.perf_counter() - t0
    value = steps / w.units / dt * w.batch * w.layers
    sample = (f"{steps} unit decodes ({w.group} query heads each, 1/{w.units} of a step) of {w.name}; "
              f"one-round k-means oracle index built before timing")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1000.0 / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "layers": w.layers, "n_q_heads": w.n_q_heads,
                       "n_kv_heads": w.n_kv_heads, "n_ctx": w.n_ctx, "clusters": w.clusters},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


CSRC = os.path.join(ROOT, "clustered_sparse_kv_gb300", "csrc")
DECODE_SOURCES = ["wi_decode.cu", "wi_pipe.cuh", "wi_tc.cuh", "wi_common.cuh", "wi_internal.h"]
KERNEL_NAMES = {"scores": "k_scores", "select_estimate": "k_select_estimate", "exact_merge": "k_exact_merge"}
EXTRA_CONFIGS = ["llama3-8b-b16-120k", "llama3-8b-1m-32l", "qwen2.5-7b-b8-262k"]


def decode_source_hash() -> str:
    """Hash of the decode kernels' sources: names the build that an ncu capture measured."""
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


_TRAFFIC_RE = re.compile(r"traffic: kernel=(\S+) workload=(\S+) source=([0-9a-f]{16}) dram_bytes_per_launch=(\d+)")


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of `kernel` on
    `workload`, from a `traffic:` line of an ncu summary under profiles/ that was captured from
    the current decode sources (same hash); None when no capture matches them."""
    want = decode_source_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for m in _TRAFFIC_RE.finditer(f.read()):
                if m.group(1) == kernel and m.group(2) == workload and m.group(3) == want:
                    return int(m.group(4))
    return None


def rank_seed(w, rank):
    """Each rank decodes its own independent replicas (weak scaling): seeds differ per rank."""
    return w.seed + 1000 * rank


def max_over_ranks(x, dist, device):
    """The job's time is the slowest rank's: max over ranks (identity on one rank)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, steps, batch, layers, seconds):
    """Whole-job throughput: every rank runs `steps` steps of batch x layers in `seconds` (max over ranks)."""
    return world * steps * batch * layers / seconds


def profile_run(wi, torch, w, dev, steps, dense=False, device_gen=False, tier=None):
    """One index of the workload and `steps` decode steps (each followed by a dense comparator step
    if asked; with `tier`, the index behind the host memory tier with that fraction of its pages
    cacheable, a replacement round after every step), nothing timed: the small case of the ncu
    captures."""
    if device_gen:
        g = kvsynth.DeviceGen(w, device=dev)
        kd, vd = g.kv_cache()
        qs = [g.queries(s) for s in range(steps)]
    else:
        k, v = kvsynth.kv_cache(w)
        kd = torch.from_numpy(k.view(np.int16)).to(dev)
        vd = torch.from_numpy(v.view(np.int16)).to(dev)
        qs = [torch.from_numpy(kvsynth.queries(w, step=s).view(np.int16)).to(dev) for s in range(steps)]
    ix = wi.WaveIndex.build(wi.config_from_workload(w), kd, vd)
    if tier is not None:
        ix.attach_tier(int(tier * (w.n_ctx // 16)), 512, async_rounds=False)
    for s in range(steps):
        ix.decode(qs[s])
        if dense:
            ix.dense_decode(qs[s])
        if tier is not None:
            ix.tier_round()
    torch.cuda.synchronize()
    ix.check()
    ix.free()
    print(json.dumps({"profile_steps": steps, "workload": w.name, "units": w.units}), flush=True)


class Timer:
    """CUDA-graph replays timed with CUDA events on one stream (the stream the library launches on)."""

    def __init__(self, torch, stream):
        self.torch, self.stream = torch, stream
        self.calls = {}  # id(graph) -> calls of fn captured in it

    def graph(self, fn, n):
        g = self.torch.cuda.CUDAGraph()
        with self.torch.cuda.graph(g, stream=self.stream):
            for s in range(n):
                fn(s)
        self.calls[id(g)] = n
        return g

    def replay(self, graphs):
        """Replay `graphs` in order between two events; milliseconds."""
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for g in graphs:
                g.replay()
            e1.record(self.stream)
        self.stream.synchronize()
        return e0.elapsed_time(e1)

    def replay_each(self, graphs, out):
        """Replay `graphs` in order with an event after each; appends (milliseconds, graph) per graph
        to `out` (a list, so that a thread can fill it)."""
        torch = self.torch
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
        with torch.cuda.stream(self.stream):
            ev[0].record(self.stream)
            for i, g in enumerate(graphs):
                g.replay()
                ev[i + 1].record(self.stream)
        self.stream.synchronize()
        out.extend((ev[i].elapsed_time(ev[i + 1]), g) for i, g in enumerate(graphs))

    def steps_plan(self, fn, steps, chunk):
        """Graphs covering exactly `steps` calls of fn (chunks of `chunk`), each replayed once untimed."""
        full, rest = divmod(steps, chunk)
        g_full = self.graph(fn, chunk) if full else None
        g_rest = self.graph(lambda s: fn(full * chunk + s), rest) if rest else None
        for g in (g_full, g_rest):
            if g is not None:
                self.replay([g])
        return [g_full] * full + ([g_rest] if g_rest is not None else [])


def algorithmic_bytes(w, vs_bytes, exact_rows_per_step, union_fraction):
    """Algorithmic bytes per launch of each decode kernel (index and K/V bytes the method must read;
    scratch traffic excluded), and per step (plus queries in and outputs out)."""
    cand = {"scores": w.units * w.clusters * (128 * 2 + 4),                  # mean keys + counts
            "select_estimate": w.units * w.clusters * (128 * vs_bytes + 4),   # value sums + counts
            "exact_merge": exact_rows_per_step * union_fraction * ROW_BYTES}   # GQA union of the rows
    step = sum(cand.values()) + w.units * w.group * 128 * (2 + 4)
    return cand, step


def union_fraction(replicas, w):
    """Rows in the union over each kv head's query heads / rows the heads select one by one
    (last step of every replica; steady rows counted once per head in both)."""
    loaded = union = 0
    steady = w.n_sink + w.local_window
    for ix in replicas:
        ids, _ = ix.selection()
        counts = np.empty((ix.units, ix.clusters), np.int32)
        import clustered_sparse_kv_gb300 as wi
        wi.wi_index_export(ix.handle, counts=counts)
        ids = ids.cpu().numpy()
        for uu in range(w.units):
            per_head = [ids[uu, hh][ids[uu, hh] >= 0] for hh in range(w.group)]
            loaded += sum(int(counts[uu][sel].sum()) + steady for sel in per_head)
            union += int(counts[uu][np.unique(np.concatenate(per_head))].sum()) + steady
    return union / max(loaded, 1)


def measure_decode(wi, torch, timer, w, replicas, qs, outs, steps, chunk, vs_bytes, iso_replays=3):
    """Decode steps over rotating replicas, and each decode kernel alone.  Returns a dict of
    timings and algorithmic bytes; the graphs of the timed region are returned to be replayed
    again (clock sampling) by the caller."""
    R, L = len(replicas), len(qs)
    stream = timer.stream

    def step(s):
        replicas[s % R].decode(qs[s % L], out=outs[s % R], stream=stream)

    graphs = timer.steps_plan(step, steps, chunk)
    rows1 = sum(wi.wi_profile_read(ix.handle, times=False)[2] for ix in replicas)   # warm replays counted
    ms = timer.replay(graphs)
    rows2 = sum(wi.wi_profile_read(ix.handle, times=False)[2] for ix in replicas)
    for ix in replicas:
        ix.check()
    rows_per_step = (rows2 - rows1) / max(steps, 1)
    # each kernel alone: a graph of `chunk` launches of that kernel over the same replicas (each repeats
    # its part of the replica's last step)
    iso = {}
    for kid, name in enumerate(wi.DECODE_KERNELS):
        g = timer.graph(lambda s: wi.wi_decode_kernel(replicas[s % R].handle, kid, qs[s % L], outs[s % R], stream),
                        chunk)
        timer.replay([g])
        t = timer.replay([g] * iso_replays)
        iso[name] = 1e3 * t / (iso_replays * chunk)
    for ix in replicas:
        ix.check()
    uf = union_fraction(replicas, w)
    cand, step_bytes = algorithmic_bytes(w, vs_bytes, rows_per_step, uf)
    return {"ms": ms, "graphs": graphs, "kernels_us": iso, "rows_per_step": rows_per_step, "union": uf,
            "bytes": cand, "step_bytes": step_bytes}


def roofline_of(d, w, hbm, peak_kind):
    """Roofline of the dominant decode kernel (the longest alone): algorithmic bytes per launch
    over its average launch duration, against the measured HBM peak."""
    iso = d["kernels_us"]
    dom = max(iso, key=iso.get)
    achieved = d["bytes"][dom] / (iso[dom] * 1e-6) / 1e9 if iso[dom] > 0 else 0.0
    return {"bound": "hbm", "kernel": KERNEL_NAMES[dom], "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_kind": peak_kind, "bytes_per_launch": d["bytes"][dom],
            "duration_us": iso[dom], "duration": "the kernel alone: graph of its launches, CUDA events",
            "traffic": ncu_traffic(KERNEL_NAMES[dom], w.name), "source": decode_source_hash()}


def build_record(wi, ix, w, secs_call, tf_peak, peak_kind):
    """The index build: `seconds` from the library's events around its kernels (first to last, after
    its allocations), `seconds_with_allocation` from events around the whole call."""
    st_ = wi.wi_index_build_stats(ix.handle)
    n_idx = w.n_ctx - w.n_sink - w.local_window
    flops = 2.0 * w.iters * w.units * n_idx * w.clusters_per_seg * 128
    assign_s = st_["assign_ms"] / 1e3
    secs = st_["build_ms"] / 1e3
    tf = flops / assign_s / 1e12
    return {"seconds": secs, "seconds_with_allocation": secs_call,
            "segment_units_per_s": w.units * w.n_segments / secs, "assign_flop": flops,
            "assign_seconds": assign_s, "assign_launches": st_["assign_launches"], "assign_tflops": tf,
            "assign_roofline": {"bound": "tensor", "achieved": tf, "peak": tf_peak, "unit": "TFLOP/s",
                                "frac": tf / tf_peak, "peak_kind": peak_kind},
            "assign_tflops_over_build": flops / secs / 1e12,
            "build_frac_of_tensor_peak": flops / secs / 1e12 / tf_peak}


def timed_build(wi, torch, cfg, k, v, stream):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        ix = wi.WaveIndex.build(cfg, k, v, stream=stream)
        e1.record(stream)
    stream.synchronize()
    ix.check()
    return ix, e0.elapsed_time(e1) / 1e3


def dense_record(wi, torch, timer, w, replicas, qs, outs, steps, chunk, hbm, peak_kind, wave_ms):
    """The dense comparator (full attention over every cached token) on the same replicas and queries."""
    R, L = len(replicas), len(qs)
    stream = timer.stream
    n = max(1, min(chunk, steps))
    g = timer.graph(lambda s: replicas[s % R].dense_decode(qs[s % L], out=outs[s % R], stream=stream), n)
    timer.replay([g])
    reps = max(1, steps // n)
    d_ms = timer.replay([g] * reps) / (reps * n)
    for ix in replicas:
        ix.check()
    d_bytes = w.units * w.n_ctx * ROW_BYTES + w.units * w.group * 128 * (2 + 4)
    d_gbs = d_bytes / (d_ms * 1e-3) / 1e9
    return {"kernel": "k_dense_decode", "steps": reps * n, "ms_per_step": d_ms,
            "value": w.batch * w.layers / (d_ms / 1e3), "unit": UNIT, "bytes_per_step": d_bytes,
            "hbm_gbs": d_gbs, "peak": hbm, "frac": d_gbs / hbm, "peak_kind": peak_kind,
            "wave_index_speedup": d_ms / wave_ms,
            # against a full-attention pass that would stream its bytes at the measured copy peak
            "wave_index_speedup_vs_dense_at_peak": d_bytes / (hbm * 1e9) / (wave_ms * 1e-3)}


def measure_config(wi, torch, timer, name, dev, hbm, tf_burst, peak_kind, steps, dense_steps):
    """Full-size record of one more workload, generated on the device: build, decode steps, kernels
    alone, dense comparator, and (append workloads) the decode steps that append a token."""
    w = kvsynth.get_workload(name)
    stream = timer.stream
    t0 = time.perf_counter()
    gen = kvsynth.DeviceGen(w, device=dev, stream=stream)
    k, v = gen.kv_cache(stream=stream)
    stream.synchronize()
    gen_s = time.perf_counter() - t0
    cfg = wi.config_from_workload(w)
    ix, build_s = timed_build(wi, torch, cfg, k, v, stream)
    build = build_record(wi, ix, w, build_s, tf_burst, peak_kind)
    L = min(32, steps)
    qs = [gen.queries(s, stream=stream) for s in range(L)]
    out = torch.empty((w.batch, w.layers, w.n_q_heads, 128), dtype=torch.float32, device=dev)
    for s in range(3):
        ix.decode(qs[s], out=out, stream=stream)
    stream.synchronize()
    ix.check()
    d = measure_decode(wi, torch, timer, w, [ix], qs, [out], steps, L, 4, iso_replays=2)
    ms_per_step = d["ms"] / steps
    rec = {"workload": w.name, "batch": w.batch, "layers": w.layers, "n_q_heads": w.n_q_heads,
           "n_kv_heads": w.n_kv_heads, "n_ctx": w.n_ctx, "units": w.units, "clusters": w.clusters,
           "k": ix.k_max, "steps": steps, "ms_per_step": ms_per_step, "steps_per_s": 1e3 / ms_per_step,
           "value": w.batch * w.layers * 1e3 / ms_per_step, "unit": "steps/s (batch×layer)",
           "step_bytes": d["step_bytes"], "step_hbm_gbs": d["step_bytes"] / (ms_per_step * 1e-3) / 1e9,
           "kernels_us_alone": d["kernels_us"], "roofline": roofline_of(d, w, hbm, peak_kind),
           "exact_rows_per_step": d["rows_per_step"], "exact_union_fraction": d["union"],
           "decode_layout": wi.wi_decode_layout(ix.handle), "generate_s": gen_s,
           "l2": f"one replica: {d['step_bytes'] / 1e9:.2f} GB per step, far above L2", "build": build}
    rec["step_frac"] = rec["step_hbm_gbs"] / hbm
    if dense_steps > 0:
        rec["dense_comparator"] = dense_record(wi, torch, timer, w, [ix], qs, [out], dense_steps, 8, hbm,
                                               peak_kind, ms_per_step)
    ix.free()
    if w.append and w.decode_steps > 0:
        # the workload's decode on a fresh build: every step attends, then appends its token (not
        # graph-replayable: the append slot advances), launched step by step, timed with events
        T = w.decode_steps
        ka, va = gen.kv_cache(p0=w.n_ctx, p1=w.n_ctx + T, stream=stream)
        kn = [ka[:, :, :, t].contiguous() for t in range(T)]
        vn = [va[:, :, :, t].contiguous() for t in range(T)]
        qa = [gen.queries(t, stream=stream) for t in range(T)]
        gen.kv_cache(out_k=k, out_v=v, stream=stream)   # the unpermuted cache again
        ix2, _ = timed_build(wi, torch, cfg, k, v, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for t in range(T):
                ix2.decode(qa[t], kn[t], vn[t], out=out, stream=stream)
            e1.record(stream)
        stream.synchronize()
        ix2.check()
        a_ms = e0.elapsed_time(e1) / T
        rec["append"] = {"steps": T, "ms_per_step": a_ms, "steps_per_s": 1e3 / a_ms,
                         "value": w.batch * w.layers * 1e3 / a_ms,
                         "timing": f"{T} steps launched one by one (each appends its token), CUDA events"}
        ix2.free()
    del k, v, gen
    torch.cuda.empty_cache()
    return rec


def variant_accuracy(wi, torch, w, k_dev, v_dev, qs, dev, stream):
    """Relative L2 of the wave-index output against full attention (the dense comparator, itself
    checked against the float64 definition by the tests) per (unit, query head), for the default
    index and its two variants: information only."""
    res = {}
    for name, vsb, grp in (("default", 0, 0), ("valsum_bf16", 1, 0), ("group_topk", 0, 1)):
        cfg = wi.config_from_workload(w)
        cfg.valsum_bf16, cfg.group_topk = vsb, grp
        ix = wi.WaveIndex.build(cfg, k_dev.clone(), v_dev.clone(), stream=stream)
        errs = []
        for q in qs:
            o = ix.decode(q, stream=stream)
            r = ix.dense_decode(q, stream=stream)
            stream.synchronize()
            o64 = o.double().reshape(-1, 128)
            r64 = r.double().reshape(-1, 128)
            errs.append((torch.linalg.norm(o64 - r64, dim=1) / torch.linalg.norm(r64, dim=1)).cpu().numpy())
        ix.check()
        ix.free()
        e = np.concatenate(errs)
        res[name] = {"rel_l2_mean": float(e.mean()), "rel_l2_max": float(e.max()), "samples": int(e.size)}
    return res


def h2d_copy_gbs(torch, dev, stream, gib=1.0):
    """Host-to-device copy rate from page-locked memory (the copy engines over the CPU-GPU link),
    the reference rate for rows read from host memory."""
    n = int(gib * (1 << 30))
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        d.copy_(h, non_blocking=True)
        e0.record(stream)
        for _ in range(3):
            d.copy_(h, non_blocking=True)
        e1.record(stream)
    e1.synchronize()
    rate = 3 * n / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del h, d
    return rate


def tier_record(wi, torch, w, k_dev, v_dev, dev, stream, steps=256, warmup=16):
    """The host memory tier (wave buffer) on the main workload: K/V rows in page-locked host memory,
    a device page cache with LRU rounds on the library's thread.  Each case builds a fresh index,
    attaches the tier and runs steps as a decoding loop does: each step launched, then its output
    waited for before the next (no graphs: the rounds enqueue work between steps); the untiered index
    is timed the same way.  Two query streams: a fresh query every step (the bench's stream) and each
    query held for 8 steps (temporal locality, which the pages credit real decoding with); last, one query
    for the whole run, whose pages all end up cached (the hit path alone)."""
    cfg = wi.config_from_workload(w)
    pages = w.n_ctx // 16
    qs = [torch.from_numpy(kvsynth.queries(w, step=s, seed=w.seed + 77).view(np.int16)).to(dev)
          for s in range(steps + warmup)]
    out = torch.empty((w.batch, w.layers, w.n_q_heads, 128), dtype=torch.float32, device=dev)

    def run(ix, hold, rounds_async):
        with torch.cuda.stream(stream):
            for s in range(warmup):
                ix.decode(qs[s // hold], out=out, stream=stream)
                stream.synchronize()
                if getattr(ix, "_tier", False) and not rounds_async:
                    ix.tier_round(stream=stream)   # rounds after every warm-up step, none while timed
            before = ix.tier_stats() if getattr(ix, "_tier", False) else None
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for s in range(warmup, warmup + steps):
                ix.decode(qs[s // hold], out=out, stream=stream)
                stream.synchronize()
            e1.record(stream)
            e1.synchronize()
        return e0.elapsed_time(e1) / steps, before

    cases = []
    every = steps + warmup
    for frac, hold, rounds_async in [(None, 1, True), (0.0, 1, True), (0.25, 1, True), (0.25, 8, True),
                                     (1.0, 8, True), (1.0, every, True), (None, every, True), (1.0, every, False)]:
        ix = wi.WaveIndex.build(cfg, k_dev.clone(), v_dev.clone(), stream=stream)
        stream.synchronize()
        slots = 0 if frac is None else int(frac * pages)
        if frac is not None:
            ix.attach_tier(slots, 512, async_rounds=rounds_async, stream=stream)
            ix._tier = True
        ms, before = run(ix, hold, rounds_async)
        rec = {"slots_fraction": frac, "query_held_steps": hold, "rounds_while_timed": rounds_async and frac is not None,
               "ms_per_step": ms, "steps_per_s": 1e3 / ms}
        if not rounds_async or frac is None:   # the exact kernel alone: a graph of 64 launches of it
            timer = Timer(torch, stream)
            kid = wi.DECODE_KERNELS.index("exact_merge")
            g = timer.graph(lambda s_: wi.wi_decode_kernel(ix.handle, kid, qs[-1], out, stream), 64)
            timer.replay([g])
            rec["exact_alone_us"] = 1e3 * timer.replay([g] * 3) / (3 * 64)
            del g
        if frac is not None:
            st = ix.tier_stats()
            rc = st["rows_from_cache"] - before["rows_from_cache"]
            rh = st["rows_from_host"] - before["rows_from_host"]
            rec.update(slots_per_unit=slots, pages_per_unit=pages,
                       row_hit_ratio=rc / max(rc + rh, 1),
                       host_bytes_per_step=rh * 512 / steps,
                       host_read_gbs=rh * 512 / steps / (ms * 1e-3) / 1e9,
                       rounds=st["rounds"] - before["rounds"],
                       admitted=st["admitted"] - before["admitted"], evicted=st["evicted"] - before["evicted"])
        ix.check()
        ix.free()
        cases.append(rec)
    link = h2d_copy_gbs(torch, dev, stream)
    for rec in cases:   # the miss path's roofline: rows read from host memory against the link's copy rate
        if "host_read_gbs" in rec:
            rec["link_frac"] = rec["host_read_gbs"] / link
    return {"workload": w.name, "page_rows": 16, "admit_per_round": 512,
            "device_kv_bytes_untiered": w.units * w.n_ctx * 512,
            "h2d_copy_gbs": link,
            "timing": f"{steps} steps after {warmup}, each launched after the previous step's output was waited "
                      f"for; CUDA events on the launching stream around the loop",
            "cases": cases}


def spawn_ranks(n):
    """--gpus N without a launcher: run this script under torch.distributed.run with N ranks."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--replicas", type=int, default=8)
    ap.add_argument("--chunk", type=int, default=64, help="decode steps per captured graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-build-timing", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--configs", default=",".join(EXTRA_CONFIGS),
                    help="comma-separated further workloads measured at full size (empty: none)")
    ap.add_argument("--config-steps", type=int, default=256, help="decode steps timed per further workload")
    ap.add_argument("--no-accuracy", action="store_true", help="skip the variant accuracy record")
    ap.add_argument("--no-tier", action="store_true", help="skip the host memory tier record")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="profiling run: build one index of the workload, run this many decode steps, "
                         "print nothing else (a small case for ncu captures)")
    ap.add_argument("--profile-dense", action="store_true",
                    help="with --profile-steps: also run the dense comparator after every decode step")
    ap.add_argument("--profile-device-gen", action="store_true",
                    help="with --profile-steps: generate the workload on the device")
    ap.add_argument("--profile-tier", type=float, default=None,
                    help="with --profile-steps: the index behind the host memory tier, this fraction of its "
                         "pages cacheable")
    ap.add_argument("--profile-units", default="",
                    help="with --profile-steps: batch,layers,kv_heads of a smaller case of the workload "
                         "(query heads per kv head kept), for captures whose traffic scales by units")
    ap.add_argument("--valsum-bf16", action="store_true",
                    help="the index variant whose decode reads a bf16 copy of the value sums")
    ap.add_argument("--group-topk", action="store_true",
                    help="the variant whose query heads share one top-k per kv head (summed scores)")
    ap.add_argument("--dense-steps", type=int, default=640,
                    help="dense comparator steps timed after the wave-index region (0: skip)")
    args = ap.parse_args()

    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(spawn_ranks(args.gpus))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}")
    w = kvsynth.get_workload(args.workload)

    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import torch
    import clustered_sparse_kv_gb300 as wi

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    seed = rank_seed(w, rank)
    if args.profile_steps > 0:
        if args.profile_units:
            b, l, h = (int(x) for x in args.profile_units.split(","))
            w = w.with_(batch=b, layers=l, n_kv_heads=h, n_q_heads=h * w.group)
        profile_run(wi, torch, w, dev, args.profile_steps, dense=args.profile_dense,
                    device_gen=args.profile_device_gen, tier=args.profile_tier)
        return
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    k, v = kvsynth.kv_cache(w, seed=seed)
    k_dev = torch.from_numpy(k.view(np.int16)).to(dev)
    v_dev = torch.from_numpy(v.view(np.int16)).to(dev)
    cfg = wi.config_from_workload(w)
    cfg.valsum_bf16 = 1 if args.valsum_bf16 else 0
    cfg.group_topk = 1 if args.group_topk else 0
    vs_bytes = 2 if args.valsum_bf16 else 4
    R = args.replicas
    stream = torch.cuda.Stream(device=dev)
    timer = Timer(torch, stream)
    replicas = []
    build = None
    for r in range(R):
        ix, secs = timed_build(wi, torch, cfg, k_dev.clone(), v_dev.clone(), stream)
        if r == 1 and not args.no_build_timing:   # replica 0 is the warm-up build
            build = build_record(wi, ix, w, secs, tf_burst, peak_kind)
        replicas.append(ix)

    # queries: one per step of a chunk, resident on the device before timing
    L = args.chunk
    qs = [torch.from_numpy(kvsynth.queries(w, step=s, seed=seed).view(np.int16)).to(dev) for s in range(L)]
    outs = [torch.empty((w.batch, w.layers, w.n_q_heads, 128), dtype=torch.float32, device=dev) for _ in range(R)]
    with torch.cuda.stream(stream):
        for s in range(max(args.warmup, 3)):
            replicas[s % R].decode(qs[s % L], out=outs[s % R], stream=stream)
        stream.synchronize()
    for ix in replicas:
        ix.check()

    K = args.steps
    barrier()
    d = measure_decode(wi, torch, timer, w, replicas, qs, outs, K, L, vs_bytes)
    barrier()
    ms = max_over_ranks(d["ms"], dist, dev)
    # clocks under the same load: the timed graphs replayed for ~1.6 s (another thread) while the
    # sampler runs inside that window
    import threading
    soak = max(1, int(math.ceil(1.6 / max(d["ms"] / 1e3, 1e-6))))
    soak_ms = []
    th = threading.Thread(target=timer.replay_each, args=(d["graphs"] * soak, soak_ms))
    th.start()
    time.sleep(0.05)
    with ClockSampler(local) as clocks:
        time.sleep(0.8)
    th.join()
    ms_per_step = ms / K
    value = job_value(world, K, w.batch, w.layers, ms / 1e3)
    # spread of the step time: each graph replay of the clock-sampling window gives its mean step time
    per_step_us = [1e3 * t / timer.calls[id(g)] for t, g in soak_ms]
    step_dist = {"p10": float(np.percentile(per_step_us, 10)), "median": float(np.median(per_step_us)),
                 "p90": float(np.percentile(per_step_us, 90)), "samples": len(per_step_us), "unit": "us",
                 "over": f"mean step time of each graph replay (graphs of up to {L} steps) in the "
                         f"clock-sampling window"}
    step_bytes = d["step_bytes"]

    # e2e: host buffers through the C ABI, copies inside the timed region
    qh = [torch.from_numpy(kvsynth.queries(w, step=L + s, seed=seed).view(np.int16)).pin_memory()
          for s in range(8)]
    oh = torch.empty((w.batch, w.layers, w.n_q_heads, 128), dtype=torch.float32).pin_memory()
    qbuf = torch.empty_like(qh[0]).pin_memory()  # the caller's input buffer, refilled every step
    for s in range(max(3, R)):  # every replica once: its first host-buffer call captures its graph
        qbuf.copy_(qh[s % 8])
        wi.wi_decode_step_host(replicas[s % R].handle, qbuf, oh, stream=stream)
    E = max(1, min(args.e2e_steps, K))
    barrier()
    t0 = time.perf_counter()
    for s in range(E):
        qbuf.copy_(qh[s % 8])
        wi.wi_decode_step_host(replicas[s % R].handle, qbuf, oh, stream=stream)
    e2e_s = time.perf_counter() - t0
    barrier()
    e2e_s = max_over_ranks(e2e_s, dist, dev)
    e2e_val = job_value(world, E, w.batch, w.layers, e2e_s)
    for ix in replicas:
        ix.check()

    dense = None
    if args.dense_steps > 0:
        dense = dense_record(wi, torch, timer, w, replicas, qs, outs, args.dense_steps, L, hbm, peak_kind,
                             ms_per_step)

    accuracy = None
    if rank == 0 and world == 1 and not args.no_accuracy:
        accuracy = variant_accuracy(wi, torch, w, k_dev, v_dev, qs[:4], dev, stream)

    tier = None
    if rank == 0 and world == 1 and not args.no_tier:
        tier = tier_record(wi, torch, w, k_dev, v_dev, dev, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, k, v)

    line_cfg = {"workload": w.name, "batch": w.batch, "layers": w.layers, "n_q_heads": w.n_q_heads,
                "n_kv_heads": w.n_kv_heads, "head_dim": 128, "n_ctx": w.n_ctx, "seg_len": w.seg_len,
                "clusters_per_seg": w.clusters_per_seg, "clusters": w.clusters,
                "k": replicas[0].k_max, "steady": w.n_sink + w.local_window,
                "l2": f"inputs larger than L2: {R} rotating index+KV replicas "
                      f"({R * (w.units * w.n_ctx * 512 + d['bytes']['scores'] + d['bytes']['select_estimate']) / 1e9:.1f} GB)",
                "timing": f"CUDA graphs of {L} steps replayed (each once untimed first); events on the "
                          f"launching stream",
                "decode_layout": wi.wi_decode_layout(replicas[0].handle),
                "valsum": "bf16" if args.valsum_bf16 else "fp32",
                "retrieval": "per kv head (summed scores)" if args.group_topk else "per query head"}
    for ix in replicas:
        ix.free()
    replicas = []
    del k_dev, v_dev
    torch.cuda.empty_cache()

    configs = []
    names = [c for c in args.configs.split(",") if c] if world == 1 else []
    for name in names:
        if name == w.name:
            continue
        steps_c = args.config_steps if name != "llama3-8b-1m-32l" else max(8, args.config_steps // 8)
        configs.append(measure_config(wi, torch, timer, name, dev, hbm, tf_burst, peak_kind, steps_c,
                                      dense_steps=16 if args.dense_steps > 0 else 0))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "accumulate": "fp32", "data": "synthetic",
            "config": line_cfg,
            "roofline": roofline_of(d, w, hbm, peak_kind),
            "step_us_dist": step_dist,
            "step_hbm_gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
            "step_frac": step_bytes / (ms_per_step * 1e-3) / 1e9 / hbm,
            "step_bytes": step_bytes,
            "exact_rows_per_step": d["rows_per_step"],
            "exact_union_fraction": d["union"],
            "kernels_us_alone": d["kernels_us"],
            "gpu_launches": K * wi.WI_NUM_DECODE_KERNELS,
            "e2e": {"value": e2e_val, "unit": UNIT, "steps": E,
                    "h2d_bytes_per_step": w.units * w.group * 128 * 2,
                    "d2h_bytes_per_step": w.units * w.group * 128 * 4},
            "cpu_baseline": cpu,
            "clocks": dict(clocks.summary(), window="nvidia-smi every 100 ms while the timed graphs are "
                                                    "replayed for ~1.6 s right after the timed region"),
        }
        if build is not None:
            line["build"] = build
        if dense is not None:
            line["dense_comparator"] = dense
        if accuracy is not None:
            line["variant_accuracy"] = accuracy
        if tier is not None:
            line["wave_buffer"] = tier
        if configs:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
