#!/usr/bin/env python
"""Wave-index decode benchmark (one JSON line on rank 0).

Workload: the Llama-3-8B-shaped single-layer decode -- 131072 tokens, 32 query
heads over 8 kv heads, head size 128, bf16 KV, 16 segments x 512 clusters per
kv head, retrieval budget 148 clusters (1.8%), steady zone 4 + 64 tokens --
on seeded synthetic data (kvsynth).  A step is one decode step of the whole
batch: centroid scoring with the fused estimation, top-k, union, exact
attention over steady + retrieved rows, LSE merge.

Timing: the decode steps are captured in CUDA graphs and replayed; each
step runs on one of R independent index + KV replicas in turn (R x ~90 MB
of index and retrieved rows per step, 4.7 GB of replicas in total, far above
the 129 MB L2), with a different query per step.  Kernel durations come from
CUDA events that the library records around each kernel on the launching
stream inside the same timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
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
    return {"value": steps_equiv / dt * w.batch * w.layers, "unit": UNIT, "cores": blas_threads(),
            "kind": "oracle",
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
    # one step = one query head of one unit (1/32 of a decode step), bounded to ~2 min in total
    t_one = time.perf_counter()
    q = kvsynth.queries(w, step=0)
    Q = oracle.bf16_from_bits(q).reshape(w.units, w.group, 128)
    oracle.decode_unit(Q[0][:1], K[0], V[0], idx[0], p)
    t_one = time.perf_counter() - t_one
    steps = min(args.steps, max(1, int(120.0 / max(t_one, 1e-4))))
    for s in range(args.warmup):
        oracle.decode_unit(Q[s % w.units][:1], K[s % w.units], V[s % w.units], idx[s % w.units], p)
    t0 = time.perf_counter()
    for s in range(steps):
        u, h = (s // w.group) % w.units, s % w.group
        if h == 0 and u == 0:
            Q = oracle.bf16_from_bits(kvsynth.queries(w, step=s)).reshape(w.units, w.group, 128)
        oracle.decode_unit(Q[u][h:h + 1], K[u], V[u], idx[u], p)
    dt = time.perf_counter() - t0
    per_step = w.units * w.group
    value = steps / per_step / dt * w.batch * w.layers
    sample = (f"{steps} query-head decodes (1/{per_step} of a step each) of {w.name}; one-round k-means oracle "
              f"index built before timing")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1000.0 / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "layers": w.layers, "n_q_heads": w.n_q_heads,
                       "n_kv_heads": w.n_kv_heads, "n_ctx": w.n_ctx, "clusters": w.clusters},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture of the
# current kernels on this workload (profiles/decode_kernels_llama3-8b-131k.md); to be retaken whenever
# a kernel changes.
NCU_TRAFFIC = {("llama3-8b-131k", "exact_merge"): 38_799_104 + 20_992}


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


def profile_run(wi, torch, w, dev, steps, dense=False):
    """One index of the workload and `steps` decode steps (each followed by a dense comparator step
    if asked), nothing timed."""
    k, v = kvsynth.kv_cache(w)
    kd = torch.from_numpy(k.view(np.int16)).to(dev)
    vd = torch.from_numpy(v.view(np.int16)).to(dev)
    ix = wi.WaveIndex.build(wi.config_from_workload(w), kd, vd)
    for s in range(steps):
        q = torch.from_numpy(kvsynth.queries(w, step=s).view(np.int16)).to(dev)
        ix.decode(q)
        if dense:
            ix.dense_decode(q)
    torch.cuda.synchronize()
    ix.check()
    ix.free()
    print(json.dumps({"profile_steps": steps, "workload": w.name}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--replicas", type=int, default=8)
    ap.add_argument("--chunk", type=int, default=64, help="decode steps per captured graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-build-timing", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--no-kernel-events", action="store_true",
                    help="do not record per-kernel events inside the timed region (value only)")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="profiling run: build one index of the workload, run this many decode steps, "
                         "print nothing else (a small case for ncu captures)")
    ap.add_argument("--profile-dense", action="store_true",
                    help="with --profile-steps: also run the dense comparator after every decode step")
    ap.add_argument("--valsum-bf16", action="store_true",
                    help="the index variant whose decode reads a bf16 copy of the value sums")
    ap.add_argument("--group-topk", action="store_true",
                    help="the variant whose query heads share one top-k per kv head (summed scores)")
    ap.add_argument("--dense-steps", type=int, default=640,
                    help="dense comparator steps timed after the wave-index region (0: skip)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
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
        profile_run(wi, torch, w, dev, args.profile_steps, dense=args.profile_dense)
        return
    k, v = kvsynth.kv_cache(w, seed=seed)
    k_dev = torch.from_numpy(k.view(np.int16)).to(dev)
    v_dev = torch.from_numpy(v.view(np.int16)).to(dev)
    cfg = wi.config_from_workload(w)
    cfg.valsum_bf16 = 1 if args.valsum_bf16 else 0
    cfg.group_topk = 1 if args.group_topk else 0
    vs_bytes = 2 if args.valsum_bf16 else 4
    R = args.replicas
    stream = torch.cuda.Stream(device=dev)
    replicas = []
    build = None
    with torch.cuda.stream(stream):
        for r in range(R):
            kr, vr = k_dev.clone(), v_dev.clone()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ix = wi.WaveIndex.build(cfg, kr, vr, stream=stream)
            e1.record(stream)
            stream.synchronize()
            ix.check()
            if r == 1 and not args.no_build_timing:   # replica 0 is the warm-up build
                secs = e0.elapsed_time(e1) / 1e3
                st_ = wi.wi_index_build_stats(ix.handle)
                n_idx = w.n_ctx - w.n_sink - w.local_window
                flops = 2.0 * w.iters * w.units * n_idx * w.clusters_per_seg * 128
                assign_s = st_["assign_ms"] / 1e3
                tf = flops / assign_s / 1e12
                build = {"seconds": secs, "segment_units_per_s": w.units * w.n_segments / secs,
                         "assign_flop": flops, "assign_seconds": assign_s,
                         "assign_launches": st_["assign_launches"], "assign_tflops": tf,
                         "assign_roofline": {"bound": "tensor", "achieved": tf, "peak": peaks()[1],
                                             "unit": "TFLOP/s", "frac": tf / peaks()[1],
                                             "peak_kind": peaks()[3]},
                         "assign_tflops_over_build": flops / secs / 1e12}
            replicas.append(ix)
    del k_dev, v_dev

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
    full, rest = divmod(K, L)

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in range(nsteps):
                replicas[s % R].decode(qs[s], out=outs[s % R], stream=stream)
        return g

    def run_region(g_full, g_rest):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(full):
                g_full.replay()
            if g_rest is not None:
                g_rest.replay()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1)

    # graphs without per-kernel events: the timed region of `value`
    g_full = capture(L) if full else None
    g_rest = capture(rest) if rest else None
    # graphs with per-kernel events recorded by the library: kernel durations (a second region)
    gk_full = gk_rest = None
    if not args.no_kernel_events:
        for ix in replicas:
            wi.wi_profile_begin(ix.handle, max(1, math.ceil(L / R)))
        gk_full = capture(L) if full else None
        gk_rest = capture(rest) if rest else None
    stream.synchronize()
    rows0 = [wi.wi_profile_read(ix.handle, times=False)[2] for ix in replicas]

    barrier()
    with ClockSampler(local) as clocks:
        ms = run_region(g_full, g_rest)
    barrier()
    ms = max_over_ranks(ms, dist, dev)
    for ix in replicas:
        ix.check()
    ms_events = None
    if gk_full is not None or gk_rest is not None:
        rows0 = [wi.wi_profile_read(ix.handle, times=False)[2] for ix in replicas]
        ms_events = run_region(gk_full, gk_rest)

    # per-kernel durations (events recorded by the library in the timed region)
    kern_ms = {n: 0.0 for n in wi.DECODE_KERNELS}
    kern_steps = 0
    rows = 0
    for ix, r0 in zip(replicas, rows0):
        d, st, rr = wi.wi_profile_read(ix.handle)
        for n in kern_ms:
            kern_ms[n] += d[n]
        kern_steps += st
        rows += rr - r0
    mean_us = {n: 1e3 * kern_ms[n] / max(kern_steps, 1) for n in kern_ms}
    rows_per_step = rows / max(K, 1)          # rows loaded by exact attention, per query head
    # the algorithmic exact-zone bytes count each row once per kv head (union over the group's heads);
    # measure the union / per-head ratio on each replica's last step
    loaded = union = 0
    for ix in replicas:
        ids, _ = ix.selection()
        counts = ix.export()["counts"]
        ids, counts = ids.cpu().numpy(), counts.cpu().numpy()
        steady = w.n_sink + w.local_window
        for uu in range(w.units):
            per_head = [ids[uu, hh][ids[uu, hh] >= 0] for hh in range(w.group)]
            loaded += sum(int(counts[uu][sel].sum()) + steady for sel in per_head)
            union += int(counts[uu][np.unique(np.concatenate(per_head))].sum()) + steady
    dedup = union / max(loaded, 1)
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    bytes_d1 = w.units * w.clusters * (INDEX_BYTES_PER_CLUSTER - 128 * (4 - vs_bytes))
    bytes_d3 = rows_per_step * dedup * ROW_BYTES
    cand = {"scores": w.units * w.clusters * (128 * 2 + 4),              # mu + count
            "select_estimate": w.units * w.clusters * (128 * vs_bytes + 4),  # value sums + count
            "exact_merge": bytes_d3}
    dom = max(cand, key=lambda n: mean_us[n])
    achieved = cand[dom] / (mean_us[dom] * 1e-6) / 1e9 if mean_us[dom] > 0 else 0.0
    step_bytes = bytes_d1 + bytes_d3 + w.units * w.group * 128 * (2 + 4)
    ms_per_step = ms / K
    value = job_value(world, K, w.batch, w.layers, ms / 1e3)

    # e2e: host buffers through the C ABI, copies inside the timed region
    for ix in replicas:
        wi.wi_profile_begin(ix.handle, 0)
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

    # the dense comparator (full attention over every cached token) on the same replicas and queries:
    # graphs of L steps, CUDA events on the launching stream, after the wave-index regions
    dense = None
    if args.dense_steps > 0:
        with torch.cuda.stream(stream):
            for s in range(3):
                replicas[s % R].dense_decode(qs[s % L], out=outs[s % R], stream=stream)
            stream.synchronize()
            gd = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gd, stream=stream):
                for s in range(L):
                    replicas[s % R].dense_decode(qs[s], out=outs[s % R], stream=stream)
            nd = max(1, args.dense_steps // L)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(nd):
                gd.replay()
            e1.record(stream)
        stream.synchronize()
        for ix in replicas:
            ix.check()
        d_ms = max_over_ranks(e0.elapsed_time(e1) / (nd * L), dist, dev)
        d_bytes = w.units * w.n_ctx * ROW_BYTES + w.units * w.group * 128 * (2 + 4)
        d_gbs = d_bytes / (d_ms * 1e-3) / 1e9
        dense = {"kernel": "k_dense_decode", "steps": nd * L, "ms_per_step": d_ms,
                 "value": job_value(world, 1, w.batch, w.layers, d_ms / 1e3), "unit": UNIT,
                 "bytes_per_step": d_bytes, "hbm_gbs": d_gbs, "peak": hbm, "frac": d_gbs / hbm,
                 "peak_kind": peak_kind, "wave_index_speedup": d_ms / ms_per_step}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, k, v)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "ms_per_step_with_kernel_events": (ms_events / K if ms_events else None),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "accumulate": "fp32", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "layers": w.layers, "n_q_heads": w.n_q_heads,
                       "n_kv_heads": w.n_kv_heads, "head_dim": 128, "n_ctx": w.n_ctx, "seg_len": w.seg_len,
                       "clusters_per_seg": w.clusters_per_seg, "clusters": w.clusters,
                       "k": replicas[0].k_max, "steady": w.n_sink + w.local_window,
                       "l2": f"inputs larger than L2: {R} rotating index+KV replicas "
                             f"({R * (w.units * w.n_ctx * 512 + bytes_d1) / 1e9:.1f} GB)",
                       "timing": f"CUDA graphs of {L} steps replayed; events on the launching stream",
                       "decode_layout": wi.wi_decode_layout(replicas[0].handle),
                       "valsum": "bf16" if args.valsum_bf16 else "fp32",
                       "retrieval": "per kv head (summed scores)" if args.group_topk else "per query head"},
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_kind": peak_kind,
                         "bytes_per_launch": cand[dom], "traffic": NCU_TRAFFIC.get((w.name, dom))},
            "step_hbm_gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
            "step_bytes": step_bytes,
            "exact_rows_per_step": rows_per_step,
            "exact_union_fraction": dedup,
            "kernels_us": mean_us,
            "gpu_launches": K * wi.WI_NUM_DECODE_KERNELS,
            "e2e": {"value": e2e_val, "unit": UNIT, "steps": E,
                    "h2d_bytes_per_step": w.units * w.group * 128 * 2,
                    "d2h_bytes_per_step": w.units * w.group * 128 * 4},
            "cpu_baseline": cpu,
            "clocks": clocks.summary(),
        }
        if build is not None:
            line["build"] = build
        if dense is not None:
            line["dense_comparator"] = dense
        print(json.dumps(line), flush=True)
    for ix in replicas:
        ix.free()
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
