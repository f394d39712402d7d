#!/usr/bin/env python3
"""Throughput of the BeaconKV eviction step on GB300, one JSON line on stdout.

A step is one eviction period of the whole hot path for every layer and
sequence of the workload: one bkv_evict (RoPE table, one fused kernel for
scoring, keep-set selection and in-place K/V compaction, FPS of beacons +
recents) followed by the
period's bkv_append_queries calls (one per decode step). The metric is
evictions per second, one eviction being one (layer, sequence) pair.

Default workload: Qwen3-4B head shape (36 layers, 32 query / 8 KV heads,
d = 128), batch 192, budget 2048, period 16, prefix 4, recent 16, FPS 32 -> 16.
Its K/V cache (58 GB) is larger than L2, so no flush is needed between steps.
Inputs are synthetic and seeded (synth/).

--impl reference times the CPU oracle (oracle/) on this host's cores on a
bounded sample of the same workload.
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

FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples taken every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def aggregate(per_rank_evictions: int, elapsed_s_max: float, world: int) -> float:
    """Whole-job evictions/s: every rank processes its own full workload (weak scaling)."""
    return per_rank_evictions * world / elapsed_s_max


def max_over_ranks(ms: float, world: int, device) -> float:
    """The largest of the ranks' elapsed times: the job ends with its slowest rank."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- byte model

def kernel_bytes(w, R: int, rows_moved_per_launch: float, heads_total: int, n_fps: int) -> dict:
    """Algorithmic DRAM bytes each launch must move (inputs read once, outputs written once)."""
    L = w.max_cache
    units = w.units
    row = w.d * 2
    return {
        # scoring reads K once and the rows, writes the keep set; the fused
        # compaction reads the moved V rows and writes the moved K and V rows
        "score_select": units * (L * row + R * row + w.budget * 4) + 3 * row * rows_moved_per_launch,
        "fps": heads_total * (n_fps * row + w.fps_keep * (row + 1)),
        "append": heads_total * 2 * row,
        "rope": 0,
    }


def path_bytes(w, R: int, rows_moved_per_eviction: float, heads_total: int) -> float:
    """Bytes of one whole period, counting K once (the minimum the method needs):
    K read, observation rows read, kept written, moved rows (V read, K and V
    written), new beacons written, one query row per head and step."""
    row = w.d * 2
    units = w.units
    return (units * (w.max_cache * row + R * row + w.budget * 4) + 3 * row * rows_moved_per_eviction
            + heads_total * w.fps_keep * row + w.period * heads_total * 2 * row)


# ----------------------------------------------------------------------------- oracle legs

def _oracle_job(args):
    """One unit's eviction on the CPU oracle from a seeded steady state; returns seconds."""
    import numpy as np
    from oracle import UnitOracle
    (seed, G, d, theta, budget, prefix, recent, fps_cap, fps_keep, L, period) = args
    rng = np.random.default_rng(seed)

    def bf16(x):
        b = x.astype(np.float32).view(np.uint32)
        b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
        return b.astype(np.uint16)

    n_rq = fps_cap - fps_keep
    t = 4 * L + 1000
    uo = UnitOracle(G, d, theta, budget, prefix, recent, fps_cap, fps_keep)
    qs = lambda n: bf16(rng.standard_normal((n, d)) / math.sqrt(d))
    uo.load_state([qs(fps_keep) for _ in range(G)], [qs(min(period, n_rq)) for _ in range(G)],
                  list(range(t - min(period, n_rq) + 1, t + 1)),
                  bf16(rng.standard_normal((L, d))), bf16(rng.standard_normal((L, d))),
                  list(range(t - L + 1, t + 1)))
    t0 = time.perf_counter()
    uo.evict(t)
    return time.perf_counter() - t0


def oracle_pool():
    """A spawn-context process pool over every host core, one BLAS thread each."""
    import multiprocessing as mp
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    cores = len(os.sched_getaffinity(0))
    return mp.get_context("spawn").Pool(cores), cores


def oracle_rate(w, n_units: int, pool, cores: int, seed: int = 1234):
    """Evictions/s of the CPU oracle on n_units sampled units, all host cores."""
    jobs = [(seed + i, w.group, w.d, w.theta, w.budget, w.prefix, w.recent, w.fps_cap, w.fps_keep,
             w.max_cache, w.period) for i in range(n_units)]
    t0 = time.perf_counter()
    times = pool.map(_oracle_job, jobs, chunksize=1)
    wall = time.perf_counter() - t0
    return {"value": n_units / wall / w.kv_heads, "cores": cores, "wall_s": wall,
            "cpu_s": sum(times), "units": n_units}


def single_thread_rate(w, n_units: int, seed: int = 4321):
    """Evictions/s of the CPU oracle on one core (a one-process pool, one BLAS thread)."""
    import multiprocessing as mp
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    with mp.get_context("spawn").Pool(1) as pool:
        r = oracle_rate(w, n_units, pool, 1, seed=seed)
    # the per-unit eviction times alone (the worker's start-up and imports excluded)
    r["value"] = n_units / r["cpu_s"] / w.kv_heads
    return r


def cpu_model() -> str:
    """The host CPU's model name, from /proc/cpuinfo (x86 'model name', Arm implementer/part)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
    except OSError:
        return "unknown"
    fields = {}
    for line in info:
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    if "CPU implementer" in fields:
        return f"Arm implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    return "unknown"


def run_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    steps, warm = args.steps, args.warmup
    per_step = args.ref_units_per_step
    pool, cores = oracle_pool()
    with pool:
        for i in range(warm):
            oracle_rate(w, per_step, pool, cores, seed=10_000 * (i + 1))
        t0 = time.perf_counter()
        for i in range(steps):
            oracle_rate(w, per_step, pool, cores, seed=20_000 + 1000 * i)
        elapsed = time.perf_counter() - t0
    value = steps * per_step / w.kv_heads / elapsed
    out = {
        "impl": "reference", "metric": "KV evictions/s (all layers x batch)", "value": value,
        "unit": "evictions/s", "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": 1e3 * elapsed / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "layers": w.layers, "batch": w.batch, "heads": w.heads,
                   "kv_heads": w.kv_heads, "budget": w.budget, "period": w.period},
        "cpu_baseline": {"value": value, "unit": "evictions/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} steady-state units per step (one eviction = "
                                   f"{w.kv_heads} units), fp64 oracle, one unit per process"},
        "e2e": {"value": value, "unit": "evictions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU leg

def run_ours(args, w):
    import torch
    import torch.distributed as dist

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    from kv_cache_eviction_head_gb300.build import build
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
    from kv_cache_eviction_head_gb300 import bkv
    from synth import SyntheticStream

    stream = SyntheticStream(w, seed=0xBEAC0 + 2, device=dev)
    # one allocation per tensor for all layers; the library takes per-layer views
    K_all = torch.empty(w.layers, w.batch, w.kv_heads, w.max_cache, w.d, dtype=torch.bfloat16, device=dev)
    V_all = torch.empty_like(K_all)
    K, V = list(K_all.unbind(0)), list(V_all.unbind(0))
    for l in range(w.layers):
        stream.fill_cache(K[l], V[l], l, w.max_cache)
    kept = torch.empty(w.layers, w.batch, w.kv_heads, w.budget, dtype=torch.int32, device=dev)
    cfg = bkv.make_config(heads=w.heads, kv_heads=w.kv_heads, d=w.d, budget=w.budget,
                          period=w.period, prefix=w.prefix, recent=w.recent, fps_cap=w.fps_cap,
                          fps_keep=w.fps_keep, layers=w.layers, batch=w.batch,
                          max_cache=w.max_cache, rope_theta=w.theta,
                          flags=(bkv.BKV_FLAG_ORDER_FREE if args.order_free else 0)
                          | (bkv.BKV_FLAG_MEAN_POOL if args.pool == "mean" else 0))
    ws = torch.empty(bkv.bkv_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    cs = torch.cuda.current_stream(dev)
    h = bkv.bkv_create(cfg, ws, cs)
    import ctypes
    kptr = (ctypes.c_void_p * w.layers)(*[t.data_ptr() for t in K])
    vptr = (ctypes.c_void_p * w.layers)(*[t.data_ptr() for t in V])

    # fill the query state: one append per decode step until the cache is full
    for t in range(w.max_cache):
        bkv.bkv_append_queries(h, stream.queries(), t)
    # every period gets the stream's next queries (a repeated period would hand
    # FPS exact duplicates, which no decode stream produces)
    n_periods = args.warmup + args.steps
    qpool = torch.empty(n_periods, w.period, w.layers, w.batch, w.heads, w.d, dtype=torch.bfloat16,
                        device=dev)
    for p in range(n_periods):
        for i in range(w.period):
            qpool[p, i] = stream.queries()
    # and the keys and values its decode steps append at slots [budget, L)
    kvpool = torch.empty(n_periods, 2, w.layers, w.batch, w.kv_heads, w.period, w.d, dtype=torch.bfloat16,
                         device=dev)
    for p in range(n_periods):
        fresh_tail(stream, w, kvpool[p], w.max_cache + p * w.period)
    write_tail = TailWriter(w)
    bkv.bkv_sync(h)
    state = {"t": w.max_cache - 1, "p": 0}

    def step():
        t = state["t"]
        qper = qpool[state["p"] % n_periods]
        tail = kvpool[state["p"] % n_periods]
        bkv.bkv_evict_ptrs(h, kptr, vptr, w.max_cache, t, kept.data_ptr())
        # the period's decode steps write their keys and values into the freed slots
        write_tail(K_all, tail[0], cs)
        write_tail(V_all, tail[1], cs)
        for i in range(w.period):
            bkv.bkv_append_queries(h, qper[i], t + 1 + i)
        state["t"] = t + w.period
        state["p"] += 1

    for _ in range(args.warmup):
        step()
    bkv.bkv_sync(h)
    st0 = bkv.bkv_get_stats(h)
    heads_total = w.layers * w.batch * w.heads
    R = w.group * (st0.beacons + min(w.period, w.fps_cap - w.fps_keep))
    n_fps = st0.beacons + min(w.period, w.fps_cap - w.fps_keep)

    sampler = ClockSampler(local_rank)
    bkv.bkv_profile(h, True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(cs)
    for i in range(args.steps):
        step()
        evs[i + 1].record(cs)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    elapsed_ms = evs[0].elapsed_time(evs[-1])
    step_ms = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
    ktimes = bkv.bkv_profile_read(h)
    bkv.bkv_profile(h, False)
    bkv.bkv_sync(h)
    st1 = bkv.bkv_get_stats(h)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    evictions_per_step = w.evictions_per_round
    value = aggregate(evictions_per_step * args.steps, elapsed_ms / 1e3, world)

    # ---- per-kernel roofline from the events recorded during the timed steps
    peak, peak_kind = load_peaks()
    rows_moved = (st1.rows_moved - st0.rows_moved) / args.steps
    kb = kernel_bytes(w, R, rows_moved, heads_total, n_fps)
    kernels = {}
    for name, (ms, n) in ktimes.items():
        if n == 0:
            continue
        per = ms / n
        gbs = kb[name] / (per / 1e3) / 1e9 if kb[name] else None
        kernels[name] = {"ms_per_launch": per, "launches_per_step": n / args.steps,
                         "share": ms / sum(v[0] for v in ktimes.values()),
                         "alg_bytes_per_launch": kb[name],
                         "gbs": gbs, "frac": (gbs / peak) if gbs else None}
    dom = max(kernels, key=lambda k: kernels[k]["ms_per_launch"] * kernels[k]["launches_per_step"])
    traffic_key = w.name + ("+order-free" if args.order_free else "") + ("+mean" if args.pool == "mean" else "")
    traffic = read_traffic(dom, traffic_key)
    roofline = {"kernel": dom, "bound": "hbm", "achieved": kernels[dom]["gbs"], "peak": peak,
                "unit": "GB/s", "frac": kernels[dom]["frac"], "traffic": traffic,
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                else "fallback 6.8 TB/s"}
    pbytes = path_bytes(w, R, rows_moved, heads_total)

    # ---- future-query coverage of the observation sets (diagnostic, untimed step)
    coverage = None
    if args.coverage > 0:
        # the stream's next queries (the synthetic recipe), as the observation
        # sets would meet them
        qf = torch.stack([stream.queries() for _ in range(args.coverage)])
        cov = torch.empty(w.layers, w.batch, w.heads, args.coverage, dtype=torch.float64, device=dev)
        for _ in range(2):
            bkv.bkv_coverage(h, qf, cov)
        bkv.bkv_profile(h, True)
        ca, cb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ca.record(cs)
        for _ in range(3):
            bkv.bkv_coverage(h, qf, cov)
        cb.record(cs)
        torch.cuda.synchronize(dev)
        bkv.bkv_profile(h, False)
        ms = ca.elapsed_time(cb) / 3
        st = bkv.bkv_get_stats(h)
        pairs = heads_total * (st.beacons + st.recents) * args.coverage
        coverage = {"n_future": args.coverage, "obs_rows_per_head": st.beacons + st.recents,
                    "ms_per_launch": ms, "exact_cosines_per_s": pairs / (ms / 1e3)}

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        del qpool, kvpool
        e2e = run_e2e(args, w, bkv, h, K_all, V_all, kept, kptr, vptr, stream, state, dev, cs)
        e2e["elapsed_ms"] = max_over_ranks(e2e["elapsed_ms"], world, dev)
        e2e = {"value": aggregate(evictions_per_step * e2e["steps"], e2e["elapsed_ms"] / 1e3, world),
               "unit": "evictions/s", "h2d_bytes_per_step": e2e["h2d"],
               "d2h_bytes_per_step": e2e["d2h"], "steps": e2e["steps"], "h2d_warmup": e2e["h2d_warmup"]}

    bkv.bkv_destroy(h)

    # ---- prefill: initial beacons from a prompt of args.prefill queries (timed alone)
    prefill = None
    if args.prefill > 0:
        P = min(args.prefill, w.max_cache)
        # a prompt from a fresh stream of the same synthetic recipe
        pstream = SyntheticStream(w, seed=0xBEAC0 + 7, device=dev)
        qp = torch.empty(P, w.layers, w.batch, w.heads, w.d, dtype=torch.bfloat16, device=dev)
        for i in range(P):
            qp[i] = pstream.queries()
        ms = []
        for rep in range(4):
            ws2 = torch.empty(bkv.bkv_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
            h2 = bkv.bkv_create(cfg, ws2, cs)
            pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            pa.record(cs)
            bkv.bkv_prefill(h2, qp, 0)
            pb.record(cs)
            torch.cuda.synchronize(dev)
            bkv.bkv_sync(h2)
            bkv.bkv_destroy(h2)
            if rep > 0:
                ms.append(pa.elapsed_time(pb))
        N = P - min(w.fps_cap - w.fps_keep, P)
        prefill = {"prompt": P, "older_queries_per_head": N, "ms": statistics.median(ms),
                   "heads": heads_total, "candidates_per_s": heads_total * N / (statistics.median(ms) / 1e3)}
        del qp
    del K, V
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        pool, cores = oracle_pool()
        with pool:
            r = oracle_rate(w, args.cpu_units, pool, cores)
        single = single_thread_rate(w, max(8, args.cpu_units // 32))
        cpu = {"value": r["value"], "unit": "evictions/s", "cores": r["cores"], "kind": "oracle",
               "sample": f"{r['units']} steady-state units of {w.name} (one eviction = "
                         f"{w.kv_heads} units), fp64 oracle, one unit per process, "
                         f"{r['cpu_s']:.1f} s of CPU work in {r['wall_s']:.1f} s",
               "single_thread": {"value": single["value"], "unit": "evictions/s",
                                 "units": single["units"]},
               "cpu_model": cpu_model()}

    if rank == 0:
        out = {
            "metric": "KV evictions/s (all layers x batch)", "value": value, "unit": "evictions/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "us_per_eviction": 1e3 * elapsed_ms / args.steps / evictions_per_step,
            "step_ms": {"median": statistics.median(step_ms),
                        "p95": step_ms[min(len(step_ms) - 1, math.ceil(0.95 * len(step_ms)) - 1)]},
            "config": {"workload": w.name, "layers": w.layers, "batch": w.batch,
                       "heads": w.heads, "kv_heads": w.kv_heads, "d": w.d, "budget": w.budget,
                       "period": w.period, "prefix": w.prefix, "recent": w.recent,
                       "fps": f"{w.fps_cap}->{w.fps_keep}", "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (K/V cache %.1f GB)" % (
                           2 * w.layers * w.batch * w.kv_heads * w.max_cache * w.d * 2 / 1e9),
                       "step": f"1 eviction + {w.period} query appends + the period's fresh K/V rows "
                               f"written to slots [budget, L) (one 2-D device copy per tensor)",
                       "compaction": "order-free (holes filled from the kept tail)" if args.order_free
                       else "slot order (eq. 8)",
                       "pooling": args.pool},
            "gpu_launches": int(sum(n for _, n in ktimes.values())),
            "roofline": roofline,
            "path": {"alg_bytes_per_step": pbytes,
                     "gbs": pbytes / (elapsed_ms / args.steps / 1e3) / 1e9,
                     "frac": pbytes / (elapsed_ms / args.steps / 1e3) / 1e9 / peak,
                     "rows_moved_per_unit": rows_moved / w.units, "obs_rows_per_unit": R},
            "kernels": kernels,
            "clocks": clocks,
            "coverage": coverage,
            "prefill": prefill,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def fresh_tail(stream, w, out, pos0: int) -> None:
    """The synthetic stream's keys and values of positions pos0 .. pos0 +
    period - 1 (what a period's decode steps append to the cache), into
    out [2][layers][batch][kv_heads][period][d] (keys, then values)."""
    for i in range(w.period):
        k, v = stream.keys_values(pos0 + i)
        out[0, :, :, :, i] = k
        out[1, :, :, :, i] = v


class TailWriter:
    """Writes a period's new keys and values into cache slots [budget, L) of
    every (layer, sequence, KV head): one 2-D device copy per tensor
    (cudaMemcpy2DAsync: layers x batch x kv_heads rows of period x d values,
    source rows packed, destination rows max_cache x d apart), which moves
    the rows at about 2 TB/s where a strided tensor copy reached 1.3 TB/s.
    Falls back to the tensor copy when no CUDA runtime library can be loaded."""

    def __init__(self, w):
        import ctypes
        self.w = w
        self.rt = None
        for name in ("libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
            try:
                rt = ctypes.CDLL(name)
                rt.cudaMemcpy2DAsync.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                                 ctypes.c_size_t, ctypes.c_size_t, ctypes.c_size_t,
                                                 ctypes.c_int, ctypes.c_void_p]
                self.rt = rt
                break
            except OSError:
                continue

    def __call__(self, dst_all, src, stream) -> None:
        """dst_all: [layers][batch][kv_heads][max_cache][d]; src: its period's
        rows [layers][batch][kv_heads][period][d], contiguous; on `stream`."""
        import ctypes
        w = self.w
        if self.rt is None:
            dst_all[:, :, :, w.budget:w.max_cache].copy_(src)
            return
        row = w.d * 2
        err = self.rt.cudaMemcpy2DAsync(ctypes.c_void_p(dst_all.data_ptr() + w.budget * row), w.max_cache * row,
                                        ctypes.c_void_p(src.data_ptr()), w.period * row, w.period * row,
                                        w.layers * w.batch * w.kv_heads, 3, ctypes.c_void_p(stream.cuda_stream))
        if err != 0:
            raise RuntimeError(f"cudaMemcpy2DAsync failed ({err})")


def e2e_plan(period_bytes: int, warmup: int, steps: int, host_cap_bytes: int):
    """(warm-up, timed) steps of the e2e run: one host period of queries per
    step, at least one warm-up step, and no more periods than host_cap_bytes
    holds (then one warm-up and the rest timed, at least one)."""
    warm, timed = max(1, warmup), steps
    fit = max(2, host_cap_bytes // period_bytes)
    if warm + timed > fit:
        warm, timed = 1, fit - 1
    return warm, timed


def run_e2e(args, w, bkv, h, K_all, V_all, kept, kptr, vptr, stream, state, dev, cs,
            host_cap_bytes=48 << 30, nbuf=2, copy_events=None, warm_link=True):
    """Same step through the C ABI, with each step's inputs coming from pinned
    host memory (the period's queries and the new K/V rows) and the keep sets
    going back to the host, all inside the timed region. The copies run on a
    second stream into nbuf staging buffers (default two), so that the next
    steps' inputs travel while step k's eviction runs: inputs land in device
    staging buffers, and the new K/V rows move into the cache (a device copy)
    once the eviction that reads those slots is done. copy_events, when a
    list, receives per step the (start, end) timing events of its input copy.

    Every step gets a period of fresh queries and fresh keys and values from
    the stream (a repeated period would hand FPS exact duplicates and the
    scoring the same rows again), generated before the timed region straight
    into pinned host memory. The pool is capped at host_cap_bytes; a workload
    whose periods do not fit runs fewer e2e steps (one warm-up and at least
    one timed), and the returned step count says so."""
    import torch
    q_bytes = w.period * w.layers * w.batch * w.heads * w.d * 2
    kv_bytes = w.layers * 2 * w.batch * w.kv_heads * w.period * w.d * 2
    warm, steps = e2e_plan(q_bytes + kv_bytes, args.warmup, args.steps, host_cap_bytes)
    total = warm + steps
    q_host = torch.empty(total, w.period, w.layers, w.batch, w.heads, w.d, dtype=torch.bfloat16,
                         pin_memory=True)
    for p in range(total):
        for i in range(w.period):
            q_host[p, i].copy_(stream.queries())
    # the new K/V rows of each period, host side
    tail_host = torch.empty(total, 2, w.layers, w.batch, w.kv_heads, w.period, w.d, dtype=torch.bfloat16,
                            pin_memory=True)
    tmp = torch.empty(tail_host.shape[1:], dtype=torch.bfloat16, device=dev)
    for p in range(total):
        fresh_tail(stream, w, tmp, state["t"] + 1 + p * w.period)
        tail_host[p].copy_(tmp)
    del tmp
    write_tail = TailWriter(w)
    xs = torch.cuda.Stream(dev)
    qstage = [torch.empty(q_host.shape[1:], dtype=q_host.dtype, device=dev) for _ in range(nbuf)]
    link = warm_h2d(q_host[0], qstage[0], xs) if warm_link else None
    tstage = [torch.empty(tail_host.shape[1:], dtype=tail_host.dtype, device=dev) for _ in range(nbuf)]
    kept_dev = [kept] + [torch.empty_like(kept) for _ in range(nbuf - 1)]
    kept_host = [torch.empty(kept.shape, dtype=kept.dtype).pin_memory() for _ in range(nbuf)]
    ev = {name: [torch.cuda.Event() for _ in range(nbuf)] for name in ("staged", "used", "evicted", "read")}

    def stage(k):
        """Copy stream: step k's queries and new K/V rows into staging buffer k % nbuf."""
        b = k % nbuf
        with torch.cuda.stream(xs):
            if k >= nbuf:
                xs.wait_event(ev["used"][b])  # step k - nbuf is done with this buffer
            if copy_events is not None:
                ce = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ce[0].record(xs)
            qstage[b].copy_(q_host[k], non_blocking=True)
            tstage[b].copy_(tail_host[k], non_blocking=True)
            if copy_events is not None:
                ce[1].record(xs)
                copy_events.append(ce)
            ev["staged"][b].record(xs)

    def step(k):
        b = k % nbuf
        t = state["t"]
        if k >= nbuf:
            cs.wait_event(ev["read"][b])  # step k - nbuf's keep sets have reached the host
        bkv.bkv_evict_ptrs(h, kptr, vptr, w.max_cache, t, kept_dev[b].data_ptr())
        ev["evicted"][b].record(cs)
        with torch.cuda.stream(xs):
            xs.wait_event(ev["evicted"][b])
            kept_host[b].copy_(kept_dev[b], non_blocking=True)
            ev["read"][b].record(xs)
        cs.wait_event(ev["staged"][b])
        write_tail(K_all, tstage[b][0], cs)
        write_tail(V_all, tstage[b][1], cs)
        for i in range(w.period):
            bkv.bkv_append_queries(h, qstage[b][i], t + 1 + i)
        ev["used"][b].record(cs)
        state["t"] = t + w.period

    for k in range(min(nbuf, total)):
        stage(k)
    for k in range(warm):
        step(k)
        if k + nbuf < total:
            stage(k + nbuf)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cs)
    for k in range(warm, total):
        step(k)
        if k + nbuf < total:
            stage(k + nbuf)
    cs.wait_event(ev["read"][(total - 1) % nbuf])  # the last keep sets are on the host
    e1.record(cs)
    torch.cuda.synchronize(dev)
    bkv.bkv_sync(h)
    return {"elapsed_ms": e0.elapsed_time(e1), "steps": steps,
            "h2d": qstage[0].numel() * 2 + tstage[0].numel() * 2, "d2h": kept_host[0].numel() * 4,
            "h2d_warmup": link}


def warm_h2d(src, dst, xs, min_gbs=100.0, need=3, max_copies=40):
    """Untimed warm-up of the host-to-device path before the e2e region.
    Without it, on the GB300 machines, the first six to nine staged copies of a
    run (about half a second) took 45-135 ms for 1.36 GB (10-30 GB/s) before
    settling at 6-10 ms, whatever buffer was copied, and the e2e rate ranged
    from 165K to 260K evictions/s; with it (3-4 copies of one step's queries
    at ~210 GB/s) four runs gave 263K-272K. Repeats the copy until `need`
    copies in a row reach min_gbs (at most max_copies); returns the copies
    made and the last rate."""
    import torch
    nbytes = src.numel() * src.element_size()
    run, gbs, n = 0, 0.0, 0
    while n < max_copies and run < need:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(xs):
            a.record(xs)
            dst.copy_(src, non_blocking=True)
            b.record(xs)
        b.synchronize()
        gbs = nbytes / (a.elapsed_time(b) / 1e3) / 1e9
        run = run + 1 if gbs >= min_gbs else 0
        n += 1
    return {"copies": n, "last_gbs": gbs}


def kernel_source_digest(kernel: str):
    """SHA-256 prefix of a kernel's source file followed by every csrc/*.cuh
    (sorted): any change to the kernel or a header it may include changes it."""
    import glob
    import hashlib
    src = {"score_select": "k_score.cu", "fps": "k_fps.cu",
           "append": "k_append.cu", "rope": "k_append.cu"}.get(kernel)
    if not src:
        return None
    csrc = os.path.join(ROOT, "kv_cache_eviction_head_gb300", "csrc")
    h = hashlib.sha256()
    for p in [os.path.join(csrc, src)] + sorted(glob.glob(os.path.join(csrc, "*.cuh"))):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the
    current kernel source (profiles/traffic.md lists the source digest)."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    digest = kernel_source_digest(kernel)
    if not digest or not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cells) >= 4 and cells[0] == kernel and cells[1] == workload and cells[2] == digest:
                try:
                    return float(cells[3])
                except ValueError:
                    return None
    return None


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_4b_b192")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (smaller cases for profiling)")
    ap.add_argument("--cpu-units", type=int, default=1024)
    ap.add_argument("--ref-units-per-step", type=int, default=32)
    ap.add_argument("--order-free", action="store_true",
                    help="order-free compaction (BKV_FLAG_ORDER_FREE) instead of slot order")
    ap.add_argument("--budget", type=int, default=None, help="override the workload's budget")
    ap.add_argument("--pool", choices=["max", "mean"], default="max",
                    help="aggregation of the attention weights over observation rows")
    ap.add_argument("--fps-keep", type=int, default=None,
                    help="beacons kept per head (recent queries = 32 - this), Table 1's splits")
    ap.add_argument("--prefill", type=int, default=0,
                    help="also time bkv_prefill over a prompt of this many steps (fresh state)")
    ap.add_argument("--coverage", type=int, default=0,
                    help="also time bkv_coverage over this many future queries (diagnostic)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    from synth import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(batch=args.batch, name=f"{w.name}_batch{args.batch}")
    if args.fps_keep is not None:
        w = w.with_(fps_keep=args.fps_keep, name=f"{w.name}_keep{args.fps_keep}")
    if args.budget is not None:
        w = w.with_(budget=args.budget, name=f"{w.name}_budget{args.budget}")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
