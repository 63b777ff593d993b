#!/usr/bin/env python3
"""Decode-attention throughput of the KV4 hot path (libkv4) on GB300.

One step = one kv4_decode_attention call (plan + split-K attention + merge)
over the whole batch of the workload, with the paged INT4 cache and INT8 side
buffers already filled by one prefill kv4_append. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kv4|reference]
                  [--workload qwen3-8b|qwen3-4b|long-tail]

--impl reference times the CPU oracle (the method's plain definition) on the
host cores on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs its own batch (weak scaling, no collective
in the data path); the timing barrier and the max-over-ranks use torch.distributed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from int8_hybrid_paged_gb300 import bytes_model, inputs  # noqa: E402

METRIC = "decode-attn context tokens/s and achieved HBM GB/s (% GB300 peak), 1 GPU"
UNIT = "context tokens/s"
DTYPE = "s8 x u4/u8 -> s32 dots, fp32 softmax/accumulate"
L2_BYTES = 129 * 2 ** 20
LONG_TAIL_POOL_BYTES = 120 * 10 ** 9     # page budget of the 36-layer long-tail stack
ORACLE_SAMPLE_SEQS = 16                  # sequences of the CPU oracle's timed sample
SPLIT_SOURCES = ["int8_hybrid_paged_gb300/csrc/decode.cu",
                 "int8_hybrid_paged_gb300/csrc/device_common.cuh",
                 "int8_hybrid_paged_gb300/csrc/kv4_internal.h"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["kv4", "reference"], default="kv4")
    ap.add_argument("--workload", default="qwen3-8b", choices=["qwen3-8b", "qwen3-4b", "long-tail"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work of the oracle baseline sample")
    ap.add_argument("--sink", type=int, default=None,
                    help="override the sink size s (with --window 0 and --sink 0: unprotected KV4)")
    ap.add_argument("--window", type=int, default=None, help="override the recent window w")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-full", action="store_true",
                    help="time the CPU oracle once over the whole workload (no GPU) and exit")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-append", action="store_true", help="skip the append-stress measurement")
    ap.add_argument("--format", choices=["int4-hybrid", "int8", "nvfp4", "mxfp4"], default="int4-hybrid",
                    help="cache format of the main measurement: the method (INT4 pages + INT8 "
                         "side buffer), the whole-cache 8-bit format (KV8, s = w = 0) or the "
                         "whole-cache NVFP4 / MXFP4 formats (s = w = 0)")
    ap.add_argument("--no-qkv", action="store_true",
                    help="skip the fused projection + append measurement")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the unprotected KV4 (s = w = 0), whole-cache 8-bit and NVFP4 measurements")
    return ap.parse_args()


# --------------------------------------------------------------------------- environment

def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (torch.cuda.is_available() and args.impl == "kv4") else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max_sum(world, t_max, v_sum, device):
    if world == 1:
        return t_max, v_sum
    import torch.distributed as dist
    a = torch.tensor([t_max], dtype=torch.float64, device=device)
    b = torch.tensor([v_sum], dtype=torch.float64, device=device)
    dist.all_reduce(a, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(a.item()), float(b.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.25)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


def split_kernel_traffic():
    """dram bytes per launch of the split kernel from the committed ncu summary, if the
    kernel sources are unchanged since it was taken."""
    p = os.path.join(ROOT, "profiles", "decode_split_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    h = hashlib.sha256()
    for f in SPLIT_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if d.get("source_sha256") != h.hexdigest():
        return None
    return d


# --------------------------------------------------------------------------- workload

def workload_from_args(args):
    """The named workload, with the protected region overridden if asked (the 8-bit
    format has none)."""
    import dataclasses
    wl = inputs.workload(args.workload)
    fmt = getattr(args, "format", "int4-hybrid")
    if fmt in ("int8", "nvfp4", "mxfp4"):
        what = {"int8": "8-bit", "nvfp4": "NVFP4", "mxfp4": "MXFP4"}[fmt]
        return dataclasses.replace(wl, sink=0, window=0,
                                   name=wl.name + f" (whole-cache {what} format)")
    if args.sink is not None or args.window is not None:
        s = wl.sink if args.sink is None else args.sink
        w = wl.window if args.window is None else args.window
        wl = dataclasses.replace(wl, sink=s, window=w,
                                 name=wl.name + f" (protected region overridden: s={s}, w={w})")
    return wl


def pool_pages_for(wl):
    """Physical pages of a workload's pool: its sequences' pages plus 1 % spare, or, for
    the long-tail stack, the share of a 120 GB page budget that one of its layers gets
    (pages scattered over the whole budget)."""
    need = sum((L + 15) // 16 for L in wl.context_lens)
    if wl.layers > 1:
        budget = LONG_TAIL_POOL_BYTES // wl.layers
        return max(need + 64, budget // (wl.num_kv_heads * 2176))
    return need + max(64, need // 100)


def build_workload(wl, seed, device, sample_seqs=0, fmt=0):
    """Fill a cache with the workload's sequences (one prefill append). Host copies
    (bf16 bits) of the first `sample_seqs` sequences' K/V are kept for the CPU
    baseline; the device K/V are freed once appended."""
    from int8_hybrid_paged_gb300.kv4 import KV4Cache

    lens = list(wl.context_lens)
    B, H, Hq = wl.batch, wl.num_kv_heads, wl.num_q_heads
    num_pages = pool_pages_for(wl)
    bt = inputs.block_tables(lens, 16, num_pages, seed)
    cache = KV4Cache(H, num_pages, max_slots=B, max_batch=B, max_q_heads=Hq, sink=wl.sink,
                     window=wl.window, fmt=fmt)
    total = sum(lens)
    k, v = inputs.kv_tokens(total, H, seed * 1_000_003 + 17, device=device)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    slots = torch.arange(B, dtype=torch.int32, device=device)
    bt_dev = torch.from_numpy(bt).to(device)
    cache.append(k, v, torch.from_numpy(cu).to(device), slots,
                 torch.zeros(B, dtype=torch.int32, device=device), bt_dev)
    host_kv = [(inputs.bf16_bits(k[cu[b]:cu[b + 1]]), inputs.bf16_bits(v[cu[b]:cu[b + 1]]))
               for b in range(min(sample_seqs, B))]
    del k, v
    q = inputs.queries(B, Hq, seed, device=device)
    cl = torch.tensor(lens, dtype=torch.int32, device=device)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    err = cache.device_error()
    if err:
        raise RuntimeError(f"device error {err} while filling the cache")
    return dict(cache=cache, host_kv=host_kv, cu=cu, bt=bt, bt_dev=bt_dev, q=q, cl=cl,
                slots=slots, lens=lens, num_pages=num_pages)


def oracle_sample(wl, st, cpu_seconds, threads, kv8=False, nvfp4=False, mxfp4=False):
    """Time the CPU oracle's decode over a bounded sample of the workload (its first
    sequences, the same inputs as the GPU run): with OpenMP over (sequence, q head) on
    the host cores, and with one thread. Returns the cpu_baseline dict."""
    import oracle

    lens = st["lens"]
    pick = list(range(len(st["host_kv"])))
    H, G = wl.num_kv_heads, wl.group
    maxL = max(lens[b] for b in pick)
    oc = oracle.OracleCache(H, wl.sink, wl.window, maxL, num_slots=len(pick), kv8=kv8,
                            nvfp4=nvfp4, mxfp4=mxfp4)
    for i, b in enumerate(pick):
        oc.append(i, 0, st["host_kv"][b][0], st["host_kv"][b][1])
    qb = inputs.bf16_bits(st["q"][pick])
    slots = np.arange(len(pick), dtype=np.int32)
    sl = np.array([lens[b] for b in pick], np.int32)
    used = min(threads, len(pick) * wl.num_q_heads)

    def timed(nthreads, seconds):
        reps, t0 = 0, time.perf_counter()
        while True:
            oc.decode_batch(slots, sl, G, qb, 1 / math.sqrt(128), threads=nthreads)
            reps += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return float(sl.sum()) * reps / el, reps, el

    v_all, reps, el = timed(used, cpu_seconds)
    v_one, reps1, el1 = timed(1, cpu_seconds / 2)
    return {"value": v_all, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"first {len(pick)} of {len(lens)} sequences ({int(sl.sum())} context "
                      f"tokens, {wl.num_q_heads} q heads) x {reps} repetitions in {el:.1f} s, "
                      f"OpenMP over (sequence, q head); host CPU: {cpu_model()}",
            "one_thread": {"value": v_one, "unit": UNIT, "cores": 1,
                           "sample": f"the same sample x {reps1} repetitions in {el1:.1f} s"}}


def call_bytes_for(wl, fmt):
    """Algorithmic bytes of one decode call over the workload's batch (with the LSE)."""
    lens, Hq, H = list(wl.context_lens), wl.num_q_heads, wl.num_kv_heads
    if fmt == "int8":
        return bytes_model.decode_call_bytes_kv8(lens, Hq, H, with_lse=True)
    if fmt == "nvfp4":
        return bytes_model.decode_call_bytes_nvfp4(lens, Hq, H, with_lse=True)
    if fmt == "mxfp4":
        return bytes_model.decode_call_bytes_nvfp4(lens, Hq, H, with_lse=True,
                                                   per_position=bytes_model.MXFP4_POSITION_HEAD_BYTES)
    return bytes_model.decode_call_bytes(lens, Hq, H, wl.sink, wl.window, with_lse=True)


def workload_config(wl, world, call_bytes, pool_pages, copies=1):
    """The config object of a bench line (both arms print the same one)."""
    per_cycle = call_bytes * copies * wl.layers
    if copies > 1:
        l2 = (f"{copies} distinct cache copies cycled: {per_cycle / 1e9:.2f} GB read per cycle vs "
              f"{L2_BYTES / 2**20:.0f} MiB L2, no flush")
    else:
        l2 = (f"inputs larger than L2: {call_bytes / 1e9:.2f} GB read per call vs "
              f"{L2_BYTES / 2**20:.0f} MiB L2, no flush")
    return {"workload": wl.name, "batch": wl.batch, "q_heads": wl.num_q_heads,
            "kv_heads": wl.num_kv_heads, "head_dim": 128, "page_size": 16, "sink": wl.sink,
            "window": wl.window, "layers": wl.layers,
            "context_tokens_per_step": int(sum(wl.context_lens)) * wl.layers * copies,
            "max_context": max(wl.context_lens), "pool_pages": pool_pages, "l2": l2,
            "parallelism": f"replicas x{world} (independent batches)"}


# --------------------------------------------------------------------------- arms

def run_kv4(args, rank, world, local):
    from int8_hybrid_paged_gb300 import build as kbuild
    from int8_hybrid_paged_gb300 import kv4

    kbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workload_from_args(args)
    kv8, fp4, mx = args.format == "int8", args.format == "nvfp4", args.format == "mxfp4"
    seed = wl.seed + rank
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    st = build_workload(wl, seed, dev, sample_seqs=ORACLE_SAMPLE_SEQS if want_cpu else 0,
                        fmt=(kv4.FORMAT_INT8 if kv8 else kv4.FORMAT_NVFP4 if fp4
                             else kv4.FORMAT_MXFP4 if mx else kv4.FORMAT_INT4_HYBRID))
    cache = st["cache"]
    B, Hq, H = wl.batch, wl.num_q_heads, wl.num_kv_heads
    lens = st["lens"]
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    layers = wl.layers

    def step():
        for _ in range(layers):
            kv4.kv4_decode_attention(cache.handle, st["q"], st["slots"], st["cl"], st["bt_dev"],
                                     out, lse, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if cache.device_error():
        raise RuntimeError("device error during warm-up")

    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms = e0.elapsed_time(e1)
    if cache.device_error():
        raise RuntimeError("device error during the timed region")

    # per-kernel times: a separate pass with the library's events between the three
    # launches (each kernel then runs alone, so the events time it)
    prof_steps = min(args.steps, 500)
    kv4.kv4_profile_start(cache.handle, prof_steps * layers)
    for _ in range(prof_steps):
        step()
    torch.cuda.synchronize()
    prof = kv4.kv4_profile_stop(cache.handle)

    tokens_step = float(sum(lens)) * layers
    t_max, tok_sum = reduce_max_sum(world, ms, tokens_step * args.steps, dev)
    value = tok_sum / (t_max * 1e-3)

    call_bytes = call_bytes_for(wl, args.format)
    # the split kernel reads 144-byte query records (written by the prep kernel) instead
    # of the bf16 queries; the outputs are written by the merge
    split_bytes = call_bytes - B * Hq * (128 * 4 + 4) - B * Hq * (128 * 2 - 144)
    split_ms = prof["split_ms"] / max(1, prof["calls"])
    peak, peak_src = measured_peaks()
    achieved = split_bytes / (split_ms * 1e-3) / 1e9
    traffic = None if (kv8 or fp4 or mx) else split_kernel_traffic()
    step_gbs = call_bytes * layers / (ms / args.steps * 1e-3) / 1e9

    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic (seeded bf16 N(0,1) K/V/q, 4 K outlier channels x20, lognormal lengths)",
        "config": workload_config(wl, world, call_bytes, st["num_pages"]),
        "achieved_hbm_gbs": step_gbs,
        "pct_hbm_peak": 100.0 * step_gbs / peak,
        "roofline": {"bound": "hbm", "kernel": "kv4_decode_split_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": split_bytes,
                     "avg_launch_ms": split_ms,
                     "traffic": (traffic["dram_bytes_per_launch"] if traffic else None),
                     "plan_ms": prof["plan_ms"] / max(1, prof["calls"]),
                     "merge_ms": prof["merge_ms"] / max(1, prof["calls"]),
                     "kernel_timing": f"separate {prof_steps}-step pass with CUDA events "
                                      "between the three launches of each call"},
        "gpu_launches": 3 * args.steps * layers,
        "clocks": clk,
    }

    # ---- append stress (the quantize + pack + side-write path), only on rank 0 at N = 1
    if world == 1 and not args.no_append:
        res["append_stress"] = run_append_stress(dev, peak)

    # ---- the attention input projection with the append fused into its epilogue
    hybrid = not (kv8 or fp4 or mx)
    if world == 1 and not args.no_qkv and hybrid:
        res["qkv_append"] = run_qkv_append(dev)

    # ---- the other workloads of the method's configuration, rank 0 at N = 1
    if world == 1 and not args.no_variants and hybrid and args.workload == "qwen3-8b":
        res["qwen3_4b"] = run_cache_set("qwen3-4b", dev, peak, min(args.steps, 200))
        res["long_tail"] = run_cache_set("long-tail", dev, peak, min(args.steps, 50))

    # ---- the same workload without the protected region (pure KV4), rank 0 at N = 1
    if world == 1 and not args.no_variants and hybrid and (wl.sink > 0 or wl.window > 0):
        res["kv4_unprotected"] = run_unprotected(wl, seed, dev, peak, value, min(args.steps, 500))
    if world == 1 and not args.no_variants and hybrid:
        res["kv8"] = run_whole_cache(wl, seed, dev, peak, value, min(args.steps, 500), "int8")
        res["nvfp4"] = run_whole_cache(wl, seed, dev, peak, value, min(args.steps, 500), "nvfp4")
        res["mxfp4"] = run_whole_cache(wl, seed, dev, peak, value, min(args.steps, 500), "mxfp4")

    # ---- end to end through the public API from pinned host buffers
    if not args.no_e2e:
        res["e2e"] = run_e2e(st, wl, args, dev, world)

    # ---- CPU oracle baseline (rank 0, one GPU)
    if want_cpu:
        res["cpu_baseline"] = oracle_sample(wl, st, args.cpu_seconds, host_cores(), kv8, fp4, mx)
    cache.close()
    if rank == 0:
        print(json.dumps(res), flush=True)


def time_calls(step, cache, steps, layers):
    """Mean ms per step over `steps` timed steps (CUDA events on the stream, no
    per-kernel events inside), then the per-kernel times from a second pass with the
    library's events between the launches."""
    from int8_hybrid_paged_gb300 import kv4

    stream = torch.cuda.current_stream()
    for _ in range(20):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    kv4.kv4_profile_start(cache.handle, steps * layers)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    return ms, kv4.kv4_profile_stop(cache.handle)


def run_cache_set(name, dev, peak, steps):
    """A workload over several caches at once, each step one decode call per cache:
    the Qwen3-4B-shaped layer in 4 distinct copies cycled (one copy, about 0.13 GB per
    call, is about the L2's size), or the long-tail stack of 36 layers (each its own
    cache, pages scattered over a 120 GB page budget) with the 36 calls of a step
    captured in one CUDA graph. Context tokens/s over the whole step, and the split
    kernel's HBM rate from a second pass with events between the launches."""
    from int8_hybrid_paged_gb300 import kv4

    base = inputs.workload(name)
    copies = 4 if base.layers == 1 else base.layers
    B, Hq = base.batch, base.num_q_heads
    sts = []
    try:
        for i in range(copies):
            sts.append(build_workload(base, base.seed + 101 * (i + 1), dev))
        out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)

        def step():
            stream = torch.cuda.current_stream(dev)     # the capture stream inside the graph
            for st in sts:
                kv4.kv4_decode_attention(st["cache"].handle, st["q"], st["slots"], st["cl"],
                                         st["bt_dev"], out, lse, stream=stream)

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        del graph
        ms = e0.elapsed_time(e1) / steps
        # per-kernel times: eager calls with the library's events between the launches
        for st in sts:
            kv4.kv4_profile_start(st["cache"].handle, steps)
        for _ in range(steps):
            step()
        torch.cuda.synchronize()
        profs = [kv4.kv4_profile_stop(st["cache"].handle) for st in sts]
        if any(st["cache"].device_error() for st in sts):
            raise RuntimeError(f"device error in the {name} measurement")
        call_bytes = call_bytes_for(base, "int4-hybrid")
        split_bytes = call_bytes - B * Hq * (128 * 4 + 4) - B * Hq * (128 * 2 - 144)
        split_ms = sum(p["split_ms"] for p in profs) / max(1, sum(p["calls"] for p in profs))
        gbs = split_bytes / (split_ms * 1e-3) / 1e9
        tokens = float(sum(base.context_lens)) * copies
        return {"case": base.name + (f", {copies} distinct cache copies cycled" if base.layers == 1 else
                                     f", {copies} layer caches, one CUDA graph of {3 * copies} launches"
                                     " per step"),
                "value": tokens / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": steps,
                "config": workload_config(base, 1, call_bytes, sts[0]["num_pages"],
                                          copies=copies if base.layers == 1 else 1),
                "step_gbs": call_bytes * copies / (ms * 1e-3) / 1e9,
                "step_frac_of_hbm_peak": call_bytes * copies / (ms * 1e-3) / 1e9 / peak,
                "split_us": split_ms * 1e3, "split_algorithmic_bytes": split_bytes,
                "split_achieved_gbs": gbs, "split_frac_of_hbm_peak": gbs / peak}
    finally:
        for st in sts:
            st["cache"].close()
        sts.clear()
        torch.cuda.empty_cache()


def run_unprotected(wl, seed, dev, peak, protected_value, steps):
    """The same sequences, KV and queries with s = w = 0 (every position in the INT4
    pages, no side cache): context tokens/s of the whole decode call, the split
    kernel's HBM rate, and the share of it the protected configuration keeps."""
    import dataclasses
    from int8_hybrid_paged_gb300 import kv4

    wl0 = dataclasses.replace(wl, sink=0, window=0)
    st = build_workload(wl0, seed, dev)
    cache = st["cache"]
    B, Hq = wl0.batch, wl0.num_q_heads
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    try:
        def step():
            for _ in range(wl0.layers):
                kv4.kv4_decode_attention(cache.handle, st["q"], st["slots"], st["cl"],
                                         st["bt_dev"], out, lse, stream=stream)
        ms, prof = time_calls(step, cache, steps, wl0.layers)
        if cache.device_error():
            raise RuntimeError("device error in the unprotected decode")
        value = float(sum(st["lens"])) * wl0.layers / (ms * 1e-3)
        call_bytes = bytes_model.decode_call_bytes(st["lens"], Hq, wl0.num_kv_heads, 0, 0,
                                                   with_lse=True)
        split_bytes = call_bytes - B * Hq * (128 * 4 + 4) - B * Hq * (128 * 2 - 144)
        split_ms = prof["split_ms"] / max(1, prof["calls"])
        gbs = split_bytes / (split_ms * 1e-3) / 1e9
        return {"case": "the same workload with s = w = 0 (no INT8 side cache)",
                "value": value, "unit": UNIT, "ms_per_step": ms, "steps": steps,
                "split_us": split_ms * 1e3, "split_algorithmic_bytes": split_bytes,
                "split_achieved_gbs": gbs, "split_frac_of_hbm_peak": gbs / peak,
                "protected_retains": protected_value / value}
    finally:
        cache.close()
        torch.cuda.empty_cache()


def run_whole_cache(wl, seed, dev, peak, kv4_value, steps, fmt_name):
    """The same sequences, KV and queries in a whole-cache format with no protected
    region: the 8-bit format (every position's 8-bit codes in its page, the protected
    path's arithmetic) or NVFP4 (E2M1 codes, E4M3 block scales). Context tokens/s of the
    whole decode call and the split kernel's HBM rate."""
    import dataclasses
    from int8_hybrid_paged_gb300 import kv4

    kv8, mx = fmt_name == "int8", fmt_name == "mxfp4"
    wlw = dataclasses.replace(wl, sink=0, window=0)
    st = build_workload(wlw, seed, dev, fmt=(kv4.FORMAT_INT8 if kv8 else kv4.FORMAT_MXFP4 if mx
                                             else kv4.FORMAT_NVFP4))
    cache = st["cache"]
    B, Hq = wlw.batch, wlw.num_q_heads
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    try:
        def step():
            for _ in range(wlw.layers):
                kv4.kv4_decode_attention(cache.handle, st["q"], st["slots"], st["cl"],
                                         st["bt_dev"], out, lse, stream=stream)
        ms, prof = time_calls(step, cache, steps, wlw.layers)
        if cache.device_error():
            raise RuntimeError(f"device error in the {fmt_name} decode")
        value = float(sum(st["lens"])) * wlw.layers / (ms * 1e-3)
        if kv8:
            call_bytes = bytes_model.decode_call_bytes_kv8(st["lens"], Hq, wlw.num_kv_heads, with_lse=True)
        else:
            call_bytes = bytes_model.decode_call_bytes_nvfp4(
                st["lens"], Hq, wlw.num_kv_heads, with_lse=True,
                per_position=(bytes_model.MXFP4_POSITION_HEAD_BYTES if mx
                              else bytes_model.NVFP4_POSITION_HEAD_BYTES))
        split_bytes = call_bytes - B * Hq * (128 * 4 + 4) - B * Hq * (128 * 2 - 144)
        split_ms = prof["split_ms"] / max(1, prof["calls"])
        gbs = split_bytes / (split_ms * 1e-3) / 1e9
        what = ("whole-cache 8-bit format (KV8: 264 B per token-head)" if kv8 else
                "whole-cache MXFP4 format (E2M1 + E8M0 scales per 32: 136 B per token-head)" if mx else
                "whole-cache NVFP4 format (E2M1 + E4M3 block scales: 152 B per token-head)")
        return {"case": "the same workload, " + what,
                "value": value, "unit": UNIT, "ms_per_step": ms, "steps": steps,
                "split_us": split_ms * 1e3, "split_algorithmic_bytes": split_bytes,
                "split_achieved_gbs": gbs, "split_frac_of_hbm_peak": gbs / peak,
                "kv4_speedup": kv4_value / value}
    finally:
        cache.close()
        torch.cuda.empty_cache()


def run_qkv_append(dev):
    """kv4_qkv_append (the QKV projection on the tcgen05 tensor cores with RoPE, the
    Hadamard rotation and the 4-bit append fused into its epilogue) against the same
    work in two steps (kv4_linear_bf16, then kv4_append), on Qwen3-8B attention shapes
    (d_model 4096, 32 q heads, 8 KV heads): decode steps of 256 and of 128 single tokens
    (the second on the split-K cluster path) and a re-prefill chunk of 8 x 2048 tokens. The two-step path also gathers the K and V
    columns into [T][H][128] tensors for the append. Device time per call from one
    replay of a CUDA graph of repeated calls, each on the next of four weight copies;
    seeded random bf16 weights and hidden states."""
    from int8_hybrid_paged_gb300 import kv4
    from int8_hybrid_paged_gb300.kv4 import KV4Cache
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak_tf = float(peaks.get("bf16_tflops", 1900.0))
    peak_hbm = float(peaks.get("hbm_gbs", 6800.0))
    H, Hq, d = 8, 32, 4096
    N = (Hq + 2 * H) * 128
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    # four copies of W_qkv (4 x 50 MB, above the 129 MB L2), one per call in turn: no
    # call finds its weights in L2
    ws = [(torch.randn((N, d), generator=g, device=dev) / d ** 0.5).to(torch.bfloat16) for _ in range(4)]
    out = {}
    for tag, B, T, start_pos, reps in (("decode", 256, 1, 600, 50), ("decode_b128", 128, 1, 600, 50),
                                       ("prefill", 8, 2048, 0, 10)):
        stride = (start_pos + T + 15) // 16 + 1
        num_pages = B * stride + 8
        bt = torch.from_numpy(inputs.block_tables([stride * 16] * B, 16, num_pages, 3)).to(dev)
        x = torch.randn((B * T, d), generator=g, device=dev).to(torch.bfloat16)
        cu = torch.arange(0, B * T + 1, T, dtype=torch.int32, device=dev)
        slots = torch.arange(B, dtype=torch.int32, device=dev)
        start = torch.full((B,), start_pos, dtype=torch.int32, device=dev)
        tab = torch.from_numpy(inputs.rope_table(start_pos + T + 16)).to(dev)
        caches = [KV4Cache(H, num_pages, B + 1, B, Hq, 16, 128) for _ in range(2)]
        y = torch.empty((B * T, N), dtype=torch.bfloat16, device=dev)
        q = torch.empty((B * T, Hq, 128), dtype=torch.bfloat16, device=dev)
        try:
            for c in caches:
                c.set_rope(tab)

            def fused(w):
                caches[0].qkv_append(x, w, Hq, cu, slots, start, bt, q_out=q)

            def apart(w):
                kv4.kv4_linear_bf16(x, w, y)
                kvp = y[:, Hq * 128:].view(B * T, H, 2, 128)      # the append takes [T][H][128] rows
                caches[1].append(kvp[:, :, 0].contiguous(), kvp[:, :, 1].contiguous(), cu, slots, start, bt)

            res = {}
            for name, fn in (("fused", fused), ("apart", apart)):
                for i in range(4):
                    fn(ws[i])
                torch.cuda.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    for i in range(reps):
                        fn(ws[i % len(ws)])
                graph.replay()
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                graph.replay()
                e1.record()
                torch.cuda.synchronize()
                del graph
                res[name] = e0.elapsed_time(e1) / reps
            if caches[0].device_error() or caches[1].device_error():
                raise RuntimeError("device error in the projection + append measurement")
            flops = 2.0 * B * T * N * d
            # bytes the fused call must move: W_qkv and X read, Q written in bf16, the INT4
            # pages and INT8 side rows of the new tokens written
            side_rows = B * T if start_pos == 0 else B
            nbytes = (N * d + B * T * d + B * T * Hq * 128) * 2 + \
                bytes_model.append_call_bytes(B * T, H, min(side_rows, B * 144) * H) - B * T * H * 512
            tfl = flops / (res["fused"] * 1e-3) / 1e12
            gbs = nbytes / (res["fused"] * 1e-3) / 1e9
            out[tag] = {"case": f"{B} sequences x {T} token(s) from position {start_pos}: X [{B * T}][{d}] "
                                f"x W_qkv [{N}][{d}], RoPE + Hadamard + 4-bit append of 8 KV heads; "
                                f"{len(ws)} copies of W_qkv cycled (weights never in L2)",
                        "fused_us": res["fused"] * 1e3, "apart_us": res["apart"] * 1e3,
                        "bound": "tensor" if flops / nbytes > peak_tf * 1e12 / (peak_hbm * 1e9) else "hbm",
                        "fused_tflops": tfl, "fused_frac_of_bf16_peak": tfl / peak_tf,
                        "algorithmic_bytes": nbytes, "fused_gbs": gbs, "fused_frac_of_hbm_peak": gbs / peak_hbm,
                        "speedup_over_apart": res["apart"] / res["fused"]}
        finally:
            for c in caches:
                c.close()
            del x, y, q
            torch.cuda.empty_cache()
    return out


def run_append_stress(dev, peak):
    """kv4_append on the append-stress shapes: (a) one new token for 512 sequences at
    position 2000, (b) a 16384-token re-prefill chunk for 8 sequences from position 0;
    8 KV heads, seeded bf16 K/V with outlier channels; each also with pre-RoPE keys and
    RoPE fused into the append (the table's reads are not counted). Device time per call:
    CUDA events around one replay of a CUDA graph of the repeated calls, after warm-up;
    GB/s counts bf16 K/V read, INT4 pages and INT8 side rows written."""
    from int8_hybrid_paged_gb300.kv4 import KV4Cache
    H, s, w = 8, 16, 128
    out = {}
    cases = (("b", 8, 16384, 0, 20, False), ("a", 512, 1, 2000, 200, False),
             ("b_rope", 8, 16384, 0, 20, True), ("a_rope", 512, 1, 2000, 200, True))
    for tag, B, T, start_pos, reps, rope in cases:
        stride = (start_pos + T + 15) // 16 + 1
        num_pages = B * stride + 8
        bt = torch.from_numpy(inputs.block_tables([stride * 16] * B, 16, num_pages, 1)).to(dev)
        k, v = inputs.kv_tokens(B * T, H, 23, device=dev)
        cu = torch.arange(0, B * T + 1, T, dtype=torch.int32, device=dev)
        slots = torch.arange(B, dtype=torch.int32, device=dev)
        start = torch.full((B,), start_pos, dtype=torch.int32, device=dev)
        cache = KV4Cache(H, num_pages, max_slots=B, max_batch=B, max_q_heads=4 * H, sink=s, window=w)
        if rope:                             # pre-RoPE keys: RoPE fused ahead of the Hadamard
            cache.set_rope(torch.from_numpy(inputs.rope_table(start_pos + T)).to(dev))
        try:
            for _ in range(3):
                cache.append(k, v, cu, slots, start, bt)
            torch.cuda.synchronize()
            # the calls are captured in a CUDA graph so the device time is measured, not
            # the host's launch rate (a one-token append is shorter than a Python call)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(reps):
                    cache.append(k, v, cu, slots, start, bt)
            graph.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            del graph
            if cache.device_error():
                raise RuntimeError("device error during the append stress")
            ms = e0.elapsed_time(e1) / reps
            side = B * (min(T, s + w) if start_pos == 0 else 1 + (1 if start_pos < s else 0))
            nbytes = bytes_model.append_call_bytes(B * T, H, side * H)
            gbs = nbytes / (ms * 1e-3) / 1e9
            out[tag] = {"case": f"{B} sequences x {T} token(s) from position {start_pos}, {H} KV heads"
                                + (", RoPE fused" if rope else ""),
                        "us_per_call": ms * 1e3, "algorithmic_bytes": nbytes, "achieved_gbs": gbs,
                        "frac_of_hbm_peak": gbs / peak}
        finally:
            cache.close()
            del k, v
            torch.cuda.empty_cache()
    return out


def run_e2e(st, wl, args, dev, world):
    """End to end through the public API from pinned host buffers: every step copies
    its q, context lengths, slot ids and block table in and its fp32 output out. Two
    steps are kept in flight (double buffers; inputs copied on a second stream while
    the previous step computes, the output copied out on a third stream as soon as its
    attention is done,
    the host waiting only for a buffer's previous step before reusing it); the strictly
    serial loop (host-synchronised every step) is reported beside it."""
    from int8_hybrid_paged_gb300 import kv4

    cache = st["cache"]
    B, Hq = wl.batch, wl.num_q_heads
    host = [dict(q=st["q"].cpu().pin_memory(), cl=st["cl"].cpu().pin_memory(),
                 sl=st["slots"].cpu().pin_memory(), bt=st["bt_dev"].cpu().pin_memory(),
                 out=torch.empty((B, Hq, 128), dtype=torch.float32).pin_memory()) for _ in range(2)]
    devb = [dict(q=torch.empty_like(st["q"]), cl=torch.empty_like(st["cl"]),
                 sl=torch.empty_like(st["slots"]), bt=torch.empty_like(st["bt_dev"]),
                 out=torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)) for _ in range(2)]
    comp = torch.cuda.current_stream(dev)
    copy_in = torch.cuda.Stream(device=dev)     # inputs of the next step, during this one
    copy_out = torch.cuda.Stream(device=dev)    # outputs of a finished step
    n = max(1, min(args.steps, 500))

    def enqueue(i, done):
        h, d = host[i % 2], devb[i % 2]
        if done[i % 2] is not None:
            done[i % 2].synchronize()          # the buffer's previous step has been read back
        ready = torch.cuda.Event()
        with torch.cuda.stream(copy_in):
            for k in ("q", "cl", "sl", "bt"):
                d[k].copy_(h[k], non_blocking=True)
            ready.record(copy_in)
        comp.wait_event(ready)
        for _ in range(wl.layers):
            kv4.kv4_decode_attention(cache.handle, d["q"], d["sl"], d["cl"], d["bt"], d["out"], None,
                                     stream=comp)
        computed = torch.cuda.Event()
        computed.record(comp)
        fin = torch.cuda.Event()
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(computed)
            h["out"].copy_(d["out"], non_blocking=True)
            fin.record(copy_out)
        done[i % 2] = fin

    def serial_step():
        h, d = host[0], devb[0]
        for k in ("q", "cl", "sl", "bt"):
            d[k].copy_(h[k], non_blocking=True)
        for _ in range(wl.layers):
            kv4.kv4_decode_attention(cache.handle, d["q"], d["sl"], d["cl"], d["bt"], d["out"], None,
                                     stream=comp)
        h["out"].copy_(d["out"], non_blocking=True)
        comp.synchronize()

    done = [None, None]
    for i in range(min(args.warmup, 5) + 2):
        enqueue(i, done)
    torch.cuda.synchronize()
    done = [None, None]
    barrier(world)
    t0 = time.perf_counter()
    for i in range(n):
        enqueue(i, done)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    for _ in range(3):
        serial_step()
    t1 = time.perf_counter()
    for _ in range(n):
        serial_step()
    el_serial = time.perf_counter() - t1
    toks = float(sum(st["lens"])) * wl.layers * n
    t_max, tok = reduce_max_sum(world, el, toks, dev)
    ts_max, _ = reduce_max_sum(world, el_serial, toks, dev)
    h0 = host[0]
    h2d = h0["q"].numel() * 2 + h0["cl"].numel() * 4 + h0["sl"].numel() * 4 + h0["bt"].numel() * 4
    d2h = h0["out"].numel() * 4
    return {"value": tok / t_max, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n,
            "serial_value": tok / ts_max,
            "how": "pinned host q, context_lens, slot_ids, block_table copied in and the fp32 "
                   "output copied out every step; two steps in flight (inputs on a copy stream "
                   "during the previous step's attention), wall clock over all steps; "
                   "serial_value: host-synchronised after every step"}


def run_reference(args, rank, world):
    """The CPU oracle on the host cores: every step decodes the same bounded sample as
    the main line's cpu_baseline (the workload's first sequences, drawn with the same
    recipe on the host), with OpenMP over (sequence, q head)."""
    if rank != 0:
        return
    import oracle

    oracle.load()
    wl = workload_from_args(args)
    lens = list(wl.context_lens)
    H, G, Hq = wl.num_kv_heads, wl.group, wl.num_q_heads
    threads = host_cores()
    nseq = min(ORACLE_SAMPLE_SEQS, wl.batch)
    seed = wl.seed
    cu = np.concatenate([[0], np.cumsum(lens[:nseq])]).astype(np.int64)
    k, v = inputs.kv_tokens(int(cu[-1]), H, seed * 1_000_003 + 17)
    kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
    qb = inputs.bf16_bits(inputs.queries(wl.batch, Hq, seed))[:nseq]
    oc = oracle.OracleCache(H, wl.sink, wl.window, max(lens[:nseq]), num_slots=nseq,
                            kv8=args.format == "int8", nvfp4=args.format == "nvfp4",
                            mxfp4=args.format == "mxfp4")
    for i in range(nseq):
        oc.append(i, 0, kb[cu[i]:cu[i + 1]], vb[cu[i]:cu[i + 1]])
    slots = np.arange(nseq, dtype=np.int32)
    sl = np.array(lens[:nseq], np.int32)
    used = min(threads, nseq * Hq)

    def step():
        oc.decode_batch(slots, sl, G, qb, 1 / math.sqrt(128), threads=used)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = float(sl.sum()) * args.steps / el
    sample = (f"first {nseq} of {len(lens)} sequences per step ({int(sl.sum())} context tokens, "
              f"{Hq} q heads; the main line's cpu_baseline sample, values drawn on the host), "
              f"OpenMP over (sequence, q head); host CPU: {cpu_model()}")
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "fp32/fp64 (CPU oracle)", "data": "synthetic",
           "config": workload_config(wl, world, call_bytes_for(wl, args.format), pool_pages_for(wl)),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def run_oracle_full(args):
    """The CPU oracle over a whole workload once: every sequence of the batch (of the
    long-tail stack, its first layer: the other 35 have the same shape), its caches built
    and decoded in groups of 16 sequences. Only the decodes are timed, with OpenMP over
    (sequence, q head) on the host cores and with one thread. The K/V and queries come
    from the CPU generator (the same shapes and distributions as the GPU run, not the
    same values: the GPU run draws them on the device). Prints one JSON line."""
    import oracle

    wl = inputs.workload(args.workload)
    kv8, fp4, mx = args.format == "int8", args.format == "nvfp4", args.format == "mxfp4"
    lens = list(wl.context_lens)
    H, G, Hq = wl.num_kv_heads, wl.group, wl.num_q_heads
    sink, window = (0, 0) if (kv8 or fp4 or mx) else (wl.sink, wl.window)
    t_build = time.perf_counter()
    k, v = inputs.kv_tokens(sum(lens), H, wl.seed * 1_000_003 + 17)
    q = inputs.bf16_bits(inputs.queries(wl.batch, Hq, wl.seed))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    build = time.perf_counter() - t_build
    threads = host_cores()
    t_omp = t_one = 0.0
    for g0 in range(0, wl.batch, 16):
        pick = list(range(g0, min(wl.batch, g0 + 16)))
        t0 = time.perf_counter()
        oc = oracle.OracleCache(H, sink, window, max(lens[b] for b in pick), num_slots=len(pick), kv8=kv8,
                                nvfp4=fp4, mxfp4=mx)
        for i, b in enumerate(pick):
            oc.append(i, 0, inputs.bf16_bits(k[cu[b]:cu[b + 1]]), inputs.bf16_bits(v[cu[b]:cu[b + 1]]))
        build += time.perf_counter() - t0
        slots = np.arange(len(pick), dtype=np.int32)
        sl = np.array([lens[b] for b in pick], np.int32)
        for nthreads in (threads, 1):
            t0 = time.perf_counter()
            oc.decode_batch(slots, sl, G, q[pick], 1 / math.sqrt(128), threads=nthreads)
            el = time.perf_counter() - t0
            if nthreads == 1:
                t_one += el
            else:
                t_omp += el
        del oc
    tokens = float(sum(lens))
    print(json.dumps({"impl": "oracle-full", "workload": wl.name, "format": args.format,
                      "context_tokens": int(tokens), "q_heads": Hq,
                      "decode_seconds": t_omp, "value": tokens / t_omp, "unit": UNIT, "cores": threads,
                      "one_thread": {"decode_seconds": t_one, "value": tokens / t_one, "cores": 1},
                      "cache_build_seconds_untimed": build,
                      "layers_note": ("one layer of the stack; the step is 36 such layers"
                                      if wl.layers > 1 else "the whole batch"),
                      "host_cpu": cpu_model(),
                      "inputs": "CPU generator stream: same shapes and distributions as the GPU run"}))


def main():
    args = parse()
    if args.oracle_full:
        run_oracle_full(args)
        return
    rank, world, local = dist_init(args)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_kv4(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
