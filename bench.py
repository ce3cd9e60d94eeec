"""Benchmark of the FP8 paged-KV decode step on GB300.

One step = one decode step of one layer of the workload: the tag check of
every request, the FP8 quantise-on-append of each passing request's new
token, and the split-K paged decode attention with its log-sum-exp combine,
all in one launch (kvq_decode_step).  --two-launch times the same step as
kvq_tag_check_append then kvq_decode_attn, --fused-append as kvq_tag_check
then kvq_decode_attn_append.  Default workload: 8 requests x 8,193 tokens,
GQA 64/8, head_dim 128, page 16, FP8 e4m3 cache with per-head scales, K/V ~
N(0,1) with 1 % outliers x20.

Prints one JSON line.  `value` is KV-read GB/s of the whole step (algorithmic
FP8 K+V bytes of all attended tokens / device time of the step); tokens/s,
the fraction of HBM peak and the BF16-cache comparison ride along.

  python bench.py [--steps K] [--warmup W] [--workload uniform8]
  python bench.py --impl reference     # the CPU oracle on the same workload
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 paged decode attn: KV-read GB/s (% of HBM peak) and decode tokens/s"
L2_FLUSH_BYTES = 512 << 20          # > 129 MB L2: written between timed steps
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_split_uniform8.json")
W4_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "w4a16_m1.json")
W4_SOURCES = ("kvq_w4a16.cu", "kvq_ptx.cuh")


def _code_only(text: str) -> str:
    """C/CUDA source without comments and with whitespace collapsed: what a
    kernel is built from, so that editing a comment keeps a profile valid."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(names=("kvq_decode.cu", "kvq_ptx.cuh")) -> str:
    """Hash of the code (comments aside) of a kernel's sources (by default the
    decode kernel, the one the decode roofline reports)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_quantised_paged_kv_gb300", "csrc")
    for name in names:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(path, workload, names=("kvq_decode.cu", "kvq_ptx.cuh")):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    summary is missing, is for another workload or predates the kernel's
    current source."""
    if not os.path.exists(path):
        return None
    prof = json.load(open(path))
    if prof.get("source_hash") == kernel_source_hash(names) and prof.get("workload") == workload:
        return prof.get("dram_bytes_per_launch")
    return None


def size_matched_read(nbytes, flush, stream, dev, launches=50):
    """Mean time of kvq_read_probe reading nbytes (random data) in one launch,
    L2 flushed before each launch, events around it on `stream`."""
    import torch
    import fp8_quantised_paged_kv_gb300 as kvq
    nbytes = nbytes // 16 * 16
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=dev, generator=g)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    evs = []
    with torch.cuda.stream(stream):
        for i in range(3 + launches):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            kvq.kvq_read_probe(src, sink, stream)
            e1.record(stream)
            if i >= 3:
                evs.append((e0, e1))
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    del src
    return {"what": "kvq_read_probe: one plain streaming kernel reading the same bytes, "
                    "L2 flushed, events around it",
            "us": round(ms * 1e3, 2), "gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
            "frac_of_peak": round(nbytes / (ms / 1e3) / 1e9 / measured_peaks()[0], 4)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clock / throttle samples (every 100 ms), each stamped with the
    host time it arrived, so the ones inside the timed region can be picked."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.samples = []

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self

        def reader():
            for line in self.proc.stdout:
                self.samples.append((time.perf_counter(), line))

        threading.Thread(target=reader, daemon=True).start()
        t0 = time.perf_counter()
        while not self.samples and time.perf_counter() - t0 < 5.0:   # wait for the first sample
            time.sleep(0.02)
        return self

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in list(self.samples):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        where = "timed region"
        if not inside:      # a region shorter than the 200 ms sampling period
            inside = [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25]
            where = "within 250 ms of the timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        reasons = sorted({n for r in inside for n, v in zip(self.NAMES, r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "samples": len(inside),
                "window": where, "reasons": reasons}


def aggregate_ranks(step_ms: float, kv_bytes: int, requests: int, device="cpu"):
    """Whole-job figures over all ranks: the slowest rank's step time, and the
    bytes / requests every rank processed in it (weak scaling, replicas)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        ms, total_bytes, total_req = step_ms, kv_bytes, requests
    else:
        t = torch.tensor([step_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        n = torch.tensor([kv_bytes, requests], dtype=torch.float64, device=device)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
        ms, total_bytes, total_req = float(t.item()), float(n[0].item()), float(n[1].item())
    return {"ms_per_step": ms, "value_gbs": total_bytes / (ms / 1e3) / 1e9,
            "tokens_per_s": total_req / (ms / 1e3)}


# ---------------------------------------------------------------- CPU oracle

def cpu_oracle_step_runner(workload: str, seed: int = 0, requests: int = 1):
    """The oracle on a bounded sample of the workload: its first ``requests``
    requests, same shapes and recipe (numpy inputs, host only).
    Returns (run_one_step, kv_bytes_per_step, cores, sub_workload)."""
    import dataclasses
    import oracle
    import workloads as W
    full = W.make(workload, seed)
    k = min(requests, full.batch)
    w = dataclasses.replace(full, batch=k, seq_lens=full.seq_lens[:k].copy(),
                            block_table=full.block_table[:k].copy(),
                            expected_tags=full.expected_tags[:k].copy())
    hv = W.host_values(w, seed)
    kc = np.zeros(w.cache_shape(), np.uint8)
    vc = np.zeros(w.cache_shape(), np.uint8)
    oracle.append(kc, vc, hv.k_prefill, hv.v_prefill, w.prefill_slot_mapping(), hv.k_scale,
                  hv.v_scale, page_size=w.page_size)
    slots = w.append_slot_mapping()

    def run():
        flags = oracle.tag_check(w.block_table, w.expected_tags, w.seq_lens, w.page_tags,
                                 page_size=w.page_size)
        oracle.append(kc, vc, hv.k_new, hv.v_new, slots, hv.k_scale, hv.v_scale, flags,
                      page_size=w.page_size)
        oracle.decode_attn(hv.q, kc, vc, hv.k_scale, hv.v_scale, w.block_table, w.seq_lens,
                           w.softmax_scale, flags)

    return run, w.kv_bytes(1), oracle.num_threads(), w


def cpu_baseline(workload: str, budget_s: float = 12.0):
    run, kv_bytes, cores, w = cpu_oracle_step_runner(workload, requests=1)
    t0 = time.perf_counter()
    n = 0
    while True:
        run()
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(kv_bytes * n / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{n} decode steps of {w.batch} of the {workload} requests "
                      f"({w.kv_tokens()} tokens each step: tag check, append, attention) "
                      f"in {dt:.1f} s, fp64 C oracle on the host CPU"}


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    import workloads as W
    full = W.make(args.workload, seed=0)               # the workload the GPU arm times
    run, kv_bytes, cores, w = cpu_oracle_step_runner(args.workload, requests=1)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = kv_bytes / (ms / 1e3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "batch": full.batch, "kv_tokens": full.kv_tokens(),
                   "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "page_size": w.page_size, "cache": "fp8_e4m3",
                   "out": "bf16", "step": "tag check, append and attention of each sampled request",
                   "sampled_requests": w.batch, "kv_tokens_per_step": w.kv_tokens(),
                   "parallelism": "host cores of rank 0"},
        "tokens_per_s": round(w.batch / (ms / 1e3), 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step = the decode step (tag check, append, attention) "
                                   f"of {w.batch} of the {args.workload} requests "
                                   f"({w.kv_tokens()} tokens), fp64 C oracle"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    import fp8_quantised_paged_kv_gb300 as kvq
    import workloads as W
    from kvq_harness import DeviceWorkload

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    kvq.load()
    kvq.kvq_device_error(clear=True)

    w = W.make(args.workload, seed=rank)
    dw = DeviceWorkload(w, kvq.KVQ_CACHE_FP8_E4M3, device=dev)
    ws = dw.workspace(args.num_splits)
    out = dw.out(False)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    kv_bytes = w.kv_bytes(1)
    split_tokens, max_splits, ws_bytes = kvq.kvq_decode_plan(dw.desc, w.batch, w.num_q_heads,
                                                             w.max_pages_per_seq, args.num_splits)
    counter_bytes = (w.batch * w.num_kv_heads * 4 + 255) // 256 * 256
    combine = ("none" if max_splits == 1 else
               "cluster (distributed shared memory)" if ws_bytes == counter_bytes else
               "workspace (last-arriving split)")

    one_launch = not (args.two_launch or args.fused_append)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if one_launch:                    # tag check + append + attention, one launch
            if ev is not None:
                ev[1].record(stream)
            dw.decode_step(out, ws, args.num_splits, stream)
            if ev is not None:
                ev[2].record(stream)
            return
        if args.fused_append:
            dw.tag_check(stream)               # batched tag check
        else:
            dw.tag_check_append(stream)        # batched tag check + FP8 append, one launch
        if ev is not None:
            ev[1].record(stream)
        if args.fused_append:                  # append of the new token inside the decode launch
            kvq.kvq_decode_attn_append(dw.desc, dw.q, dw.k_cache, dw.v_cache, dw.k_scale,
                                       dw.v_scale, dw.block_table, dw.seq_lens, w.softmax_scale,
                                       dw.abort, dw.k_new, dw.v_new, out, ws, args.num_splits,
                                       stream)
        else:
            kvq.kvq_decode_attn(dw.desc, dw.q, dw.k_cache, dw.v_cache, dw.k_scale, dw.v_scale,
                                dw.block_table, dw.seq_lens, w.softmax_scale, dw.abort, out, ws,
                                args.num_splits, stream)
        if ev is not None:
            ev[2].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            step()
    torch.cuda.synchronize()

    # Timed steps: events only at the step boundaries.  An event recorded
    # between the two launches would stop the decode kernel from starting
    # as a programmatic dependent of the step prologue.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local).start()
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.zero_()                 # L2 flushed before every timed step
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    t_wall = t_wall1 - t_wall0
    sampler.stop()
    if world > 1:
        dist.barrier()
    step_times = np.array([e[0].elapsed_time(e[1]) for e in evs])       # ms
    agg = aggregate_ranks(float(step_times.mean()), kv_bytes, w.batch, device=dev)
    step_ms = agg["ms_per_step"]

    # Per-kernel durations (same flush before every step), events around each
    # of the two launches; the decode kernel's is the roofline's denominator.
    k_steps = max(3, min(args.steps, 1000))
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(k_steps)]
    with torch.cuda.stream(stream):
        for i in range(k_steps):
            flush.zero_()
            step(kev[i])
    torch.cuda.synchronize()
    parts = np.array([[kev[i][j].elapsed_time(kev[i][j + 1]) for j in range(2)]
                      for i in range(k_steps)])             # ms
    pre_ms, attn_ms = (float(x) for x in parts.mean(axis=0))

    # ---- size-matched reference: how fast one plain streaming kernel reads
    # the same number of bytes on this GPU, under the same flush and event
    # protocol (kvq_read_probe over a buffer of random bytes).
    size_matched = size_matched_read(kv_bytes, flush, stream, dev)

    # ---- end to end: host (pinned) inputs -> device -> step -> host result.
    # The step's inputs (q, new K/V, slots, block table, lengths, expected
    # tags) live in one packed buffer: one host-to-device copy per step.
    host_buf, dev_buf = dw.pack_step_inputs()
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = host_buf.numel()
    d2h = out_host.numel() * out_host.element_size()
    e2e_steps = max(3, min(args.steps, 200))
    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(e2e_steps + 2):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dev_buf.copy_(host_buf, non_blocking=True)
            step()
            out_host.copy_(out, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            _ = float(out_host[0, 0, 0])      # the host reads the step's result
            if i >= 2:
                e2e_ms.append(e0.elapsed_time(e1))
    e2e_ms_mean = float(np.mean(e2e_ms))

    dev_err = kvq.kvq_device_error()
    peak, peak_kind = measured_peaks()
    achieved = kv_bytes / (attn_ms / 1e3) / 1e9
    traffic = profiled_traffic(PROFILE_SUMMARY, args.workload)

    # Steady state of a small workload: R steps back to back in one CUDA
    # graph, step r on its own copy of the cache (R copies together larger
    # than L2, so every step reads HBM), per-step time = graph time / R.
    steady = None
    if args.steady_copies > 0:
        R = args.steady_copies
        kc = [dw.k_cache.clone() for _ in range(R)]
        vc = [dw.v_cache.clone() for _ in range(R)]
        def steady_steps(st):
            for r in range(R):
                if one_launch:
                    kvq.kvq_decode_step(dw.desc, dw.q, kc[r], vc[r], dw.k_scale, dw.v_scale,
                                        dw.block_table, dw.seq_lens, dw.expected_tags, dw.page_tags,
                                        dw.abort, w.softmax_scale, dw.k_new, dw.v_new, out, ws,
                                        args.num_splits, st)
                    continue
                kvq.kvq_tag_check_append(dw.desc, dw.block_table, dw.expected_tags, dw.seq_lens,
                                         dw.page_tags, dw.k_new, dw.v_new, dw.append_slots,
                                         dw.k_scale, dw.v_scale, kc[r], vc[r], dw.abort, st)
                kvq.kvq_decode_attn(dw.desc, dw.q, kc[r], vc[r], dw.k_scale, dw.v_scale,
                                    dw.block_table, dw.seq_lens, w.softmax_scale, dw.abort, out, ws,
                                    args.num_splits, st)
        with torch.cuda.stream(stream):
            steady_steps(stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            steady_steps(torch.cuda.current_stream())
        torch.cuda.synchronize()
        gms = []
        with torch.cuda.stream(stream):
            for i in range(13):
                flush.zero_()
                g0 = torch.cuda.Event(enable_timing=True)
                g1 = torch.cuda.Event(enable_timing=True)
                g0.record(stream)
                graph.replay()
                g1.record(stream)
                if i >= 3:
                    gms.append((g0, g1))
        torch.cuda.synchronize()
        per_step_ms = float(np.mean([a.elapsed_time(b) for a, b in gms])) / R
        steady = {"copies_of_the_cache": R, "cache_bytes_total": R * 2 * dw.k_cache.numel(),
                  "us_per_step": round(per_step_ms * 1e3, 3),
                  "kv_gbs": round(kv_bytes / (per_step_ms / 1e3) / 1e9, 2),
                  "how": ("one CUDA graph of R back-to-back steps (" +
                          ("kvq_decode_step" if one_launch else "tag check + append, then decode") +
                          "), step r on cache copy r; L2 flushed before each replay")}
        del kc, vc, graph

    # BF16-cache comparison on the same workload (the same step form as the
    # FP8 kernel time it is compared with, L2 flushed)
    bf16_line = None
    if not args.skip_bf16:
        del dw
        torch.cuda.empty_cache()
        db = DeviceWorkload(w, kvq.KVQ_CACHE_BF16, device=dev)
        wsb = db.workspace(args.num_splits)
        ob = db.out(False)
        db.append()
        times = []
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush.zero_()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                if one_launch:
                    db.decode_step(ob, wsb, args.num_splits, stream)
                else:
                    db.attend(ob, wsb, None, args.num_splits, stream)
                b.record(stream)
                if i >= args.warmup:
                    times.append((a, b))
        torch.cuda.synchronize()
        bms = float(np.mean([a.elapsed_time(b) for a, b in times]))
        bf16_line = {"form": "kvq_decode_step" if one_launch else "kvq_decode_attn",
                     "kernel_us": round(bms * 1e3, 2), "kv_bytes": w.kv_bytes(2),
                     "kv_gbs": round(w.kv_bytes(2) / (bms / 1e3) / 1e9, 1),
                     "kv_bytes_per_token_per_layer": w.num_kv_heads * w.head_dim * 2 * 2,
                     "fp8_kv_bytes_per_token_per_layer": w.num_kv_heads * w.head_dim * 2,
                     "fp8_speedup": round(bms / attn_ms, 3)}

    if rank == 0:
        value = agg["value_gbs"]
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3",
            "data": "synthetic",
            "config": {"workload": args.workload, "batch": w.batch, "kv_tokens": w.kv_tokens(),
                       "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                       "head_dim": w.head_dim, "page_size": w.page_size, "cache": "fp8_e4m3",
                       "out": "bf16", "split_tokens": split_tokens, "max_splits": max_splits,
                       "split_combine": combine,
                       "step": ("kvq_decode_step (tag check, append and attention in one launch)"
                                if one_launch else
                                "kvq_tag_check, then kvq_decode_attn_append" if args.fused_append
                                else "kvq_tag_check_append, then kvq_decode_attn"),
                       "l2": "flushed before every timed step (512 MiB write)",
                       "parallelism": f"replicas x{world}"},
            "tokens_per_s": round(agg["tokens_per_s"], 1),
            "hbm_frac_of_measured": round(kv_bytes / (step_ms / 1e3) / 1e9 / peak, 4),
            "kernel_us": ({"decode_step (tag check + append + split + fused combine)": round(attn_ms * 1e3, 2)}
                          if one_launch else
                          {"tag_check": round(pre_ms * 1e3, 2),
                           "decode_attn_append (append + split + fused combine)": round(attn_ms * 1e3, 2)}
                          if args.fused_append else
                          {"tag_check_append": round(pre_ms * 1e3, 2),
                           "decode_attn (split + fused combine)": round(attn_ms * 1e3, 2)}),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "kernel": "decode_split_kernel", "peak_kind": peak_kind,
                         "algorithmic_bytes_per_launch": kv_bytes,
                         "size_matched_read": size_matched},
            "e2e": {"value": round(kv_bytes / (e2e_ms_mean / 1e3) / 1e9, 2), "unit": "GB/s",
                    "ms_per_step": round(e2e_ms_mean, 4), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": (1 if one_launch else 2) * args.steps,
            "bf16_cache": bf16_line,
            "steady_state_graph": steady,
            "clocks": sampler.summary(t_wall0, t_wall1),
            "wall_s_timed_region": round(t_wall, 3),
            "device_error_bits": dev_err,
        }
        if not args.skip_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_budget)
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_churn(args):
    """32-layer churn workload: per step one tag check, then for every layer
    the append of each request's new token and the decode attention.  Reports
    the KV bytes the step reads per second and the tag check's share of the
    step time (the pages' integrity-check overhead figure).  With --graph the
    65 launches of a step are captured once as a CUDA graph and replayed."""
    import torch
    import fp8_quantised_paged_kv_gb300 as kvq
    from kvq_churn import ChurnDevice, ChurnGraphStep, ChurnState

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    kvq.load()
    kvq.kvq_device_error(clear=True)
    st = ChurnState(seed=rank)
    dev = ChurnDevice(st, layers=32, device=f"cuda:{local}", log_layers=())
    gs = ChurnGraphStep(dev, fused_append=args.fused_append)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=f"cuda:{local}")
    if args.graph:
        gs.load()
        gs.capture()                     # consumes no step: the tables are reloaded below
    rows = []
    for i in range(args.warmup + args.steps):
        bt, exp, seq, stale, slots = gs.load()
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        if args.graph:
            gs.replay()
            e[1].record(stream)
        elif args.fused_append:
            kvq.kvq_tag_check(gs.bt, gs.exp, gs.seq, st.ps, gs.tags, dev.abort)
            e[1].record(stream)
            for l in range(dev.layers):
                kvq.kvq_decode_attn_append(dev.desc, gs.q[l], dev.k[l], dev.v[l], dev.k_scale[l],
                                           dev.v_scale[l], gs.bt, gs.seq, dev.sigma, dev.abort,
                                           gs.kn[l], gs.vn[l], gs.out[l], dev.ws)
        else:
            dev.kvq.kvq_tag_check(gs.bt, gs.exp, gs.seq, st.ps, gs.tags, dev.abort)
            e[1].record(stream)
            for l in range(dev.layers):
                kvq.kvq_append(dev.desc, gs.kn[l], gs.vn[l], gs.slots, dev.k_scale[l], dev.v_scale[l],
                               dev.abort, dev.k[l], dev.v[l])
                kvq.kvq_decode_attn(dev.desc, gs.q[l], dev.k[l], dev.v[l], dev.k_scale[l],
                                    dev.v_scale[l], gs.bt, gs.seq, dev.sigma, dev.abort, gs.out[l],
                                    dev.ws)
        e[2].record(stream)
        abort = dev.abort.cpu().numpy()
        live = (seq > 0) & (abort == 0)
        kv_bytes = int(seq[live].astype(np.int64).sum()) * dev.hkv * 256 * dev.layers
        if i >= args.warmup:
            rows.append((e[0], e[1], e[2], kv_bytes, int(live.sum())))
        st.advance(set(np.nonzero(abort)[0].tolist()))
    torch.cuda.synchronize()
    tag = np.array([a.elapsed_time(b) for a, b, _, _, _ in rows])
    step = np.array([a.elapsed_time(c) for a, _, c, _, _ in rows])
    kvb = np.array([r[3] for r in rows], np.float64)
    reqs = np.array([r[4] for r in rows], np.float64)
    value = float(kvb.sum() / (step.sum() / 1e3) / 1e9)
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(float(step.mean()), 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3",
            "data": "synthetic",
            "config": {"workload": "churn", "layers": 32, "batch": st.batch, "num_q_heads": dev.hq,
                       "num_kv_heads": dev.hkv, "page_size": st.ps,
                       "l2": "flushed before every timed step (512 MiB write)",
                       "step": "tag check once, then 32 x (append + decode attention)",
                       "launch": ("one CUDA graph replay" if args.graph else
                                  "33 launches" if args.fused_append else "65 launches"),
                       "append": ("inside each layer's decode launch" if args.fused_append
                                  else "its own launch per layer")},
            "tokens_per_s": round(float(reqs.sum() / (step.sum() / 1e3)), 1),
            "tag_check_us": None if args.graph else round(float(tag.mean() * 1e3), 2),
            "tag_check_share_of_step": None if args.graph else round(float(tag.sum() / step.sum()), 6),
            "gpu_launches": (33 if args.fused_append else 65) * args.steps,
            "device_error_bits": kvq.kvq_device_error(),
        }))
    return 0


def run_handoff(args):
    """Prefill -> decode handoff of a uniform8-sized prefill (8 requests x 8,192
    tokens, 8 KV heads, page 16): per-KV-head amax scales over the bf16 pages,
    then every page quantised into an e4m3 cache.  Reports each kernel's
    algorithmic bytes per second against the measured HBM peak."""
    import torch
    import fp8_quantised_paged_kv_gb300 as kvq

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    kvq.load()
    kvq.kvq_device_error(clear=True)
    ps, H, pages = 16, 8, 8 * 513
    g = torch.Generator(device=dev)
    g.manual_seed(rank)
    shape = (pages, H, ps, 128)
    ksrc = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    vsrc = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    src = torch.randperm(pages, generator=g, device=dev).to(torch.int32)
    dst = torch.randperm(pages, generator=g, device=dev).to(torch.int32)
    src_desc = kvq.CacheDesc(pages, ps, H, 128, kvq.KVQ_CACHE_BF16)
    dst_desc = kvq.CacheDesc(pages, ps, H, 128, kvq.KVQ_CACHE_FP8_E4M3)
    kd = torch.empty(shape, dtype=torch.uint8, device=dev)
    vd = torch.empty_like(kd)
    ks = torch.empty(H, dtype=torch.float32, device=dev)
    vs = torch.empty_like(ks)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    rows = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        kvq.kvq_amax_scales(src_desc, ksrc, vsrc, src, ks, vs)
        e[1].record(stream)
        kvq.kvq_quantize_pages(src_desc, ksrc, vsrc, src, dst_desc, kd, vd, dst, ks, vs)
        e[2].record(stream)
        if i >= args.warmup:
            rows.append(e)
    torch.cuda.synchronize()
    amax_ms = float(np.mean([r[0].elapsed_time(r[1]) for r in rows]))
    quant_ms = float(np.mean([r[1].elapsed_time(r[2]) for r in rows]))
    bf16_bytes = 2 * ksrc.numel() * 2
    amax_gbs = bf16_bytes / (amax_ms / 1e3) / 1e9
    quant_bytes = bf16_bytes + 2 * kd.numel()
    quant_gbs = quant_bytes / (quant_ms / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    value = (bf16_bytes + quant_bytes) / ((amax_ms + quant_ms) / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "prefill->decode handoff: bf16 pages -> e4m3 pages, algorithmic GB/s",
            "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(amax_ms + quant_ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3",
            "data": "synthetic",
            "config": {"workload": "handoff", "pages": pages, "page_size": ps, "num_kv_heads": H,
                       "head_dim": 128, "l2": "flushed before every timed step (512 MiB write)"},
            "kernel_us": {"amax_scales": round(amax_ms * 1e3, 2),
                          "quantize_pages": round(quant_ms * 1e3, 2)},
            "roofline": {"bound": "hbm", "kernel": "quantize_pages_kernel",
                         "achieved": round(quant_gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(quant_gbs / peak, 4), "traffic": None,
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": quant_bytes},
            "amax_scales_gbs": round(amax_gbs, 1),
            "gpu_launches": 2 * args.steps,
            "device_error_bits": kvq.kvq_device_error(),
        }))
    return 0


def run_w4a16(args):
    """INT4 weight-only product for decode: y = x W^T, W int4 [N][K/2] with a
    bf16 scale per column and 128-k group, x bf16 [M][K].  Shape: K = 8,192,
    N = 24,576 (100.7 MB of packed weights and scales, larger than L2); batch
    rows M = 1 (the value), 4 and 16.  Reports the weight bytes streamed per
    second against the measured HBM peak."""
    import torch
    import fp8_quantised_paged_kv_gb300 as kvq

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    kvq.load()
    kvq.kvq_device_error(clear=True)
    K, N = 8192, 24576
    g = torch.Generator(device=dev)
    g.manual_seed(rank)
    w = torch.randint(0, 256, (N, K // 2), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    sc = (torch.rand((N, K // 128), generator=g, device=dev) * 0.04 - 0.02).to(torch.bfloat16)
    wbytes = w.numel() + sc.numel() * 2
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()
    per_m = {}
    for M in (1, 4, 16):
        x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ts = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            kvq.kvq_w4a16_gemm(x, w, sc, y)
            e1.record(stream)
            if i >= args.warmup:
                ts.append((e0, e1))
        torch.cuda.synchronize()
        ms = float(np.mean([a.elapsed_time(b) for a, b in ts]))
        per_m[M] = {"us": round(ms * 1e3, 2), "weight_gbs": round(wbytes / (ms / 1e3) / 1e9, 1),
                    "splits": kvq.kvq_w4a16_plan(M, N, K)}
    main = per_m[1]
    size_matched = size_matched_read(wbytes, flush, stream, dev)
    if rank == 0:
        print(json.dumps({
            "metric": "INT4 weight-only decode product: weight bytes streamed per second",
            "value": main["weight_gbs"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(main["us"] / 1e3, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int4xbf16",
            "data": "synthetic",
            "config": {"workload": "w4a16", "m": 1, "k": K, "n": N, "group": 128,
                       "weight_bytes": wbytes, "l2": "flushed before every timed step (512 MiB write)"},
            "roofline": {"bound": "hbm", "kernel": "w4a16_kernel", "achieved": main["weight_gbs"],
                         "peak": peak, "unit": "GB/s", "frac": round(main["weight_gbs"] / peak, 4),
                         "traffic": profiled_traffic(W4_PROFILE_SUMMARY, "w4a16", W4_SOURCES),
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": wbytes,
                         "size_matched_read": size_matched},
            "by_batch_rows": per_m,
            "gpu_launches": args.steps * 3,
            "device_error_bits": kvq.kvq_device_error(),
        }))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="uniform8")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--skip-bf16", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true", help="churn: replay the step as a CUDA graph")
    ap.add_argument("--two-launch", action="store_true",
                    help="decode workloads: the step as kvq_tag_check_append, then kvq_decode_attn "
                         "(default: one kvq_decode_step launch)")
    ap.add_argument("--fused-append", action="store_true",
                    help="step = tag check, then decode attention with the append fused in")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--steady-copies", type=int, default=None,
                    help="also time R back-to-back steps in one CUDA graph over R cache copies "
                         "(default: 160 for tiny, else off)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.steady_copies is None:
        args.steady_copies = 160 if args.workload == "tiny" else 0
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "churn":
        return run_churn(args)
    if args.workload == "handoff":
        return run_handoff(args)
    if args.workload == "w4a16":
        return run_w4a16(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
