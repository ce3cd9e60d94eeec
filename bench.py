"""Benchmark of the FP8 paged-KV decode path on GB300.

Default run (no --workload): every workload, one JSON line.

  Headline (`value`, `config`): the churn workload -- 32 layers x 64
  requests, GQA 32/8, head_dim 128, page 16, contexts U{2,048..65,536},
  uint32 page tags, 20 % of the requests replaced and 0.5 % of the block-table
  entries stale each step.  One step: the batched tag check of every request,
  as its own launch that completes before any attention reads the cache;
  then, for each of the 32 layers, the paged decode attention over the FP8
  cache with the quantise-on-append of each passing request's new token
  (kvq_decode_attn_append; aborted requests get zeros and no write).
  value = FP8 K+V bytes the step's attention reads (every live request, all
  layers) / device time of the step.

  per_config: tiny, uniform8, ragged64 and long4 (one layer each), timed in
  the same form as the headline's layer: kvq_tag_check, then
  kvq_decode_attn_append (the attention with the append of each passing
  request's new token).  The whole step as
  one kvq_decode_step launch rides along as `one_launch`; it streams a
  split's pages before it learns the split's tag verdict, so it is not the
  timed step.  Every config also carries its BF16-cache step, a plain read
  of the same bytes, an end-to-end figure through host buffers and the CPU
  oracle's speed on a sample.

  extras: the prefill -> decode handoff quantiser and the INT4 product.

  python bench.py [--steps K] [--warmup W]
  python bench.py --workload {tiny,uniform8,ragged64,long4,churn,handoff,w4a16}
  python bench.py --impl reference    # the CPU oracle on a sample of the headline workload
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
L2_FLUSH_BYTES = 512 << 20          # > 129 MB L2: written, then another read, between timed steps
L2_FLUSH_NOTE = ("flushed before every timed step (a 512 MiB write, then a read of another "
                 "512 MiB buffer, so that no dirty line of the flush is written back inside "
                 "the timed region)")
DECODE_SOURCES = ("kvq_decode.cu", "kvq_ptx.cuh")
PROFILE_SUMMARIES = {                # committed ncu summaries of the decode kernel, by workload
    "tiny": os.path.join(ROOT, "profiles", "decode_split_tiny.json"),
    "uniform8": os.path.join(ROOT, "profiles", "decode_split_uniform8.json"),
    "ragged64": os.path.join(ROOT, "profiles", "decode_split_ragged64.json"),
    "long4": os.path.join(ROOT, "profiles", "decode_split_long4.json"),
    "churn": os.path.join(ROOT, "profiles", "decode_split_churn_layer.json"),
}
W4_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "w4a16_m1.json")
MT_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_mt_uniform8_n4.json")
# the tensor-memory kernel that takes 64 or more query rows per KV head
UMMA_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_mt_umma_uniform8_n8.json")
UMMA_SOURCES = ("kvq_decode_umma.cu", "kvq_umma.cuh", "kvq_ptx.cuh")
MULTI_TOKEN_CONFIGS = ("uniform8",)
STEADY_STATE_CONFIGS = ("tiny",)
W4_SOURCES = ("kvq_w4a16.cu", "kvq_ptx.cuh")
DECODE_CONFIGS = ("tiny", "uniform8", "ragged64", "long4")
# one layer of the churn workload's shape (64 requests, GQA 32/8, page 16,
# contexts U{2,048..65,536}) as a single-layer decode configuration: the case
# a decode-kernel profile of the headline is taken on (with --scale-down)
LAYER_SHAPES = {"churn_layer": "churn"}
HEADLINE = "churn"


def _code_only(text: str) -> str:
    """C/CUDA source without comments and with whitespace collapsed: what a
    kernel is built from, so that editing a comment keeps a profile valid."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(names=DECODE_SOURCES) -> str:
    """Hash of the code (comments aside) of a kernel's sources (by default the
    decode kernel, the one the decode roofline reports)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_quantised_paged_kv_gb300", "csrc")
    for name in names:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(path, workload, names=DECODE_SOURCES, units=None):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    summary is missing, is for another workload or predates the kernel's
    current source.  A summary taken on a smaller case of the workload
    states its algorithmic bytes; with `units` (this launch's algorithmic
    bytes) the traffic is scaled to them."""
    if path is None or not os.path.exists(path):
        return None
    prof = json.load(open(path))
    if prof.get("source_hash") != kernel_source_hash(names) or prof.get("workload") != workload:
        return None
    t = prof.get("dram_bytes_per_launch")
    if t is None or units is None or not prof.get("scaled_from_smaller_case"):
        return t
    return int(round(t * units / prof["algorithmic_bytes_per_launch"]))


def profiled_tensor_pipe(path, workload, names=DECODE_SOURCES):
    """Tensor-pipe and DRAM figures of a committed ncu summary of the
    multi-token launch, or None when it is missing or predates the source."""
    if not os.path.exists(path):
        return None
    prof = json.load(open(path))
    if prof.get("source_hash") != kernel_source_hash(names) or prof.get("workload") != workload:
        return None
    return {k: prof.get(k) for k in ("n_query", "tensor_pipe_active_pct", "dram_throughput_pct",
                                     "dram_bytes_per_launch", "gpu_time_duration_us_ncu")}


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
    host time it arrived, so the ones inside a timed region can be picked."""

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
        if not inside:      # a region shorter than the sampling period
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
                            expected_tags=full.expected_tags[:k].copy(), num_layers=1)
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


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu), or the machine type if unknown."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def cpu_baseline(workload: str, budget_s: float = 4.0, requests: int = 1):
    """The unchanged oracle, timed on the host cores for about budget_s
    seconds on a sample of the workload (its first `requests` requests, one
    layer): KV GB/s of the decode step it computes."""
    run, kv_bytes, cores, w = cpu_oracle_step_runner(workload, requests=requests)
    t0 = time.perf_counter()
    n = 0
    while True:
        run()
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(kv_bytes * n / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
            "cpu": host_cpu_model(), "nproc": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} decode steps (tag check, append, attention; one layer) of {w.batch} "
                      f"of the {workload} requests ({w.kv_tokens()} tokens each step) in "
                      f"{dt:.1f} s, fp64 C oracle on the host CPU"}


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    import workloads as W
    name = HEADLINE if args.workload in (None, "all") else args.workload
    full = W.make(name, seed=0)                        # the workload the GPU arm times
    run, kv_bytes, cores, w = cpu_oracle_step_runner(name, requests=1)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = kv_bytes / (ms / 1e3) / 1e9
    config = {"workload": name, "batch": full.batch, "num_q_heads": w.num_q_heads,
              "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
              "cache": "fp8_e4m3", "out": "bf16",
              "step": "tag check, append and attention of each sampled request, one layer",
              "sampled_requests": w.batch, "kv_tokens_per_step": w.kv_tokens(),
              "parallelism": "host cores of rank 0"}
    if name == "churn":
        config["layers"] = 32
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
        "tokens_per_s": round(w.batch / (ms / 1e3), 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "cpu": host_cpu_model(), "nproc": os.cpu_count(), "kind": "oracle",
                         "sample": f"each step = the decode step (tag check, append, attention) "
                                   f"of {w.batch} of the {name} requests in one layer "
                                   f"({w.kv_tokens()} tokens), fp64 C oracle"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm

class Env:
    """The GPU side of one run: device, stream, L2 flush buffer, peaks, clock
    samples and the rank layout."""

    def __init__(self, args):
        import torch
        import torch.distributed as dist
        import fp8_quantised_paged_kv_gb300 as kvq
        self.torch, self.dist, self.kvq, self.args = torch, dist, kvq, args
        self.rank, self.world, local = dist_info()
        torch.cuda.set_device(local)
        self.dev = f"cuda:{local}"
        if self.world > 1 and not dist.is_initialized():
            dist.init_process_group("nccl")
        kvq.load()
        kvq.kvq_device_error(clear=True)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=self.dev)
        self.flush_rd = torch.zeros(L2_FLUSH_BYTES, dtype=torch.uint8, device=self.dev)
        self.flush_sink = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.stream = torch.cuda.Stream(device=self.dev)
        self.peak, self.peak_kind = measured_peaks()
        self.sampler = ClockSampler(local).start()

    def event(self):
        return self.torch.cuda.Event(enable_timing=True)

    def flush_l2(self):
        """Write the 512 MiB buffer, then read another one: L2 holds none of
        the next step's data, and none of its lines is dirty.  (After the
        write alone, L2 holds ~129 MB of dirty lines whose write-back would
        share DRAM with the next step: +1.5 us on uniform8, +6 us on ragged64.)"""
        self.flush.zero_()
        self.kvq.kvq_read_probe(self.flush_rd, self.flush_sink, self.torch.cuda.current_stream())

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()
        self.torch.cuda.synchronize()

    def aggregate(self, ms, kv_bytes, requests):
        return aggregate_ranks(ms, kv_bytes, requests, device=self.dev)

    def close(self):
        self.sampler.stop()
        if self.world > 1 and self.dist.is_initialized():
            self.dist.destroy_process_group()


def size_matched_read(env, nbytes, launches=50):
    """Mean time of kvq_read_probe reading nbytes (random data) in one launch,
    L2 flushed before each launch, events around it on the bench stream."""
    torch, kvq = env.torch, env.kvq
    nbytes = nbytes // 16 * 16
    g = torch.Generator(device=env.dev)
    g.manual_seed(1234)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=env.dev, generator=g)
    sink = torch.zeros(1, dtype=torch.int32, device=env.dev)
    evs = []
    with torch.cuda.stream(env.stream):
        for i in range(3 + launches):
            env.flush_l2()
            e0, e1 = env.event(), env.event()
            e0.record(env.stream)
            kvq.kvq_read_probe(src, sink, env.stream)
            e1.record(env.stream)
            if i >= 3:
                evs.append((e0, e1))
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    del src
    return {"what": "kvq_read_probe: one plain streaming kernel reading the same bytes, "
                    "L2 flushed, events around it",
            "us": round(ms * 1e3, 2), "gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
            "frac_of_peak": round(nbytes / (ms / 1e3) / 1e9 / env.peak, 4)}


def _timed(env, fn, steps, warmup):
    """fn() `warmup` times untimed, then `steps` times with the L2 flushed
    before each and events around it on the bench stream: mean ms."""
    torch = env.torch
    evs = []
    with torch.cuda.stream(env.stream):
        for i in range(warmup + steps):
            env.flush_l2()
            e0, e1 = env.event(), env.event()
            e0.record(env.stream)
            fn()
            e1.record(env.stream)
            if i >= warmup:
                evs.append((e0, e1))
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in evs]))


def time_decode_config(env, name, with_cpu=True):
    """One layer of a decode workload: the step kvq_tag_check ->
    kvq_decode_attn_append timed over exactly args.steps steps, then the per-kernel
    split, the one-launch step, a plain read of the same bytes, the BF16
    cache, the host-fed step and the CPU oracle's speed."""
    import workloads as W
    from kvq_harness import DeviceWorkload
    torch, kvq, args, st = env.torch, env.kvq, env.args, env.stream
    w = W.make(LAYER_SHAPES.get(name, name), seed=env.rank, scale_down=args.scale_down)
    dw = DeviceWorkload(w, kvq.KVQ_CACHE_FP8_E4M3, device=env.dev)
    ws = dw.workspace(args.num_splits)
    out = dw.out(False)
    kv_bytes = w.kv_bytes(1)
    split_tokens, max_splits, ws_bytes = kvq.kvq_decode_plan(dw.desc, w.batch, w.num_q_heads,
                                                             w.max_pages_per_seq, args.num_splits)
    counter_bytes = (w.batch * w.num_kv_heads * 4 + 255) // 256 * 256
    combine = ("none" if max_splits == 1 else
               "cluster (distributed shared memory)" if ws_bytes == counter_bytes else
               "workspace (last-arriving split)")

    def step(mid=None):
        dw.tag_check(st)                  # the batched tag check, its own launch
        if mid is not None:
            mid.record(st)
        dw.attend_append(out, ws, args.num_splits, st)   # attention + append of passing requests

    with torch.cuda.stream(st):
        for _ in range(args.warmup):
            env.flush_l2()
            step()
    # Timed steps: events at the step boundaries only (an event between the
    # launches would stop the attention from starting as a programmatic
    # dependent of the check).
    evs = [(env.event(), env.event()) for _ in range(args.steps)]
    env.barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(st):
        for i in range(args.steps):
            env.flush_l2()
            evs[i][0].record(st)
            step()
            evs[i][1].record(st)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    env.barrier()
    agg = env.aggregate(float(np.mean([a.elapsed_time(b) for a, b in evs])), kv_bytes, w.batch)

    # per-kernel durations: an event between the two launches
    kev = [(env.event(), env.event(), env.event()) for _ in range(args.steps)]
    with torch.cuda.stream(st):
        for i in range(args.steps):
            env.flush_l2()
            kev[i][0].record(st)
            step(kev[i][1])
            kev[i][2].record(st)
    torch.cuda.synchronize()
    pre_ms = float(np.mean([a.elapsed_time(b) for a, b, _ in kev]))
    attn_ms = float(np.mean([b.elapsed_time(c) for _, b, c in kev]))
    achieved = kv_bytes / (attn_ms / 1e3) / 1e9

    one_ms = _timed(env, lambda: dw.decode_step(out, ws, args.num_splits, st), args.steps, 3)
    smr = size_matched_read(env, kv_bytes)

    # several new query tokens per request (kvq_decode_attn_mt, causal among
    # them) over the same cache: the attention launch alone
    multi = None
    if name in MULTI_TOKEN_CONFIGS:
        multi = {}
        g = torch.Generator(device=env.dev)
        g.manual_seed(77)
        for n in (2, 4, 8, 16):
            qn = torch.randn((w.batch, n, w.num_q_heads, w.head_dim), generator=g,
                             device=env.dev).to(torch.bfloat16)
            on = torch.empty_like(qn)
            wsn = kvq.workspace_for_mt(dw.desc, w.batch, n, w.num_q_heads, w.max_pages_per_seq,
                                       args.num_splits, env.dev)
            ms = _timed(env, lambda: kvq.kvq_decode_attn_mt(
                dw.desc, qn, dw.k_cache, dw.v_cache, dw.k_scale, dw.v_scale, dw.block_table,
                dw.seq_lens, w.softmax_scale, dw.abort, on, wsn, args.num_splits, st),
                args.steps, args.warmup)
            plan = kvq.kvq_decode_plan_mt(dw.desc, w.batch, n, w.num_q_heads, w.max_pages_per_seq,
                                          args.num_splits)
            multi[n] = {"us": round(ms * 1e3, 2), "kv_gbs": round(kv_bytes / (ms / 1e3) / 1e9, 1),
                        "frac_of_peak": round(kv_bytes / (ms / 1e3) / 1e9 / env.peak, 4),
                        "query_rows_per_kv_head": n * w.group, "max_splits": plan[1],
                        # the library's rule: 64 or more rows per KV head over FP8
                        "kernel": ("tcgen05, operands and accumulators in tensor memory"
                                   if n * w.group >= 64 else "mma.sync, 16 rows per CTA"),
                        "tokens_per_s": round(w.batch * n / (ms / 1e3), 1)}
            del qn, on, wsn
        mt_prof = profiled_tensor_pipe(MT_PROFILE_SUMMARY, name)
        if mt_prof is not None:
            multi["ncu_n4"] = mt_prof
        umma_prof = profiled_tensor_pipe(UMMA_PROFILE_SUMMARY, name, UMMA_SOURCES)
        if umma_prof is not None:
            multi["ncu_n8"] = umma_prof

    # Steady state of a small workload: R steps back to back in one CUDA
    # graph, step r on its own copy of the cache (the R copies together larger
    # than L2, so every step reads HBM); per-step time = graph time / R.
    steady = None
    if name in STEADY_STATE_CONFIGS:
        R = 160
        kc = [dw.k_cache.clone() for _ in range(R)]
        vc = [dw.v_cache.clone() for _ in range(R)]

        def steady_steps(s_):
            for r in range(R):
                kvq.kvq_tag_check(dw.block_table, dw.expected_tags, dw.seq_lens, w.page_size,
                                  dw.page_tags, dw.abort, s_)
                kvq.kvq_decode_attn_append(dw.desc, dw.q, kc[r], vc[r], dw.k_scale, dw.v_scale,
                                           dw.block_table, dw.seq_lens, w.softmax_scale, dw.abort,
                                           dw.k_new, dw.v_new, out, ws, args.num_splits, s_)
        with torch.cuda.stream(st):
            steady_steps(st)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            steady_steps(torch.cuda.current_stream())
        torch.cuda.synchronize()
        per_step_ms = _timed(env, graph.replay, 10, 3) / R
        steady = {"copies_of_the_cache": R, "cache_bytes_total": R * 2 * dw.k_cache.numel(),
                  "us_per_step": round(per_step_ms * 1e3, 3),
                  "kv_gbs": round(kv_bytes / (per_step_ms / 1e3) / 1e9, 2),
                  "how": "one CUDA graph of R back-to-back steps (kvq_tag_check, then "
                         "kvq_decode_attn_append), step r on cache copy r; L2 flushed before each replay"}
        del kc, vc, graph

    # end to end: the step's inputs (q, new K/V, slots, block table, lengths,
    # expected tags) copied from pinned host memory in one copy, the step,
    # and the output copied back and read on the host
    host_buf, dev_buf = dw.pack_step_inputs()
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e2e = []
    with torch.cuda.stream(st):
        for i in range(args.steps + 2):
            env.flush_l2()
            e0, e1 = env.event(), env.event()
            e0.record(st)
            dev_buf.copy_(host_buf, non_blocking=True)
            step()
            out_host.copy_(out, non_blocking=True)
            e1.record(st)
            e1.synchronize()
            _ = float(out_host[0, 0, 0])
            if i >= 2:
                e2e.append(e0.elapsed_time(e1))
    e2e_ms = float(np.mean(e2e))
    dev_err = kvq.kvq_device_error()
    del dw, ws, out, dev_buf
    torch.cuda.empty_cache()

    # the same step over the same workload in a BF16 cache (twice the bytes)
    bf16_ms = None
    if not args.skip_bf16:
        db = DeviceWorkload(w, kvq.KVQ_CACHE_BF16, device=env.dev)
        wsb = db.workspace(args.num_splits)
        ob = db.out(False)
        bf16_ms = _timed(env, lambda: (db.tag_check(st), db.attend_append(ob, wsb, args.num_splits, st)),
                         args.steps, args.warmup)
        del db, wsb, ob
        torch.cuda.empty_cache()

    res = {
        "config": {"workload": name, "batch": w.batch, "kv_tokens": w.kv_tokens(),
                   "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "page_size": w.page_size, "cache": "fp8_e4m3",
                   "out": "bf16", "split_tokens": split_tokens, "max_splits": max_splits,
                   "split_combine": combine,
                   "step": "kvq_tag_check, then kvq_decode_attn_append",
                   "l2": L2_FLUSH_NOTE},
        "value": round(agg["value_gbs"], 2), "unit": "GB/s",
        "ms_per_step": round(agg["ms_per_step"], 5),
        "tokens_per_s": round(agg["tokens_per_s"], 1),
        "hbm_frac_of_measured": round(kv_bytes / (agg["ms_per_step"] / 1e3) / 1e9 / env.peak, 4),
        "kernel_us": {"tag_check": round(pre_ms * 1e3, 2),
                      "decode_attn_append (append + split + fused combine)": round(attn_ms * 1e3, 2)},
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel", "achieved": round(achieved, 1),
                     "peak": env.peak, "unit": "GB/s", "frac": round(achieved / env.peak, 4),
                     "traffic": profiled_traffic(PROFILE_SUMMARIES.get(name), name, units=kv_bytes),
                     "peak_kind": env.peak_kind, "algorithmic_bytes_per_launch": kv_bytes,
                     "size_matched_read": smr},
        "one_launch": {"form": "kvq_decode_step (tag check folded into the attention launch: "
                               "a split streams its pages before its tag verdict)",
                       "us": round(one_ms * 1e3, 2),
                       "gbs": round(kv_bytes / (one_ms / 1e3) / 1e9, 1)},
        "bf16_cache": None if bf16_ms is None else {
            "step_us": round(bf16_ms * 1e3, 2), "kv_bytes": w.kv_bytes(2),
            "kv_gbs": round(w.kv_bytes(2) / (bf16_ms / 1e3) / 1e9, 1),
            "kv_bytes_per_token_per_layer": w.num_kv_heads * w.head_dim * 2 * 2,
            "fp8_kv_bytes_per_token_per_layer": w.num_kv_heads * w.head_dim * 2,
            "fp8_speedup": round(bf16_ms / agg["ms_per_step"], 3)},
        "e2e": {"value": round(kv_bytes / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": host_buf.numel(),
                "d2h_bytes_per_step": out_host.numel() * out_host.element_size()},
        "multi_token": multi,
        "steady_state_graph": steady,
        "gpu_launches": 2 * args.steps,
        "clocks": env.sampler.summary(t0, t1),
        "device_error_bits": dev_err,
    }
    if with_cpu and env.rank == 0 and not args.skip_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(LAYER_SHAPES.get(name, name), args.cpu_budget, requests=1)
    if args.scale_down != 1:
        res["config"]["scale_down"] = args.scale_down
    return res


def time_churn(env, with_cpu=True):
    """The 32-layer churn workload: per step the tag check (its own launch),
    then each layer's decode attention with the append of each passing
    request's token (kvq_decode_attn_append), over exactly args.steps steps;
    then a pass with events around every decode launch (the roofline), and a
    pass fed from host memory (end to end)."""
    from kvq_churn import ChurnDevice, ChurnGraphStep, ChurnState
    torch, kvq, args, st = env.torch, env.kvq, env.args, env.stream
    cs = ChurnState(seed=env.rank)
    with torch.cuda.stream(st):
        cd = ChurnDevice(cs, layers=32, device=env.dev, log_layers=())
        gs = ChurnGraphStep(cd, fused_append=not args.separate_append)
        host_in, dev_in = gs.pack_inputs()
        all_out = gs.pack_outputs()
    torch.cuda.synchronize()
    if args.graph:
        with torch.cuda.stream(st):
            gs.load()
        gs.capture()

    def one_step(timed_rows=None, layer_rows=None, from_host=False):
        with torch.cuda.stream(st):
            bt, exp, seq, stale, slots = gs.load()
            if from_host:
                host_in.copy_(dev_in)               # this step's inputs, now in host memory
                torch.cuda.synchronize()
            env.flush_l2()
            e = [env.event() for _ in range(3)]
            lev = None if layer_rows is None else [(env.event(), env.event()) for _ in range(cd.layers)]
            e[0].record(st)
            if from_host:
                dev_in.copy_(host_in, non_blocking=True)
            if args.graph and lev is None:
                gs.replay()
                e[1].record(st)
            else:
                gs.launch(st, after_check=e[1], layer_events=lev)
            if from_host:
                out_host.copy_(all_out, non_blocking=True)
                abort_host.copy_(cd.abort, non_blocking=True)
            e[2].record(st)
            e[2].synchronize()
            abort = (abort_host if from_host else cd.abort.cpu()).numpy()
        live = (seq > 0) & (abort == 0)
        layer_bytes = int(seq[live].astype(np.int64).sum()) * cd.hkv * 256
        if timed_rows is not None:
            timed_rows.append((e[0], e[1], e[2], layer_bytes * cd.layers, int(live.sum())))
        if layer_rows is not None:
            layer_rows.extend((a, b, layer_bytes) for a, b in lev)
        cs.advance(set(np.nonzero(abort)[0].tolist()))

    out_host = torch.empty(all_out.shape, dtype=all_out.dtype).pin_memory()
    abort_host = torch.empty(cd.abort.shape, dtype=cd.abort.dtype).pin_memory()
    for _ in range(args.warmup):
        one_step()
    rows = []
    env.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step(rows)
    t1 = time.perf_counter()
    env.barrier()
    tag = np.array([a.elapsed_time(b) for a, b, _, _, _ in rows])
    step = np.array([a.elapsed_time(c) for a, _, c, _, _ in rows])
    kvb = np.array([r[3] for r in rows], np.float64)
    reqs = np.array([r[4] for r in rows], np.float64)
    mean_ms = float(step.mean())
    agg = env.aggregate(mean_ms, float(kvb.mean()), float(reqs.mean()))

    lrows = []
    for _ in range(min(args.steps, 5)):
        one_step(layer_rows=lrows)
    torch.cuda.synchronize()
    l_ms = np.array([a.elapsed_time(b) for a, b, _ in lrows])
    l_bytes = np.array([c for _, _, c in lrows], np.float64)
    achieved = float(l_bytes.sum() / (l_ms.sum() / 1e3) / 1e9)
    per_launch = int(l_bytes.mean())

    erows = []
    for _ in range(args.steps):
        one_step(erows, from_host=True)
    e2e_ms = np.array([a.elapsed_time(c) for a, _, c, _, _ in erows])
    e2e_bytes = np.array([r[3] for r in erows], np.float64)
    dev_err = kvq.kvq_device_error()
    launches_per_step = 1 + cd.layers * (1 if gs.fused_append else 2)
    res = {
        "config": {"workload": "churn", "layers": cd.layers, "batch": cs.batch,
                   "num_q_heads": cd.hq, "num_kv_heads": cd.hkv, "head_dim": cd.D,
                   "page_size": cs.ps, "context": f"U{{{cs.lo}..{cs.hi}}}", "cache": "fp8_e4m3",
                   "out": "bf16",
                   "step": ("kvq_tag_check, then 32 x kvq_decode_attn_append" if gs.fused_append
                            else "kvq_tag_check, then 32 x (kvq_append, kvq_decode_attn)"),
                   "launch": "one CUDA graph replay" if args.graph else f"{launches_per_step} launches",
                   "churn": "20 % of requests replaced per step, 0.5 % of table entries stale",
                   "l2": L2_FLUSH_NOTE},
        "value": round(agg["value_gbs"], 2), "unit": "GB/s",
        "ms_per_step": round(agg["ms_per_step"], 5),
        "tokens_per_s": round(agg["tokens_per_s"], 1),
        "hbm_frac_of_measured": round(float(kvb.mean()) / (mean_ms / 1e3) / 1e9 / env.peak, 4),
        "kernel_us": {"tag_check": None if args.graph else round(float(tag.mean() * 1e3), 2),
                      "decode_attn per layer (mean)": round(float(l_ms.mean() * 1e3), 2)},
        "tag_check_share_of_step": None if args.graph else round(float(tag.sum() / step.sum()), 6),
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel", "achieved": round(achieved, 1),
                     "peak": env.peak, "unit": "GB/s", "frac": round(achieved / env.peak, 4),
                     "traffic": profiled_traffic(PROFILE_SUMMARIES["churn"], "churn",
                                                 units=per_launch),
                     "peak_kind": env.peak_kind, "algorithmic_bytes_per_launch": per_launch,
                     "launches_timed": len(lrows)},
        "e2e": {"value": round(float(e2e_bytes.sum() / (e2e_ms.sum() / 1e3) / 1e9), 2),
                "unit": "GB/s", "ms_per_step": round(float(e2e_ms.mean()), 4),
                "h2d_bytes_per_step": host_in.numel(),
                "d2h_bytes_per_step": out_host.numel() * out_host.element_size() + abort_host.numel()},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": env.sampler.summary(t0, t1),
        "device_error_bits": dev_err,
    }
    del gs, cd
    torch.cuda.empty_cache()
    if with_cpu and env.rank == 0 and not args.skip_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline("churn", args.cpu_budget, requests=1)
    return res


def time_handoff(env):
    """Prefill -> decode handoff of a uniform8-sized prefill (8 requests x 8,192
    tokens, 8 KV heads, page 16): per-KV-head amax scales over the bf16 pages,
    then every page quantised into an e4m3 cache."""
    torch, kvq, args = env.torch, env.kvq, env.args
    dev, st = env.dev, env.stream
    ps, H, pages = 16, 8, 8 * 513
    g = torch.Generator(device=dev)
    g.manual_seed(env.rank)
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
    rows = []
    with torch.cuda.stream(st):
        for i in range(args.warmup + args.steps):
            env.flush_l2()
            e = [env.event() for _ in range(3)]
            e[0].record(st)
            kvq.kvq_amax_scales(src_desc, ksrc, vsrc, src, ks, vs, st)
            e[1].record(st)
            kvq.kvq_quantize_pages(src_desc, ksrc, vsrc, src, dst_desc, kd, vd, dst, ks, vs, st)
            e[2].record(st)
            if i >= args.warmup:
                rows.append(e)
    torch.cuda.synchronize()
    amax_ms = float(np.mean([r[0].elapsed_time(r[1]) for r in rows]))
    quant_ms = float(np.mean([r[1].elapsed_time(r[2]) for r in rows]))
    bf16_bytes = 2 * ksrc.numel() * 2
    quant_bytes = bf16_bytes + 2 * kd.numel()
    quant_gbs = quant_bytes / (quant_ms / 1e3) / 1e9
    value = (bf16_bytes + quant_bytes) / ((amax_ms + quant_ms) / 1e3) / 1e9
    del ksrc, vsrc, kd, vd
    torch.cuda.empty_cache()
    return {
        "metric": "prefill->decode handoff: bf16 pages -> e4m3 pages, algorithmic GB/s",
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(amax_ms + quant_ms, 5),
        "dtype": "bf16->e4m3",
        "config": {"workload": "handoff", "pages": pages, "page_size": ps, "num_kv_heads": H,
                   "head_dim": 128, "l2": L2_FLUSH_NOTE},
        "kernel_us": {"amax_scales": round(amax_ms * 1e3, 2),
                      "quantize_pages": round(quant_ms * 1e3, 2)},
        "roofline": {"bound": "hbm", "kernel": "quantize_pages_kernel",
                     "achieved": round(quant_gbs, 1), "peak": env.peak, "unit": "GB/s",
                     "frac": round(quant_gbs / env.peak, 4), "traffic": None,
                     "peak_kind": env.peak_kind, "algorithmic_bytes_per_launch": quant_bytes},
        "amax_scales_gbs": round(bf16_bytes / (amax_ms / 1e3) / 1e9, 1),
        "gpu_launches": 2 * args.steps,
        "device_error_bits": kvq.kvq_device_error(),
    }


def time_w4a16(env):
    """INT4 weight-only product for decode: y = x W^T, W int4 [N][K/2] with a
    bf16 scale per column and 128-k group, x bf16 [M][K].  Shape: K = 8,192,
    N = 24,576 (100.7 MB of packed weights and scales, larger than L2); batch
    rows M = 1 (the value), 4 and 16."""
    torch, kvq, args = env.torch, env.kvq, env.args
    dev, st = env.dev, env.stream
    K, N = 8192, 24576
    g = torch.Generator(device=dev)
    g.manual_seed(env.rank)
    w = torch.randint(0, 256, (N, K // 2), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    sc = (torch.rand((N, K // 128), generator=g, device=dev) * 0.04 - 0.02).to(torch.bfloat16)
    wbytes = w.numel() + sc.numel() * 2
    per_m = {}
    for M in (1, 4, 16):
        x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ms = _timed(env, lambda: kvq.kvq_w4a16_gemm(x, w, sc, y, stream=st), args.steps, args.warmup)
        per_m[M] = {"us": round(ms * 1e3, 2), "weight_gbs": round(wbytes / (ms / 1e3) / 1e9, 1),
                    "splits": kvq.kvq_w4a16_plan(M, N, K)}
    main = per_m[1]
    smr = size_matched_read(env, wbytes)
    del w, sc
    torch.cuda.empty_cache()
    return {
        "metric": "INT4 weight-only decode product: weight bytes streamed per second",
        "value": main["weight_gbs"], "unit": "GB/s", "ms_per_step": round(main["us"] / 1e3, 5),
        "dtype": "int4xbf16",
        "config": {"workload": "w4a16", "m": 1, "k": K, "n": N, "group": 128,
                   "weight_bytes": wbytes, "l2": L2_FLUSH_NOTE},
        "roofline": {"bound": "hbm", "kernel": "w4a16_kernel", "achieved": main["weight_gbs"],
                     "peak": env.peak, "unit": "GB/s", "frac": round(main["weight_gbs"] / env.peak, 4),
                     "traffic": profiled_traffic(W4_PROFILE_SUMMARY, "w4a16", W4_SOURCES),
                     "peak_kind": env.peak_kind, "algorithmic_bytes_per_launch": wbytes,
                     "size_matched_read": smr},
        "by_batch_rows": per_m,
        "gpu_launches": args.steps * 3,
        "device_error_bits": kvq.kvq_device_error(),
    }


PHASES = ("entry", "wait returned", "first chunk landed", "streaming done", "merge done",
          "combine synchronised", "exit")


def run_phase_stamps(args):
    """Where the time of one decode step goes: the library built with
    per-CTA %globaltimer stamps (libkvq_stamps.so) runs the step of a decode
    workload (default uniform8) in three forms -- the conforming two-launch
    step (the tag check, then the attention with the append), the one-launch
    step and the attention launch alone -- with the L2
    flushed before each step; prints, per form, the median over steps of the
    min / median / max over CTAs of each phase's time from the step's first
    CTA entry, in microseconds."""
    import ctypes
    import torch
    import importlib
    import fp8_quantised_paged_kv_gb300 as kvq
    import workloads as W
    from kvq_harness import DeviceWorkload
    kbuild = importlib.import_module("fp8_quantised_paged_kv_gb300.build")
    kvq.load(kbuild.build(stamps=True))          # every call of this run goes to the instrumented build
    env = Env(args)
    lib = kvq.load()
    lib.kvq_phase_stamps.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t]
    lib.kvq_phase_stamps.restype = ctypes.c_int
    name = args.workload if args.workload in DECODE_CONFIGS else "uniform8"
    w = W.make(name)
    dw = DeviceWorkload(w, kvq.KVQ_CACHE_FP8_E4M3, device=env.dev)
    ws = dw.workspace(args.num_splits)
    out = dw.out(False)
    st = env.stream
    _, max_splits, _ = kvq.kvq_decode_plan(dw.desc, w.batch, w.num_q_heads, w.max_pages_per_seq,
                                           args.num_splits)
    n_cta = max_splits * w.num_kv_heads * w.batch
    dec = np.zeros(n_cta * 8, np.uint64)
    chk = np.zeros(w.batch * 2, np.uint64)
    forms = {
        "two_launch (kvq_tag_check, then kvq_decode_attn_append)":
            lambda: (dw.tag_check(st), dw.attend_append(out, ws, args.num_splits, st)),
        "one_launch (kvq_decode_step)": lambda: dw.decode_step(out, ws, args.num_splits, st),
        "attention alone (kvq_decode_attn)":
            lambda: dw.attend(out, ws, dw.abort, args.num_splits, st),
    }
    report = {}
    for form, fn in forms.items():
        rows = []
        with torch.cuda.stream(st):
            for i in range(args.warmup + args.steps):
                env.flush_l2()
                # the host synchronises after every step to read the stamps;
                # keep the GPU busy ~50 us so that the step's launches are all
                # queued before it runs (as they are in the timed loops)
                torch.cuda._sleep(100000)
                fn()
                torch.cuda.synchronize()
                if i < args.warmup:
                    continue
                assert lib.kvq_phase_stamps(0, dec.ctypes.data, dec.size) == 0
                assert lib.kvq_phase_stamps(2, chk.ctypes.data, chk.size) == 0
                d = dec.reshape(n_cta, 8).astype(np.int64)
                # nothing is cleared between launches: a CTA that streamed and
                # finished has an exit stamp later than its entry stamp
                streamed = d[d[:, 6] >= d[:, 0]]
                uses_check = form.startswith("two_launch")
                c = chk.reshape(w.batch, 2).astype(np.int64)
                t0 = min(int(c[:, 0].min()) if uses_check else 1 << 62, int(d[d[:, 0] > 0, 0].min()))
                row = {}
                if uses_check:
                    row["check kernel: first entry"] = (c[:, 0] - t0) / 1e3
                    row["check kernel: flags written"] = (c[:, 1] - t0) / 1e3
                for k, ph in enumerate(PHASES):
                    row[f"decode: {ph}"] = (streamed[:, k] - t0) / 1e3
                rows.append(row)
        summary = {}
        for key in rows[0]:
            stats = np.array([[np.min(r[key]), np.median(r[key]), np.max(r[key])] for r in rows])
            summary[key] = [round(float(x), 2) for x in np.median(stats, axis=0)]
        report[form] = summary
    if env.rank == 0:
        print(json.dumps({"what": "per-phase %globaltimer stamps, us from the step's first CTA entry: "
                                  "[min, median, max] over CTAs, median over steps",
                          "workload": name, "steps": args.steps, "ctas": n_cta,
                          "streaming_ctas_per_step": int(len(streamed)), "phases": report}))
    env.close()
    return 0


def _line(env, head, name):
    """The JSON line of the run whose headline is `head` (workload `name`)."""
    args = env.args
    line = {"metric": head.pop("metric", METRIC), "value": head.pop("value"),
            "unit": head.pop("unit", "GB/s"), "n_gpus": env.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head.pop("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": head.pop("dtype", "fp8_e4m3"), "data": "synthetic"}
    cfg = head.pop("config")
    cfg["parallelism"] = f"replicas x{env.world}"
    line["config"] = cfg
    line.update(head)
    return line


def run_gpu(args):
    env = Env(args)
    name = args.workload
    try:
        if name in (None, "all"):
            per = {}
            for c in DECODE_CONFIGS:
                per[c] = time_decode_config(env, c)
            extras = {}
            if not args.skip_extras:
                extras = {"handoff": time_handoff(env), "w4a16": time_w4a16(env)}
            head = time_churn(env)
            line = _line(env, head, HEADLINE)
            line["per_config"] = per
            line["extras"] = extras
        elif name in DECODE_CONFIGS or name in LAYER_SHAPES:
            line = _line(env, time_decode_config(env, name), name)
        elif name == "churn":
            line = _line(env, time_churn(env), name)
        elif name == "handoff":
            line = _line(env, time_handoff(env), name)
        elif name == "w4a16":
            line = _line(env, time_w4a16(env), name)
        else:
            raise SystemExit(f"unknown workload {name}")
        if env.rank == 0:
            print(json.dumps(line))
    finally:
        env.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all",
                    help="all (default: churn headline + every config), or one of "
                         "tiny, uniform8, ragged64, long4, churn, handoff, w4a16")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-bf16", action="store_true", help="decode configs: no BF16-cache step")
    ap.add_argument("--scale-down", type=int, default=1,
                    help="decode configs: context lengths divided by this (profiling cases)")
    ap.add_argument("--skip-extras", action="store_true", help="all: leave out handoff and w4a16")
    ap.add_argument("--graph", action="store_true", help="churn: replay the step as a CUDA graph")
    ap.add_argument("--separate-append", action="store_true",
                    help="churn: kvq_append and kvq_decode_attn per layer instead of "
                         "kvq_decode_attn_append")
    ap.add_argument("--phase-stamps", action="store_true",
                    help="per-phase breakdown of a decode workload's step (instrumented library)")
    ap.add_argument("--cpu-budget", type=float, default=4.0,
                    help="seconds of oracle time per CPU baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.phase_stamps:
        return run_phase_stamps(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
