"""Decode-step benchmark: RoPE-fused cache write + split-K paged attention +
log-sum-exp merge, on seeded synthetic inputs, one GPU per rank.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  `value` is the paged decode-attention KV-read
throughput: the attention's algorithmic bytes (every context token's K and V
row for every KV head, plus q, the fp32 output, the block-table entries in
use and the context lengths) per step, divided by the device time of the
whole step (write + partial + merge), summed over ranks.  Each rank is an
independent replica (the step has no exchange between GPUs).

The default workload is longctx_b256 (256 sequences, Llama-3.2-1B head
shapes, context U[512, 32768] with three 1-token contexts, bf16 KV, split-K
partition 512): about 9 GB of KV, far larger than the 129 MB L2, so no L2
flush is needed between steps.

--impl reference times the fp64 CPU oracle (the only other implementation of
this step) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode-attention KV-read GB/s (% of HBM peak) and decode steps/s"

# DRAM bytes (read + write) per launch of the partial kernel from an ncu
# capture, keyed by traffic_key(); trusted only while the kernel sources
# (comments aside) hash to the recorded value.
TRAFFIC = {
    # long-context step: ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum on the
    # decode launch of its first 64 sequences (2.2 GB of KV: a small capture), read + write,
    # scaled to the full launch by the algorithmic bytes (x 4.0724; traffic grows with the
    # pages read)
    "longctx_b256|native|seqs=all|part=default": {"bytes": 9045096923,
                                                  "measured": (2215400704 + 5686784, "seqs=64"),
                                                  "kernel_hash": "573448d600bc69c6"},
    "longctx_b256|fp8|seqs=all|part=default": {"bytes": 4520287318,
                                               "measured": (1106558720 + 3436800, "seqs=64"),
                                               "kernel_hash": "597c80618898b419"},
    # Qwen3 batch (0.5 GB of KV): the full launch, read + write
    "qwen3_ragged64|native|seqs=all|part=default": {"bytes": 545184512 + 3255808,
                                                    "kernel_hash": "573448d600bc69c6"},
    "qwen3_ragged64|fp8|seqs=all|part=default": {"bytes": 271084800 + 3226368,
                                                 "kernel_hash": "597c80618898b419"},
}


def traffic_key(args) -> str:
    return "%s|%s|seqs=%s|part=%s" % (args.workload, args.kv_dtype, args.max_seqs or "all",
                                      args.partition or "default")


# Sources of the decode kernel each KV dtype runs (the counters in TRAFFIC are
# tied to a hash of these files).
KERNEL_SOURCES = {
    "native": ("common.cuh", "internal.h", "paged_decode.cuh", "paged_decode_mma.cuh",
               "paged_decode_bf16.cu", "paged_decode_f32.cu"),
    "fp8": ("common.cuh", "internal.h", "paged_decode.cuh", "paged_decode_mma.cuh",
            "paged_decode_fp8.cu"),
}


def _strip_comments(src: bytes) -> bytes:
    """C/C++ source without // and /* */ comments or blank lines (string
    literals in these files hold no comment markers), so that editing a
    comment does not invalidate recorded counters."""
    text = re.sub(rb"/\*.*?\*/", b"", src, flags=re.S)
    text = re.sub(rb"//[^\n]*", b"", text)
    return b"\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kv_dtype: str = "native") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_write_gb300", "csrc")
    for f in KERNEL_SOURCES[kv_dtype]:
        if os.path.exists(os.path.join(csrc, f)):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + b"\0" + _strip_comments(fh.read()))
    return h.hexdigest()[:16]


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t_start=None, t_end=None, margin=0.25):
        """Samples taken in [t_start - margin, t_end + margin] (wall clock),
        or all samples when no window is given."""
        import datetime
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            if t_start is not None:
                try:
                    ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if ts < t_start - margin or ts > t_end + margin:
                    continue
            try:
                sm.append(float(f[2]))
                mx.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over the ranks of the default process group (the
    value itself without one, or with one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput_gbs(bytes_per_rank_step: int, world: int, ms_step_max: float) -> float:
    """Whole-job GB/s of N independent replicas: every rank's bytes over the
    slowest rank's step time."""
    return bytes_per_rank_step * world / (ms_step_max * 1e-3) / 1e9


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


L2_BYTES = 129 * 1024 * 1024
FLUSH_BELOW = 8 * L2_BYTES  # steps reading less than this are timed one by one with an L2 flush

# Other workloads timed in the same run, beside the headline (name, KV dtype).
EXTRA_WORKLOADS = (("qwen3_ragged64", "native"), ("qwen3_ragged64", "fp8"),
                   ("longctx_b256", "fp8"), ("cb_batch16", "native"),
                   ("llama1b_single", "native"), ("tiny_fp32", "native"))


def time_step(pk, wl, fp8, dev, stream, local, world, steps, warmup, seed, q_rope="none",
              use_graph=True, traffic_key_=None):
    """Times K decode steps (write + partial + merge, all layers) of one
    workload on this rank and each kernel alone.  Returns (summary, vals).

    Steps whose KV bytes exceed FLUSH_BELOW are timed as one bracket of K
    graph replays (inputs larger than L2); smaller ones one step at a time,
    each after a write of a 2 x L2 buffer that evicts the previous step's
    lines, with the events around the step alone."""
    import torch
    import torch.distributed as dist

    vals = (synth_mod().make_values_fp8 if fp8 else synth_mod().make_values)(wl, device=dev, seed=seed)
    L = wl.num_layers
    part = wl.partition_size
    sm_host = pk.photon_slot_mapping(wl.block_tables, wl.token_seq, wl.positions, wl.block_size)
    sm = torch.from_numpy(sm_host).to(dev)
    pos = torch.from_numpy(wl.positions).to(dev)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    cl = torch.from_numpy(wl.context_lens).to(dev)
    ws_bytes = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, wl.head_dim,
                                                        wl.max_context_len, part)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    out = torch.empty((L, wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
    split = ws_bytes > 0
    launches_per_step = L * (3 if split else 2) if wl.num_tokens else L * (2 if split else 1)
    q_pos = torch.from_numpy((wl.context_lens - 1).clip(min=0).astype(np.int32)).to(dev)

    def write(l):
        if fp8:
            if wl.num_tokens:
                pk.photon_kv_cache_write_fp8(vals["k"][l], vals["v"][l], pos, sm, vals["k_cache"][l],
                                             vals["v_cache"][l], vals["k_scale"][l], vals["v_scale"][l],
                                             wl.rope_theta, "neox", stream)
            return
        if q_rope == "fused":  # rotate this step's q rows in the same launch
            pk.photon_rope_q_kv_cache_write(vals["q"][l], q_pos, vals["k"][l], vals["v"][l], pos,
                                            sm, vals["k_cache"][l], vals["v_cache"][l],
                                            wl.rope_theta, "neox", stream)
            return
        if q_rope == "separate":  # the q rows in a launch of their own
            pk.photon_rope_q_kv_cache_write(vals["q"][l], q_pos, vals["k"][l][:0], vals["v"][l][:0],
                                            pos[:0], sm[:0], vals["k_cache"][l], vals["v_cache"][l],
                                            wl.rope_theta, "neox", stream)
        if wl.num_tokens:
            pk.photon_kv_cache_write(vals["k"][l], vals["v"][l], pos, sm, vals["k_cache"][l],
                                     vals["v_cache"][l], wl.rope_theta, "neox", stream)

    def partial(l):
        if fp8:
            pk.photon_paged_attention_partial_fp8(vals["q"][l], vals["k_cache"][l], vals["v_cache"][l],
                                                  vals["k_scale"][l], vals["v_scale"][l], bt, cl,
                                                  wl.scale, out[l], wl.max_context_len, part, ws,
                                                  stream)
            return
        pk.photon_paged_attention_partial(vals["q"][l], vals["k_cache"][l], vals["v_cache"][l], bt,
                                          cl, wl.scale, out[l], wl.max_context_len, part, ws, stream)

    def reduce(l):
        if split:
            pk.photon_paged_attention_reduce(cl, out[l], wl.max_context_len, part, ws, stream)

    def step():
        """One decode step over all layers: write, partial attention, merge."""
        for l in range(L):
            write(l)
            partial(l)
            reduce(l)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    def replay(g):
        with torch.cuda.stream(stream):
            g.replay()

    kvb = 1 if fp8 else None
    bytes_attn = synth_mod().kv_bytes_read(wl, kvb) * L
    flush = bytes_attn < FLUSH_BELOW
    # the flush writes a 2 x L2 buffer (evicting the step's inputs), then reads
    # another (so that L2 is left holding clean lines: dirty flush data would
    # otherwise be written back inside the next timed step)
    scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None
    scrub_r = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=dev) if flush else None

    def timed(run, n):
        """Device milliseconds of n calls of run(), with the L2 rule above."""
        if not flush:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                run()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                scrub.fill_(1)
                scrub_r.max()
                e0.record(stream)
                run()
                e1.record(stream)
        torch.cuda.synchronize()
        return sum(e0.elapsed_time(e1) for e0, e1 in evs)

    clk = ClockSampler(local).__enter__()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize()
    assert pk.photon_device_errors() == 0, "device error bits set during warm-up"
    if use_graph:
        g_step = capture(step)
        run = lambda: replay(g_step)
    else:
        run = step
    t_pre = time.time()
    while time.time() - t_pre < 0.5:  # untimed pre-roll while the clock sampler starts
        run()
        torch.cuda.synchronize()

    # timed region: K whole steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    ms_total = timed(run, steps)
    wall1 = time.time()
    clk.__exit__(None, None, None)
    if world > 1:
        dist.barrier()

    # per-kernel times: each kernel alone (all layers), K replays
    def time_kernel(fn):
        if use_graph:
            g = capture(lambda: [fn(l) for l in range(L)])
            go = lambda: replay(g)
        else:
            go = lambda: [fn(l) for l in range(L)]
        go()
        torch.cuda.synchronize()
        return timed(go, steps)

    ms_write = time_kernel(write) if wl.num_tokens else 0.0
    ms_partial = time_kernel(partial)
    ms_reduce = time_kernel(reduce) if split else 0.0
    assert pk.photon_device_errors() == 0, "device error bits set during the timed steps"
    ms_total = max_over_ranks(ms_total, dev)

    ms_step = ms_total / steps
    value = replica_throughput_gbs(bytes_attn, world, ms_step)
    peak, peak_src = hbm_peak()
    partial_ms = ms_partial / (steps * L)
    achieved = synth_mod().kv_bytes_read(wl, kvb) / (partial_ms * 1e-3) / 1e9
    kd = "fp8" if fp8 else "native"
    tr = TRAFFIC.get(traffic_key_) if traffic_key_ else None
    traffic = tr["bytes"] if (tr and tr.get("kernel_hash") == kernel_source_hash(kd)) else None
    summary = {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms_step, 5),
        "steps_per_s": round(1e3 / ms_step, 3), "pct_hbm_peak": round(100 * value / world / peak, 2),
        "config": {
            "workload": wl.name, "num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
            "kv_dtype": "fp8_e4m3" if fp8 else wl.kv_dtype, "layers": L, "partition_size": part,
            "total_context_tokens": int(wl.context_lens.sum()), "new_tokens": wl.num_tokens,
            "kv_bytes_per_step": bytes_attn,
            "l2": ("flushed before each timed step: a 2 x L2 buffer written, then another "
                   "2 x L2 buffer read (L2 left clean)" if flush
                   else "no flush: inputs larger than L2"),
        },
        "timing": ("CUDA events on the launching stream around "
                   + ("each step (L2 flushed in between)" if flush else "K whole steps")
                   + (" (replays of a CUDA graph of one step)" if use_graph else "")
                   + "; per-kernel times: each kernel alone, K "
                   + ("graph replays" if use_graph else "launch rounds")),
        "kernel_ms": {"kv_cache_write": round(ms_write / (steps * L), 5),
                      "paged_decode_partial": round(partial_ms, 5),
                      "lse_reduce": round(ms_reduce / (steps * L), 5)},
        "roofline": {"bound": "hbm", "kernel": "paged_decode_partial" + ("_fp8" if fp8 else ""),
                     "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_src,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": synth_mod().kv_bytes_read(wl, kvb)},
        "launches_per_step": launches_per_step,
        "clocks": clk.summary(wall0, wall1),
        "kernel_source_hash": kernel_source_hash(kd),
        "suspect": value / world > 1.15 * peak,  # faster than a plain copy: not doing the work
    }
    return summary, vals


def synth_mod():
    import synth
    return synth


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import paged_kv_decode_write_gb300 as pk
    import synth

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream()

    wl = synth.make(args.workload, seed=args.seed)
    if args.max_seqs:
        wl = synth.truncate(wl, args.max_seqs)
    if args.partition:
        wl = dataclasses.replace(wl, partition_size=args.partition)
    fp8 = args.kv_dtype == "fp8"
    if fp8 and (wl.kv_dtype != "bf16" or wl.head_dim not in (64, 128)):
        raise SystemExit("--kv-dtype fp8 needs a bf16 workload with head_dim 64 or 128")
    head, vals = time_step(pk, wl, fp8, dev, stream, local, world, args.steps, args.warmup,
                           args.seed + rank, q_rope=args.q_rope, use_graph=not args.no_graph,
                           traffic_key_=traffic_key(args))
    cfg = head.pop("config")
    cfg.update({"parallelism": f"replicas{world}", "seed": args.seed,
                "max_seqs": args.max_seqs or None, "q_rope": args.q_rope})
    result = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": cfg,
    }
    for key in ("steps_per_s", "pct_hbm_peak", "timing", "kernel_ms", "roofline"):
        result[key] = head[key]
    result["gpu_launches"] = head["launches_per_step"] * args.steps
    for key in ("clocks", "kernel_source_hash", "suspect"):
        result[key] = head[key]
    result["scheduler"] = time_scheduler(pk, wl)
    if not fp8:
        result["prefill"] = time_prefill(pk, dev, stream)
    if not args.no_e2e and not fp8:
        result["e2e"] = run_e2e(args, wl, vals, pk, dev, stream, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not fp8:
        result["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    del vals
    torch.cuda.empty_cache()
    if not args.no_workloads and not args.max_seqs and not args.partition:
        result["workloads"] = {}
        for name, kd in EXTRA_WORKLOADS:
            if (name, kd) == (args.workload, args.kv_dtype):
                continue
            w = synth.make(name, seed=args.seed)
            sub, v = time_step(pk, w, kd == "fp8", dev, stream, local, world, args.steps,
                               args.warmup, args.seed + rank, use_graph=not args.no_graph,
                               traffic_key_="%s|%s|seqs=all|part=default" % (name, kd))
            del v
            torch.cuda.empty_cache()
            sub["gpu_launches"] = sub.pop("launches_per_step") * args.steps
            result["workloads"]["%s|%s" % (name, kd)] = sub
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def time_scheduler(pk, wl, steps=200):
    """Host time of one two-phase scheduler step (plan + complete) with the
    workload's batch size running: requests shaped like its sequences (prompt =
    context length), enough new tokens to stay running."""
    B = wl.num_seqs
    width = max(wl.max_blocks_per_seq, 1) + steps // wl.block_size + 2
    need = int(sum(-(-int(c + steps) // wl.block_size) for c in wl.context_lens)) + B
    pool = pk.BlockPool(need, seed=1)
    sched = pk.Scheduler(pool, max_running=B,
                         max_step_tokens=int(wl.context_lens.sum()) + B * (steps + 2),
                         max_blocks_per_seq=width)
    for i, c in enumerate(wl.context_lens):
        sched.add_request(i, max(int(c), 1), steps + 2)
    sched.schedule()  # admission (prefill) step, not timed
    sched.complete_step()
    t = time.perf_counter()
    for _ in range(steps):
        sched.schedule(copy=False)
        sched.complete_step()
    us = (time.perf_counter() - t) / steps * 1e6
    return {"us_per_step": round(us, 2), "running": B, "steps": steps,
            "what": "native two-phase scheduler: plan (block growth, batch metadata) + complete, host"}


def _time_prefill_call(pk, dev, stream, wl, part, steps, seed=5):
    """Microseconds per photon_paged_attention_prefill call over the
    workload's written tokens (random bf16 queries), as CUDA-graph replays."""
    import torch
    vals = synth_values(wl, dev)
    g = torch.Generator(device=dev).manual_seed(seed)
    q = (torch.randn((wl.num_tokens, wl.num_q_heads, wl.head_dim), generator=g, device=dev) * 0.5).bfloat16()
    ts = torch.from_numpy(wl.token_seq).to(dev)
    pos = torch.from_numpy(wl.positions).to(dev)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    maxp = int(wl.positions.max())
    n = pk.photon_paged_attention_workspace_size(wl.num_tokens, wl.num_q_heads, wl.head_dim, maxp + 1, part)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
    out = torch.empty((wl.num_tokens, wl.num_q_heads, wl.head_dim), device=dev)
    call = lambda: pk.photon_paged_attention_prefill(q, ts, pos, vals["k_cache"][0], vals["v_cache"][0],
                                                     bt, wl.scale, out, maxp, part, ws, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graph.replay()
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    assert pk.photon_device_errors() == 0, "device error bits set during the prefill timing"
    return e0.elapsed_time(e1) / steps * 1e3


def synth_values(wl, dev):
    import synth
    return synth.make_values(wl, device=dev)


def time_prefill(pk, dev, stream, steps=50):
    """Causal prefill over the paged cache, timed as CUDA-graph replays:
    (1) the continuous-batching step's written tokens (4 admitted 100-token
    prompts plus every sequence's decode token, 416 query tokens, Llama heads,
    bf16, partition 64); (2) 8 whole 2048-token prompts (16384 query tokens,
    partition 512) with Llama heads (32/8, d 64) and with Qwen3 heads (16/8,
    d 128).  Attention FLOPs count 4 * d per (query head, visible key) pair."""
    import synth
    wl = synth.make("cb_batch16")
    us = _time_prefill_call(pk, dev, stream, wl, 64, steps)
    ctx = wl.positions.astype(np.int64) + 1
    kv_bytes = int(ctx.sum()) * wl.num_kv_heads * wl.head_dim * 2 * 2
    res = {"us_per_call": round(us, 2), "query_tokens": wl.num_tokens,
           "tokens_per_s": round(wl.num_tokens / (us * 1e-6), 1),
           "kv_bytes_per_call_per_query_token_reads": kv_bytes,
           "what": "causal prefill of cb_batch16's written tokens (graph replays)"}
    for key, (hq, hkv, d, heads) in (("long_prompts", (32, 8, 64, "Llama heads")),
                                     ("long_prompts_d128", (16, 8, 128, "Qwen3 heads (16/8, d 128)"))):
        lw = synth.make_custom([2048] * 8, hq, hkv, d, kv_dtype="bf16", seed=1, value_std=0.5,
                               tokens_per_seq=2048)
        lus = _time_prefill_call(pk, dev, stream, lw, 512, max(5, steps // 10))
        pairs = int((lw.positions.astype(np.int64) + 1).sum()) * lw.num_q_heads
        res[key] = {"us_per_call": round(lus, 1), "query_tokens": lw.num_tokens,
                    "tokens_per_s": round(lw.num_tokens / (lus * 1e-6), 1),
                    "attention_tflops": round(4 * lw.head_dim * pairs / (lus * 1e-6) / 1e12, 2),
                    "what": "8 whole 2048-token prompts, %s, bf16 (graph replays)" % heads}
    return res


def run_e2e(args, wl, vals, pk, dev, stream, world):
    """The same metric through the public calls with HOST buffers, as a
    serving loop runs it: every step the host builds the slot numbers, copies
    q, the new k/v, positions, slot numbers, block tables and context lengths
    from pinned memory to the device, runs write + attention, and reads the
    output back to pinned memory.  Inputs and outputs are double-buffered:
    step i+1's inputs travel on a copy stream while step i computes, and step
    i's output travels back on another while step i+1 computes.  Events order
    every reuse of a buffer; the clock stops after the last read-back."""
    import torch
    import torch.distributed as dist
    L = wl.num_layers
    part = wl.partition_size
    # every input of a step lives in one pinned staging buffer (one copy per
    # step), 256-byte aligned parts; the device side views the same layout
    T = wl.num_tokens
    parts = [("bt", torch.from_numpy(wl.block_tables)), ("cl", torch.from_numpy(wl.context_lens)),
             ("pos", torch.from_numpy(wl.positions)), ("sm", torch.zeros(T, dtype=torch.int64))]
    for l in range(L):
        parts += [("q%d" % l, vals["q"][l].cpu()), ("k%d" % l, vals["k"][l].cpu()),
                  ("v%d" % l, vals["v"][l].cpu())]
    layout, total = {}, 0
    for name, t in parts:
        nbytes = t.numel() * t.element_size()
        layout[name] = (total, nbytes, t.dtype, tuple(t.shape))
        total += (nbytes + 255) // 256 * 256
    total = max(total, 256)
    h_stage = [torch.empty(total, dtype=torch.uint8).pin_memory() for _ in range(2)]
    for hs in h_stage:
        for name, t in parts:
            off, nbytes, _, _ = layout[name]
            hs[off:off + nbytes].copy_(t.contiguous().view(-1).view(torch.uint8))
    sm_off, sm_bytes = layout["sm"][0], layout["sm"][1]
    h_sm = [hs[sm_off:sm_off + sm_bytes].view(torch.int64) for hs in h_stage]
    h_out = [torch.empty((L, wl.num_seqs, wl.num_q_heads, wl.head_dim),
                         dtype=torch.float32).pin_memory() for _ in range(2)]

    def dev_set():
        buf = torch.empty(total, dtype=torch.uint8, device=dev)

        def view(name):
            off, nbytes, dtype, shape = layout[name]
            return buf[off:off + nbytes].view(dtype).view(shape)

        return {"buf": buf, "q": [view("q%d" % l) for l in range(L)],
                "k": [view("k%d" % l) for l in range(L)], "v": [view("v%d" % l) for l in range(L)],
                "bt": view("bt"), "cl": view("cl"), "pos": view("pos"), "sm": view("sm"),
                "out": torch.empty_like(h_out[0], device=dev)}

    d = [dev_set(), dev_set()]
    ws_bytes = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, wl.head_dim,
                                                        wl.max_context_len, part)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    h2d = total
    d2h = h_out[0].numel() * h_out[0].element_size()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready, in_copied, computed, out_read = ([ev(), ev()] for _ in range(4))
    used = [False, False]  # buffer set b has been through one step (its events are recorded)

    def upload(i):
        b = i % 2
        if used[b]:
            in_copied[b].synchronize()  # h_stage[b]'s previous copy has left host memory
        if T:
            h_sm[b].numpy()[:] = pk.photon_slot_mapping(wl.block_tables, wl.token_seq,
                                                        wl.positions, wl.block_size)
        with torch.cuda.stream(up):
            if used[b]:
                up.wait_event(computed[b])  # step i-2 is done reading set b
            d[b]["buf"].copy_(h_stage[b], non_blocking=True)
            in_ready[b].record(up)
            in_copied[b].record(up)

    def compute(i):
        b = i % 2
        x = d[b]
        with torch.cuda.stream(stream):
            stream.wait_event(in_ready[b])
            if used[b]:
                stream.wait_event(out_read[b])  # step i-2's output has been read back
            for l in range(L):
                if wl.num_tokens:
                    pk.photon_kv_cache_write(x["k"][l], x["v"][l], x["pos"], x["sm"],
                                             vals["k_cache"][l], vals["v_cache"][l], wl.rope_theta,
                                             "neox", stream)
                pk.photon_paged_attention_decode(x["q"][l], vals["k_cache"][l], vals["v_cache"][l],
                                                 x["bt"], x["cl"], wl.scale, x["out"][l],
                                                 wl.max_context_len, part, ws, stream)
            computed[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(computed[b])
            h_out[b].copy_(x["out"], non_blocking=True)
            out_read[b].record(down)
        used[b] = True

    def run(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute(i)
        torch.cuda.synchronize()

    run(args.warmup)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t = time.perf_counter()
    run(args.steps)
    dt = time.perf_counter() - t
    dt = max_over_ranks(dt, dev)
    # the loop must have computed the step: its last read-back equals the same
    # decode launched on the device-resident inputs (deterministic kernels)
    ref = torch.empty_like(d[0]["out"])
    with torch.cuda.stream(stream):
        for l in range(L):
            pk.photon_paged_attention_decode(vals["q"][l], vals["k_cache"][l], vals["v_cache"][l],
                                             d[0]["bt"], d[0]["cl"], wl.scale, ref[l],
                                             wl.max_context_len, part, ws, stream)
    torch.cuda.synchronize()
    assert torch.equal(ref.cpu(), h_out[(args.steps - 1) % 2]), "end-to-end loop output differs"
    import synth
    val = replica_throughput_gbs(synth.kv_bytes_read(wl) * L, world, 1e3 * dt / args.steps)
    return {"value": round(val, 2), "unit": "GB/s", "ms_per_step": round(1e3 * dt / args.steps, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "timing": "wall clock over K steps of a double-buffered serving loop: host slot "
                      "numbers and pinned H2D of step i+1 overlap step i's kernels; every "
                      "step's output is read back to pinned memory"}


# ---------------------------------------------------------------- oracle arm

def _oracle_sample(wl, target_seconds, seed=0):
    """Picks sequences of the workload (seeded order) until their estimated
    oracle cost reaches the time target, and builds their host inputs."""
    import torch

    import oracle
    import synth
    rng = np.random.default_rng(seed)
    order = rng.permutation(wl.num_seqs)
    # calibration: ~ seconds per (token x q-head x dim) of this host
    probe = synth.make_custom([2048] * 2, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                              kv_dtype=wl.kv_dtype, seed=1)
    pv = synth.make_values(probe)
    hp = {n: synth.to_storage_numpy(pv[n][0]).copy() for n in ("q", "k_cache", "v_cache")}
    t = time.perf_counter()
    oracle.paged_attention(hp["q"], hp["k_cache"], hp["v_cache"], probe.block_tables,
                           probe.context_lens, probe.scale)
    per = (time.perf_counter() - t) / (2 * 2048 * wl.num_q_heads * wl.head_dim)
    pick, cost = [], 0.0
    for s in order:
        c = max(int(wl.context_lens[s]), 1) * wl.num_q_heads * wl.head_dim * per * wl.num_layers
        if pick and cost + c > target_seconds:
            continue
        pick.append(int(s))
        cost += c
        if cost >= 0.9 * target_seconds:
            break
    pick.sort()
    sub = synth.make_custom(wl.context_lens[pick], wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                            kv_dtype=wl.kv_dtype, seed=seed, rope_theta=wl.rope_theta,
                            value_std=wl.value_std, num_layers=wl.num_layers,
                            partition_size=wl.partition_size)
    return pick, sub


def _oracle_step_seconds(sub, host):
    import oracle
    t = time.perf_counter()
    for l in range(sub.num_layers):
        h = host[l]
        sm = oracle.slot_mapping(sub.block_tables, sub.token_seq, sub.positions, sub.block_size)
        kc, vc = h["k_cache"], h["v_cache"]
        oracle.kv_cache_write(h["k"], h["v"], sub.positions, sm, kc, vc, sub.rope_theta)
        oracle.paged_attention(h["q"], kc, vc, sub.block_tables, sub.context_lens, sub.scale)
    return time.perf_counter() - t


def cpu_baseline(wl, target_seconds):
    import oracle
    import synth
    pick, sub = _oracle_sample(wl, target_seconds)
    vals = synth.make_values(sub)
    host = [{n: synth.to_storage_numpy(vals[n][l]).copy() for n in ("q", "k", "v", "k_cache", "v_cache")}
            for l in range(sub.num_layers)]
    sec = _oracle_step_seconds(sub, host)
    b = synth.kv_bytes_read(sub) * sub.num_layers
    return {"value": round(b / sec / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(sec, 3),
            "sample": f"{len(pick)} of {wl.num_seqs} sequences ({int(sub.context_lens.sum())} context "
                      f"tokens x {sub.num_layers} layer(s)), write + attention, fp64"}


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    import synth
    oracle.set_num_threads(host_cores())  # the other ranks do no work: every core is rank 0's
    wl = synth.make(args.workload, seed=args.seed)
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    pick, sub = _oracle_sample(wl, per_step)
    vals = synth.make_values(sub)
    host = [{n: synth.to_storage_numpy(vals[n][l]).copy() for n in ("q", "k", "v", "k_cache", "v_cache")}
            for l in range(sub.num_layers)]
    for _ in range(args.warmup):
        _oracle_step_seconds(sub, host)
    secs = [_oracle_step_seconds(sub, host) for _ in range(args.steps)]
    b = synth.kv_bytes_read(sub) * sub.num_layers
    value = b * args.steps / sum(secs) / 1e9
    sample = (f"{len(pick)} of {wl.num_seqs} sequences ({int(sub.context_lens.sum())} context tokens"
              f" x {sub.num_layers} layer(s)) per step, write + attention, fp64")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(secs) / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "num_seqs": wl.num_seqs, "kv_dtype": wl.kv_dtype,
                   "sampled_seqs": len(pick), "seed": args.seed},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="longctx_b256")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="CPU-time budget of the oracle sample (cpu_baseline / reference arm)")
    ap.add_argument("--max-seqs", type=int, default=0,
                    help="keep only the first N sequences (small cases for profiler captures)")
    ap.add_argument("--partition", type=int, default=0,
                    help="override the workload's split-K partition size (tokens)")
    ap.add_argument("--kv-dtype", default="native", choices=["native", "fp8"],
                    help="fp8: E4M3 KV pools with per-head scales (bf16 workloads, head_dim 64/128)")
    ap.add_argument("--q-rope", default="none", choices=["none", "separate", "fused"],
                    help="also rotate the step's q rows: in their own launch, or inside the "
                         "cache-write launch (default: q arrives rotated)")
    ap.add_argument("--no-graph", action="store_true",
                    help="time direct launches instead of replays of a CUDA graph of the step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time only the selected workload (not the other configs beside it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
