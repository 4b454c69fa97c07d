"""Benchmark: paged decode HBM GB/s and chunked paged prefill TFLOP/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one rk_paged_attn_decode_balanced call over the decode-throughput
workload (B=64 rows, kv_len 4096 each, Hq=32/Hkv=8, d=128, page 16, 16384
shuffled pages; 1.075 GB of algorithmic traffic, larger than L2, so no flush is
needed between steps): the split-free decode on its balanced schedule, bitwise
identical to rk_paged_attn_decode, whose one-CTA-per-(row, KV head) launch is
timed beside it in "decode_one_cta_per_pair".  The same run also times rk_paged_attn_prefill on the chunked
prefill workload (B=4, 1536-token prefix + 512-token chunk) with an L2 flush
between launches, reported in the "prefill" object, the long full-causal
prefill (B=1, S=8192) in "prefill_long", the same decode step replayed from a
CUDA graph in "decode_graph", and the decode_long, kv_append, ragged-step and
prefill-backward objects.

Multi-GPU (torchrun, one rank per GPU): replicas only -- every rank runs its
own copy of the workload on its own GPU, there is no collective on the data
path; the barrier and the max-over-ranks of the timed region are the only
communication.  value = all ranks' bytes / max rank time ("scaling": "weak").

--impl reference times the float64 CPU oracle on the host cores on the same
workload, every step the whole decode-throughput batch (~0.75 s of 16 host
cores a step), with the same config object as this arm (the slow baseline
arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


# ------------------------------------------------------------ helpers ----

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def decode_step_config(w, step_bytes, world):
    """The config object of the decode step (both arms)."""
    return {"workload": w.name + " page=16 (16384 shuffled pages, fused RoPE, FP32 LSE)",
            "l2": "inputs larger than L2 (%.3f GB per step)" % (step_bytes / 1e9),
            "parallelism": "replicas x%d" % world if world > 1 else "single GPU"}


def decode_alg_bytes(w):
    """Algorithmic bytes of one decode launch: every visible K and V row once,
    Q, out, LSE and the metadata the kernel reads."""
    kv_tokens = int(w.kv_lens.clamp(min=0).sum())
    return (kv_tokens * w.Hkv * w.D * 2 * 2 + w.q.numel() * 2 * 2 + w.B * w.Hq * w.Sq * 4
            + w.block_table.numel() * 4 + w.B * 4 * 2)


def prefill_alg_flops(w):
    """4 * D * (visible query-key pairs) * Hq: QK^T and PV over causal-visible pairs."""
    pos = w.position_ids.long()
    kv = w.kv_lens.long()[:, None]
    vis = (pos + 1).clamp(min=0)
    vis = vis.where(vis < kv, kv)
    return 4.0 * w.D * float(vis.sum()) * w.Hq


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "deterministic_paged_kv_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel, src_hash):
    """Per-launch DRAM bytes from the committed ncu summary, if taken on this source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("source_hash") != src_hash:
        return None
    return d.get("dram_bytes_per_launch")


def max_over_ranks(value, world, device="cpu"):
    """Max of a per-rank float over all ranks (the slowest replica sets the time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step, steps, world, region_ms):
    """Units processed by all replicas per second over the (max) timed region."""
    return world * units_per_rank_step * steps / (region_ms * 1e-3)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# -------------------------------------------------------- CPU oracle -----

def cpu_baseline_decode(w, budget_s=15.0):
    """Time the float64 oracle on the whole decode batch (one call computes all
    rows, as in the reference arm, so the per-call conversion of the inputs is
    paid once per batch), repeated until about budget_s; then one batch on one
    host thread.  Returns GB/s of algorithmic bytes and what was run."""
    import oracle
    oracle.build()
    cores = oracle.max_threads()  # before the one-thread run below changes the OpenMP default
    step_bytes = decode_alg_bytes(w)
    n, t_total = 0, 0.0
    while n == 0 or t_total < budget_s:
        t0 = time.perf_counter()
        oracle.attention(w.q, w.k_cache, w.v_cache, w.block_table, w.kv_lens, w.position_ids,
                         w.rope_theta, w.rope_scale)
        t_total += time.perf_counter() - t0
        n += 1
    t0 = time.perf_counter()
    oracle.attention(w.q, w.k_cache, w.v_cache, w.block_table, w.kv_lens, w.position_ids,
                     w.rope_theta, w.rope_scale, threads=1)
    t1 = time.perf_counter() - t0
    return {"value": n * step_bytes / t_total / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": "the whole batch (%d rows, all 32 heads, kv_len 4096 each) %d times, %.1f s of float64 "
                      "oracle" % (w.B, n, t_total),
            "single_thread": {"value": step_bytes / t1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": "the whole batch once on one host thread, %.1f s" % t1}}


def run_reference(args):
    """--impl reference: the oracle arm (host cores), same metric and config."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from deterministic_paged_kv_gb300 import workloads
    oracle.build()
    w = workloads.decode_throughput()
    step_bytes = decode_alg_bytes(w)
    times = []
    for step in range(args.warmup + args.steps):
        # every step the whole batch: all 64 rows, all 32 query heads
        t0 = time.perf_counter()
        oracle.attention(w.q, w.k_cache, w.v_cache, w.block_table, w.kv_lens, w.position_ids,
                         w.rope_theta, w.rope_scale)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = step_bytes * len(times) / total / 1e9
    cores = oracle.max_threads()
    line = {
        "impl": "reference", "metric": "paged decode HBM GB/s", "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_step_config(w, step_bytes, 1),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "the whole batch (64 rows) every step, %d steps" % len(times)},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# -------------------------------------------------------------- ours -----

def time_launches(fn, n, stream, flush=None):
    """Per-launch CUDA-event durations (ms) on `stream`.  All n launches (and
    flushes) are queued before the first is waited for, so the GPU never sits
    between a start event and its kernel waiting for the host to issue the
    launch: the events time the kernels, not the host calls."""
    import torch
    pairs = []
    for _ in range(n):
        if flush is not None:
            flush.zero_()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        pairs.append((s, e))
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in pairs]


def time_prefill(args, w, dev, stream, world, tf_burst, peak_kind, n):
    """Time rk_paged_attn_prefill on workload `w` (L2 flushed between
    launches) and return its TFLOP/s object."""
    import torch

    from deterministic_paged_kv_gb300 import binding
    names = ("q", "k_cache", "v_cache", "block_table", "kv_lens", "position_ids")
    dp = {k: getattr(w, k).to(dev) for k in names}
    pp = binding.plan(w.B, w.Sq, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, w.block_table,
                      w.kv_lens, w.position_ids, w.rope_theta, w.rope_scale)
    pout = torch.empty_like(dp["q"])
    plse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)

    def pstep():
        binding.attn_prefill(pp, dp["q"], dp["k_cache"], dp["v_cache"], dp["block_table"],
                             dp["kv_lens"], dp["position_ids"], pout, plse, stream=stream)

    for _ in range(max(3, args.warmup)):
        pstep()
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > 129 MB L2
    pl = time_launches(pstep, n, stream, flush=flush)
    p_ms = sum(pl) / len(pl)
    pflops = prefill_alg_flops(w)
    pf_hash = source_hash("prefill.cu", "rk_device.cuh", "rk_internal.h")
    obj = {
        "metric": "paged prefill TFLOP/s", "value": world * pflops / (p_ms * 1e-3) / 1e12,
        "unit": "TFLOP/s", "ms_per_launch": p_ms, "launches": len(pl),
        "config": {"workload": w.name + " page=16", "l2": "flushed (256 MB write) between launches",
                   "flops": "4*D*visible_pairs*Hq = %.4g" % pflops},
        "roofline": {"bound": "tensor", "achieved": pflops / (p_ms * 1e-3) / 1e12, "peak": tf_burst,
                     "unit": "TFLOP/s", "traffic": traffic_for("prefill_kernel", pf_hash),
                     "kernel": "prefill_kernel", "peak_kind": peak_kind + " (bf16 dense, burst)"},
    }
    obj["roofline"]["frac"] = obj["roofline"]["achieved"] / tf_burst
    return obj


def measure_prefill(args, dev, stream, world, tf_burst, peak_kind):
    """The "prefill" object: the chunked-prefill workload."""
    from deterministic_paged_kv_gb300 import workloads
    return time_prefill(args, workloads.prefill_chunk(), dev, stream, world, tf_burst, peak_kind,
                        max(10, args.steps))


def measure_prefill_long(args, dev, stream, world, tf_burst, peak_kind):
    """The "prefill_long" object: B=1, S=8192 full causal prefill (~0.5 ms a launch)."""
    from deterministic_paged_kv_gb300 import workloads
    obj = time_prefill(args, workloads.prefill_long(), dev, stream, world, tf_burst, peak_kind,
                       max(5, min(args.steps, 20)))
    # this workload's own ncu capture (the prefill object's is the chunk's)
    obj["roofline"]["traffic"] = traffic_for("prefill_kernel_long",
                                             source_hash("prefill.cu", "rk_device.cuh", "rk_internal.h"))
    return obj


def measure_decode_graph(step, stream, n, step_bytes):
    """The decode step captured once in a CUDA graph and replayed n times
    back to back (inputs larger than L2): GB/s of the replays."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        step(s)  # warm the capture stream
        with torch.cuda.graph(g, stream=s):
            step(s)
    stream.wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for _ in range(n):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    return {"value": step_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_replay": ms, "replays": n,
            "note": "one decode launch captured in a CUDA graph, replayed back to back"}


def measure_backward(args, dev, stream, tf_burst, peak_kind):
    """Time rk_paged_attn_prefill_backward on the long full-causal prefill
    (B=1, S=8192; forward run once before timing for out / lse; L2 flushed
    between launches).  Algorithmic FLOPs: the five products of the attention
    gradient (scores, dP, dV, dK, dQ) over the causal-visible pairs,
    10 * D * pairs * Hq = 2.5 x the forward's."""
    import torch

    from deterministic_paged_kv_gb300 import binding, workloads
    names = ("q", "k_cache", "v_cache", "block_table", "kv_lens", "position_ids")
    w = workloads.prefill_long()
    d = {k: getattr(w, k).to(dev) for k in names}
    p = binding.plan(w.B, w.Sq, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, w.block_table, w.kv_lens,
                     w.position_ids, w.rope_theta, w.rope_scale)
    out = torch.empty_like(d["q"])
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    binding.attn_prefill(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                         d["position_ids"], out, lse, stream=stream)
    g = torch.Generator().manual_seed(1099)
    dout = torch.randn(w.q.shape, generator=g).to(torch.bfloat16).to(dev)
    dq = torch.empty(w.q.shape, dtype=torch.float32, device=dev)
    dk = torch.empty(w.k_cache.shape, dtype=torch.float32, device=dev)
    dv = torch.empty(w.v_cache.shape, dtype=torch.float32, device=dev)
    ws = torch.empty(binding.prefill_backward_workspace_bytes(p), dtype=torch.uint8, device=dev)

    def step():
        binding.attn_prefill_backward(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                                      d["position_ids"], out, lse, dout, dq, dk, dv, ws, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    t = time_launches(step, max(5, min(args.steps, 10)), stream, flush=flush)
    ms = sum(t) / len(t)
    flops = 2.5 * prefill_alg_flops(w)
    achieved = flops / (ms * 1e-3) / 1e12
    return {"metric": "paged prefill backward TFLOP/s", "value": achieved, "unit": "TFLOP/s",
            "ms_per_launch": ms, "launches": len(t),
            "config": {"workload": w.name + " page=16, backward (dq, dk, dv)",
                       "l2": "flushed (256 MB write) between launches",
                       "flops": "10*D*visible_pairs*Hq = %.4g" % flops},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": tf_burst, "unit": "TFLOP/s",
                         "frac": achieved / tf_burst,
                         "traffic": traffic_for("attn_bwd", source_hash("backward_tc.cu", "rk_device.cuh",
                                                                         "rk_internal.h")),
                         "traffic_note": "DRAM bytes of the dq and dk/dv launches of one call (the two "
                                         "rotation pre-passes not included)",
                         "kernel": "attn_bwd_dq_tc_kernel + attn_bwd_dkdv_tc_kernel (tcgen05)",
                         "peak_kind": peak_kind + " (bf16 dense, burst)"},
            "note": "four launches per call (rotation of q and K into the workspace, dq with delta, dk/dv); deterministic, no atomics"}


def measure_decode_long(args, dev, stream, hbm, peak_kind, splits=(1024, 1728, 2048)):
    """Time decode_long (B=1, kv 32768: 8 CTAs without splitting) through the
    split-free entry point and the fixed-split entry point at several split
    lengths (1728 tokens: 19 splits x 8 KV heads = 152 CTAs, one per SM); L2
    flushed between launches.  Returns the "decode_long" object with the best
    split named."""
    import torch

    from deterministic_paged_kv_gb300 import binding, workloads
    names = ("q", "k_cache", "v_cache", "block_table", "kv_lens", "position_ids")
    w = workloads.decode_long()
    d = {k: getattr(w, k).to(dev) for k in names}
    p = binding.plan(w.B, 1, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, w.block_table, w.kv_lens,
                     w.position_ids, w.rope_theta, w.rope_scale)
    out = torch.empty_like(d["q"])
    lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device=dev)
    scratch = torch.empty(max(binding.decode_split_scratch_bytes(p, n) for n in splits), dtype=torch.uint8,
                          device=dev)
    args_d = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"], d["position_ids"], out, lse)

    def free():
        binding.attn_decode(p, *args_d, stream=stream)

    def split_fn(n):
        return lambda: binding.attn_decode_split(p, n, *args_d, scratch, stream=stream)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    byt = decode_alg_bytes(w)
    res = {"config": {"workload": w.name + " page=16", "l2": "flushed (256 MB write) between launches",
                      "alg_bytes_per_launch": byt, "split_tokens": list(splits)}}
    for name, fn in [("split_free", free)] + [("split_%d" % n, split_fn(n)) for n in splits]:
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        t = time_launches(fn, 20, stream, flush=flush)
        ms = sum(t) / len(t)
        res[name] = {"value": byt / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_launch": ms,
                     "frac_of_peak": byt / (ms * 1e-3) / 1e9 / hbm, "peak_kind": peak_kind}
    res["best_split"] = max(("split_%d" % n for n in splits), key=lambda k: res[k]["value"])
    return res


def measure_append(args, dev, stream, hbm, peak_kind):
    """Time rk_paged_kv_append for the prefill-chunk shape (4 rows x 512 new
    tokens) and the decode-step shape (64 rows x 1 token).  Inputs larger than
    L2 instead of a flush: one CUDA graph holds a launch per distinct
    new-token buffer, enough of them that their K / V add up to more than the
    129 MB L2 (a write flush between launches would leave the L2 full of dirty
    lines that this small kernel then pays to write back), and the time of a
    replay is divided by its launches.  Bytes = new K and V read once and
    written once."""
    import torch

    from deterministic_paged_kv_gb300 import binding, workloads
    res = {}
    for name, w, n_new in (("prefill_chunk_append", workloads.prefill_chunk(), 512),
                           ("decode_step_append", workloads.decode_throughput(), 1)):
        p = binding.plan(w.B, 1, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, w.block_table, w.kv_lens,
                         w.kv_lens[:, None].clone(), w.rope_theta, w.rope_scale)
        kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
        g = torch.Generator().manual_seed(7)
        one = w.B * n_new * w.Hkv * w.D * 2 * 2  # bytes of one set of new K and V
        n_sets = min(32, max(2, -(-(192 << 20) // one)))  # a 64-token step's sets stay in L2: launch-bound
        k_new = torch.randn((n_sets, w.B, n_new, w.Hkv, w.D), generator=g).to(torch.bfloat16).to(dev)
        v_new = torch.randn((n_sets, w.B, n_new, w.Hkv, w.D), generator=g).to(torch.bfloat16).to(dev)
        bt, kl = w.block_table.to(dev), w.kv_lens.to(dev)
        for i in range(max(3, args.warmup)):
            binding.kv_append(p, n_new, k_new[i % n_sets], v_new[i % n_sets], bt, kl, kc, vc, stream=stream)
        torch.cuda.synchronize()
        # all n_sets launches in one CUDA graph, each on its own input set: the
        # graph runs them back to back (no per-launch host or graph overhead)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(n_sets):
                    binding.kv_append(p, n_new, k_new[i], v_new[i], bt, kl, kc, vc, stream=s)
        stream.wait_stream(s)
        g.replay()
        torch.cuda.synchronize()
        t = [x / n_sets for x in time_launches(g.replay, 5, torch.cuda.current_stream(dev))]
        ms = sum(t) / len(t)
        byt = 2 * 2 * w.B * n_new * w.Hkv * w.D * 2
        res[name] = {"rows": w.B, "new_tokens_per_row": n_new, "bytes_per_launch": byt, "ms_per_launch": ms,
                     "timing": "%d launches in one CUDA graph, back to back, each on its own input set "
                               "(%.1f MB of new K / V in all); time per launch" % (n_sets, n_sets * one / 1e6),
                     "value": byt / (ms * 1e-3) / 1e9, "unit": "GB/s", "frac_of_peak": byt / (ms * 1e-3) / 1e9 / hbm,
                     "peak_kind": peak_kind}
        del kc, vc, k_new, v_new, g
    return res


def measure_ragged(args, dev, stream):
    """Time one mixed serving step through rk_paged_attn_ragged: 60 decode rows
    (one query, kv 2048) and 4 prefill chunks (512 queries at 1536..2047) packed
    in one call; L2 flushed between launches."""
    import torch

    from deterministic_paged_kv_gb300 import binding, workloads
    q_lens = [1] * 60 + [512] * 4
    w = workloads.ragged_case(q_lens, [2048] * 64, seed=1007)
    q, ind, pos = workloads.pack_ragged(w)
    p, mq = binding.plan_ragged(w.B, q.shape[0], w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, ind, w.block_table,
                                w.kv_lens, pos, w.rope_theta, w.rope_scale)
    kc, vc, bt, kl = w.k_cache.to(dev), w.v_cache.to(dev), w.block_table.to(dev), w.kv_lens.to(dev)
    dq, dind, dpos = q.to(dev), ind.to(dev), pos.to(dev)
    out = torch.empty((q.shape[0], w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((q.shape[0], w.Hq), dtype=torch.float32, device=dev)

    def fn():
        binding.attn_ragged(p, mq, dind, dq, kc, vc, bt, kl, dpos, out, lse, stream=stream)

    for _ in range(max(3, args.warmup)):
        fn()
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    t = time_launches(fn, 20, stream, flush=flush)
    ms = sum(t) / len(t)

    def fn_dec():  # max_q_len 1: the decode launch alone (the chunk rows are left out)
        binding.attn_ragged(p, 1, dind, dq, kc, vc, bt, kl, dpos, out, lse, stream=stream)

    for _ in range(3):
        fn_dec()
    t = time_launches(fn_dec, 20, stream, flush=flush)
    ms_dec = sum(t) / len(t)
    dec_bytes = 60 * 2048 * w.Hkv * w.D * 2 * 2
    pf_flops = 4.0 * w.D * w.Hq * 4 * sum(1536 + s + 1 for s in range(512))
    return {"workload": "ragged step: 60 decode rows (kv 2048) + 4 prefill chunks (512 at 1536..2047)",
            "l2": "flushed (256 MB write) between launches", "ms_per_launch": ms,
            "decode_launch_alone_ms": ms_dec, "decode_rows_kv_bytes": dec_bytes, "prefill_rows_flops": pf_flops,
            "note": "one call, two launches (decode rows, prefill rows)"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    from deterministic_paged_kv_gb300 import binding, workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    binding.load()
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    hbm, tf_burst, tf_sust, peak_kind = peaks()
    names = ("q", "k_cache", "v_cache", "block_table", "kv_lens", "position_ids")
    if args.backward_only:
        bw = measure_backward(args, dev, stream, tf_burst, peak_kind)
        if rank == 0:
            print(json.dumps(bw))
        return 0
    if args.prefill_only or args.prefill_long_only:
        pf = (measure_prefill_long if args.prefill_long_only else measure_prefill)(args, dev, stream, world,
                                                                                 tf_burst, peak_kind)
        if rank == 0:
            print(json.dumps(pf))
        return 0

    # ---------------- decode: the step ----------------
    w = workloads.decode_throughput()
    d = {k: getattr(w, k).to(dev) for k in names}
    p = binding.plan(w.B, 1, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, w.block_table, w.kv_lens,
                     w.position_ids, w.rope_theta, w.rope_scale)
    out = torch.empty_like(d["q"])
    lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device=dev)

    calls = [0]  # rk_paged_attn_decode_balanced calls made; each launches one decode_bal_kernel
    scratch = torch.zeros(binding.decode_balanced_scratch_bytes(p), dtype=torch.uint8, device=dev)

    def step(st=None):
        binding.attn_decode_balanced(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                                     d["position_ids"], out, lse, scratch, stream=st or stream)
        calls[0] += 1

    def step_one_cta():
        binding.attn_decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                            d["position_ids"], out, lse, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    step_bytes = decode_alg_bytes(w)
    clk = ClockSampler(local).__enter__()
    if True:
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        calls0 = calls[0]
        for _ in range(args.steps):
            step()
        timed_launches = calls[0] - calls0  # one kernel per decode call, nothing else in the region
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        wall = time.perf_counter() - t0
    region_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    value = whole_job_rate(step_bytes, args.steps, world, region_ms) / 1e9
    per_launch = time_launches(step, max(10, args.steps), stream)
    avg_launch_ms = sum(per_launch) / len(per_launch)
    dec_hash = source_hash("decode.cu", "rk_device.cuh", "rk_internal.h")
    roof = {"bound": "hbm", "achieved": step_bytes / (avg_launch_ms * 1e-3) / 1e9, "peak": hbm,
            "unit": "GB/s", "traffic": traffic_for("decode_bal_kernel", dec_hash),
            "kernel": "decode_bal_kernel (balanced: one CTA per SM, Hkv chains, state hand-off)",
            "peak_kind": peak_kind + " (copy bandwidth, burst)", "alg_bytes_per_launch": step_bytes}
    roof["frac"] = roof["achieved"] / roof["peak"]
    for _ in range(3):
        step_one_cta()
    one_cta = time_launches(step_one_cta, max(10, args.steps), stream)
    one_ms = sum(one_cta) / len(one_cta)
    one_cta_obj = {"value": step_bytes / (one_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_launch": one_ms,
                   "frac_of_peak": step_bytes / (one_ms * 1e-3) / 1e9 / hbm, "peak_kind": peak_kind,
                   "traffic": traffic_for("decode_kernel", dec_hash),
                   "kernel": "decode_kernel (rk_paged_attn_decode: one CTA per (row, KV head), 512 CTAs)"}

    # ---------------- e2e: host buffers through the public API ----------------
    pinned = {k: getattr(w, k).pin_memory() for k in names}
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    def e2e_step(with_cache):
        for k in names:
            if with_cache or k not in ("k_cache", "v_cache"):
                d[k].copy_(pinned[k], non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    def e2e_measure(with_cache, n):
        for _ in range(2):
            e2e_step(with_cache)
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(n):
            e2e_step(with_cache)
        torch.cuda.synchronize()
        return (time.perf_counter() - t) / n

    n_e2e = max(3, min(args.steps, 10))
    t_full = e2e_measure(True, n_e2e) if not args.no_e2e else float("nan")
    t_res = e2e_measure(False, n_e2e) if not args.no_e2e else float("nan")
    h2d_full = sum(pinned[k].numel() * pinned[k].element_size() for k in names)
    h2d_res = sum(pinned[k].numel() * pinned[k].element_size() for k in names
                  if k not in ("k_cache", "v_cache"))
    d2h = h_out.numel() * 2 + h_lse.numel() * 4

    dgraph = measure_decode_graph(step, stream, max(10, args.steps), step_bytes)
    prefill = None if args.no_prefill else measure_prefill(args, dev, stream, world, tf_burst, peak_kind)
    plong = None if (args.no_prefill or args.no_long) else measure_prefill_long(args, dev, stream, world,
                                                                                tf_burst, peak_kind)
    dlong = None if args.no_long else measure_decode_long(args, dev, stream, hbm, peak_kind)
    append = None if args.no_long else measure_append(args, dev, stream, hbm, peak_kind)
    ragged = None if args.no_long else measure_ragged(args, dev, stream)
    backward = None if args.no_long else measure_backward(args, dev, stream, tf_burst, peak_kind)

    clk.__exit__(None, None, None)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_decode(w, budget_s=args.cpu_budget)

    clocks = clk.summary()
    if rank == 0:
        line = {
            "metric": "paged decode HBM GB/s", "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": region_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": decode_step_config(w, step_bytes, world),
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": world * step_bytes / t_full / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": h2d_full, "d2h_bytes_per_step": d2h,
                    "note": "every input incl. the 1 GB K/V cache copied from pinned host memory each step"},
            "e2e_resident_cache": {"value": world * step_bytes / t_res / 1e9, "unit": "GB/s",
                                   "h2d_bytes_per_step": h2d_res, "d2h_bytes_per_step": d2h,
                                   "note": "K/V cache resident in HBM; q and metadata copied each step"},
            "gpu_launches": timed_launches,
            "clocks": clocks,
            "wall_s_timed_region": wall,
            "decode_graph": dgraph,
            "decode_one_cta_per_pair": one_cta_obj,
            "prefill": prefill,
            "prefill_long": plong,
            "decode_long": dlong,
            "kv_append": append,
            "ragged_step": ragged,
            "prefill_backward": backward,
        }
        if args.no_e2e:
            line["e2e"] = line["e2e_resident_cache"] = None
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the decode_long (split-free vs fixed-split decode), kv_append and ragged_step objects")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill object (profiling runs of the decode kernel)")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only the prefill backward on the long full-causal workload")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prefill workload and print its object (profiling runs)")
    ap.add_argument("--prefill-long-only", action="store_true",
                    help="time only the long full-causal prefill and print its object (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
