#!/usr/bin/env python3
"""Benchmark of the decode-step attention core (slidingDecodeGQA / decodeGQA).

Metric: KV-read HBM bandwidth (GB/s) of `attn.core` calls -- algorithmic K and V
bytes (2 tensors x KVH x D x 2 B per attended position) divided by the device
time of the calls -- with the microseconds per layer call alongside.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole hot path over the workload's batch: one
library call (two for the paged mix: a sliding and a global call).  Inputs are
resident in HBM before timing; L2 is flushed (a write larger than L2) between
timed steps, outside the timed events.  Under torchrun each rank runs its own
replica of the workload on its own GPU (weak scaling, no collective on the data
path); rank 0 prints one JSON line with the max-over-ranks time.

`--impl reference` times the fp64 CPU oracle on the host cores over a bounded
sample of the same workload (the reference arm).
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from decode_attention_gb300 import inputs  # noqa: E402

DEFAULT_WORKLOAD = "paged_mixed_b256"
HBM_FALLBACK_GBS = 6800.0
PROFILES = os.path.join(ROOT, "profiles")
# the sources each main kernel is compiled from: a recorded DRAM traffic figure holds
# only while they hash to the value stored beside it
KERNEL_SOURCES = {
    "gqa_decode_kernel": [
        "decode_attention_gb300/csrc/kernels/decode_kernel.cuh",
        "decode_attention_gb300/csrc/kernels/policy_sliding_core.cuh",
        "decode_attention_gb300/csrc/kernels/policy_mma.cuh",
        "decode_attention_gb300/csrc/kernels/policy_mma_keqv.cuh",
        "decode_attention_gb300/csrc/kernels/ptx.cuh",
    ],
    "gqa_mq_kernel": [
        "decode_attention_gb300/csrc/kernels/decode_mq_kernel.cuh",
        "decode_attention_gb300/csrc/kernels/decode_kernel.cuh",
        "decode_attention_gb300/csrc/kernels/ptx.cuh",
    ],
}


# ---------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks only)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank scalar across all ranks (identity for one rank)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of rank r's replica: rank 0 runs the workload's own seed."""
    return int(base_seed) + 1000 * int(rank)


# ---------------------------------------------------------------------------
# workload construction and byte accounting
# ---------------------------------------------------------------------------

def attended_count(L: int, window: int, T: int = 1) -> int:
    """Positions a call reads for one sequence: the union of its T queries' ranges
    (query t at position L - T + t; the earliest window starts at L - T + 1 - window)."""
    span = window + T - 1 if window > 0 else 0
    lo = max(0, L - span) if span > 0 else 0
    return max(0, L - lo)


def kv_bytes(seq_lens, geo: dict, T: int = 1) -> int:
    """Algorithmic K+V bytes one call reads: KVH x D x 2 B x 2 tensors per attended position."""
    n = sum(attended_count(int(L), geo["window"], T) for L in np.asarray(seq_lens).tolist())
    return n * geo["KVH"] * geo["D"] * 2 * 2


class Call:
    """One library call of a step, with its inputs resident on the device."""

    def __init__(self, layer: str, geo: dict, case: dict, paged: bool, seq_lens: np.ndarray,
                 device="cuda", ring: int = 0, keqv: bool = False, raw: dict | None = None,
                 queries: int = 0):
        self.layer, self.geo, self.case, self.paged = layer, geo, case, paged
        self.queries = queries   # > 0: multi-query call with this many tokens per sequence
        self.ring = ring   # > 0: window-capped ring cache of `ring` rows
        self.keqv = keqv   # single K=V cache: only values are read
        self.raw = raw     # set: the decode-step producer writing into `case`, not a decode
        self.name = f"{layer}_ring{ring}" if ring else (f"{layer}_keqv" if keqv else layer)
        if queries:
            self.name = f"{layer}_mq{queries}"
        if raw is not None:
            self.name += "_producer"
        self.seq_lens = seq_lens
        # the producer reads no cache: it adds time, not KV bytes
        self.bytes = 0 if raw is not None else (
            kv_bytes(seq_lens, geo, max(1, queries)) // (2 if keqv else 1))
        self.times_ms = []
        if str(device).startswith("cuda"):
            B = len(seq_lens)
            shape = (B, queries, geo["H"], geo["D"]) if queries else (B, geo["H"], geo["D"])
            self.out = torch.empty(shape, dtype=torch.bfloat16, device=device)
            self.start = torch.cuda.Event(enable_timing=True)
            self.end = torch.cuda.Event(enable_timing=True)

    def launch(self, gqa, q=None, seq_lens=None):
        c = self.case
        q = c["q"] if q is None else q
        lens = c["seq_lens"] if seq_lens is None else seq_lens
        if self.raw is not None:
            r = self.raw
            gqa.gqa_prepare_decode(r["q_raw"], r["k_raw"], r["v_raw"], r["w_q"], r["w_k"], lens, q,
                                   c["k"], c["v"], ring=self.ring > 0)
        elif self.queries:
            gqa.gqa_decode_mq(q, c["k"], c["v"], lens, self.geo["window"], out=self.out)
        elif self.paged:
            gqa.gqa_decode_paged(q, c["k_pages"], c["v_pages"], c["block_table"], lens,
                                 self.geo["window"], out=self.out)
        elif self.ring:
            gqa.gqa_decode_ring(q, c["k"], c["v"], lens, self.geo["window"], out=self.out)
        elif self.keqv:
            gqa.gqa_decode_keqv(q, c["v"], c["w_k"], lens, out=self.out)
        else:
            gqa.gqa_decode(q, c["k"], c["v"], lens, self.geo["window"], out=self.out)


def build_calls(wl: inputs.Workload, seed: int, device="cuda"):
    lens = wl.lengths(np.random.default_rng(seed))
    calls = []
    if wl.paged:
        table = inputs.page_table(lens, seed, max_pages=(wl.S + 15) // 16)
        for i, layer in enumerate(wl.layers):
            geo = inputs.geometry(layer)
            case = inputs.paged_case(wl.B, geo["H"], geo["KVH"], geo["D"], lens, seed + 100 * i,
                                     device=device, table=table)
            calls.append(Call(layer, geo, case, True, lens, device))
    elif wl.queries:
        geo = inputs.geometry(wl.layers[0])
        case = inputs.mq_case(wl.B, wl.queries, wl.S, geo["H"], geo["KVH"], geo["D"], lens, seed,
                              device=device)
        calls.append(Call(wl.layers[0], geo, case, False, lens, device, queries=wl.queries))
    elif wl.keqv:
        geo = inputs.geometry(wl.layers[0])
        case = inputs.keqv_case(wl.B, wl.S, geo["H"], geo["KVH"], geo["D"], lens, seed,
                                device=device)
        calls.append(Call(wl.layers[0], geo, case, False, lens, device, keqv=True))
    elif wl.rings:
        for i, window in enumerate(wl.rings):
            geo = dict(inputs.geometry(wl.layers[0]), window=window)
            case = inputs.contiguous_case(wl.B, window, geo["H"], geo["KVH"], geo["D"], lens,
                                          seed + 100 * i, device=device)
            if wl.step:
                raw = inputs.raw_projections(wl.B, geo["H"], geo["KVH"], geo["D"], seed + 100 * i,
                                             device=device)
                calls.append(Call(wl.layers[0], geo, case, False, lens, device, ring=window,
                                  raw=raw))
            calls.append(Call(wl.layers[0], geo, case, False, lens, device, ring=window))
    else:
        layer = wl.layers[0]
        geo = inputs.geometry(layer)
        case = inputs.contiguous_case(wl.B, wl.S, geo["H"], geo["KVH"], geo["D"], lens, seed,
                                      device=device)
        calls.append(Call(layer, geo, case, False, lens, device))
    return calls, lens


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi in loop mode (20 ms) for the lifetime of the object."""

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            sel = []
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        return rows


def clock_summary(rows, t0: float, t1: float):
    """Samples whose timestamps fall in [t0, t1] (host clock), else the nearest ones."""
    def ts(r):
        try:
            return datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return 0.0
    inside = [r for r in rows if t0 - 0.05 <= ts(r) <= t1 + 0.05]
    used = inside or sorted(rows, key=lambda r: min(abs(ts(r) - t0), abs(ts(r) - t1)))[:3]
    if not used:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                "samples": 0}
    sm = [float(r[1]) for r in used if r[1].replace(".", "").isdigit()]
    mx = [float(r[2]) for r in used if r[2].replace(".", "").isdigit()]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in used for i in range(4) if r[5 + i].lower() == "active"})
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons, "samples": len(used), "samples_inside_timed_region": len(inside)}


# ---------------------------------------------------------------------------
# roofline helpers
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def main_kernel(gqa, call) -> str:
    """The kernel a call's positions stream through: multi-query calls with T >= 2 run
    on the tcgen05 kernel; a K=V call runs where the library says it does."""
    if call.queries > 1:
        return "gqa_mq_kernel"
    if call.keqv:
        cap = call.case["v"].shape[1]   # K=V calls here are contiguous
        choice = gqa.gqa_decode_keqv_kernel(len(call.seq_lens), cap, call.geo["H"],
                                            call.geo["KVH"], call.geo["D"])
        if choice == gqa.GQA_KERNEL_TCGEN05:
            return "gqa_mq_kernel"
    return "gqa_decode_kernel"


def launches_per_call(gqa, call) -> int:
    """Kernels one call launches: the producer 1; a slidingDecodeGQA decode 1 (split
    segments merge in the main kernel); a decodeGQA decode 2 (main and combine kernels);
    a K=V call on the tcgen05 kernel 3 (the scores-operand kernel first)."""
    if call.raw is not None:
        return 1
    kernel = main_kernel(gqa, call)
    if kernel == "gqa_mq_kernel":
        return 3 if call.keqv else 2
    return 1 if call.layer == "sliding" else 2


def recorded_traffic(workload: str, layer: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(PROFILES, "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    entry = rec.get(workload, {}).get(layer)
    if not entry or entry.get("kernel") != kernel or \
            entry.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    return entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

def host_slices(call: Call, b: int):
    """uint16 host copies of the attended rows of sequence b (and pos_base); for a
    ring cache, the sequence's whole ring (it holds exactly its window's rows)."""
    c, geo = call.case, call.geo
    L = int(call.seq_lens[b])
    lo = max(0, L - geo["window"]) if geo["window"] > 0 else 0
    qb = inputs.bf16_bits(c["q"][b:b + 1])
    if call.queries:
        # the union of the queries' ranges, shifted to start at row 0: the masks
        # depend only on positions relative to L, so the result is unchanged
        n = attended_count(L, geo["window"], call.queries)
        return (qb, inputs.bf16_bits(c["k"][b:b + 1, L - n:L]),
                inputs.bf16_bits(c["v"][b:b + 1, L - n:L]), n, 0)
    if call.ring:
        return qb, inputs.bf16_bits(c["k"][b:b + 1]), inputs.bf16_bits(c["v"][b:b + 1]), L, 0
    if call.keqv:
        # the oracle reads rows [0, L) of the value cache and the weight
        return qb, inputs.bf16_bits(c["w_k"]), inputs.bf16_bits(c["v"][b:b + 1, :L]), L, 0
    if call.paged:
        pages = c["block_table"][b, lo // 16:(L + 15) // 16].long()
        k = c["k_pages"][pages].reshape(1, -1, geo["KVH"], geo["D"])
        v = c["v_pages"][pages].reshape(1, -1, geo["KVH"], geo["D"])
        base = (lo // 16) * 16
    else:
        k = c["k"][b:b + 1, lo:L]
        v = c["v"][b:b + 1, lo:L]
        base = lo
    return qb, inputs.bf16_bits(k), inputs.bf16_bits(v), L, base


def oracle_sample(calls, budget_s: float, max_seqs: int | None = None):
    """Prepare host slices for the oracle, sequence by sequence, for ~budget_s of CPU work."""
    import oracle
    oracle.build()
    # estimated oracle rate: ~0.5 GFLOP/s per thread of fp64 scalar work
    rate = 0.5e9 * oracle.default_threads()
    items, est = [], 0.0
    order = [(ci, b) for b in range(len(calls[0].seq_lens)) for ci in range(len(calls))]
    for ci, b in order:
        call = calls[ci]
        n = attended_count(int(call.seq_lens[b]), call.geo["window"], max(1, call.queries))
        if n == 0 or call.raw is not None:   # the producer has no attention to sample
            continue
        flops = 4.0 * n * call.geo["H"] * call.geo["D"] * max(1, call.queries)
        if call.keqv:
            flops *= 5.0   # plus a pow, cos and sin per rotated pair of every derived key
        if items and est + flops / rate > budget_s:
            break
        items.append((call, b, host_slices(call, b),
                      n * call.geo["KVH"] * call.geo["D"] * (2 if call.keqv else 4)))
        est += flops / rate
        if max_seqs and len(items) >= max_seqs:
            break
    return items


def oracle_for(call: Call, slices):
    """The fp64 oracle's output [H, D] for one sequence, from host_slices()."""
    import oracle
    qb, kb, vb, L, base = slices
    if call.queries:
        return oracle.gqa_decode_mq_f64(qb, kb, vb, [L], call.geo["window"])[0]
    if call.ring:
        return oracle.gqa_decode_ring_f64(qb, kb, vb, [L], call.geo["window"])[0]
    if call.keqv:
        return oracle.gqa_decode_keqv_f64(qb, vb, kb, [L], 0)[0]   # kb holds w_k
    return oracle.gqa_decode_f64(qb, kb, vb, [L], call.geo["window"], pos_base=base)[0]


def run_oracle_items(items):
    t0 = time.perf_counter()
    nbytes = 0
    for call, b, slices, nb in items:
        oracle_for(call, slices)
        nbytes += nb
    return nbytes, time.perf_counter() - t0


def describe_sample(items, calls, repeats=1):
    seqs = len(items)
    total = sum(1 for c in calls if c.raw is None
                for L in c.seq_lens if attended_count(int(L), c.geo["window"]) > 0)
    return (f"{seqs} of {total} (sequence, call) pairs of the workload, in batch order"
            + (f", repeated {repeats}x" if repeats > 1 else "") + "; fp64 oracle, all heads")


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    device = "cuda" if torch.cuda.is_available() else "cpu"
    calls, _ = build_calls(wl, wl.seed, device=device)
    items = oracle_sample(calls, budget_s=2.0)
    for _ in range(args.warmup):
        run_oracle_items(items)
    tot_b, tot_t = 0, 0.0
    for _ in range(args.steps):
        nb, dt = run_oracle_items(items)
        tot_b += nb
        tot_t += dt
    value = tot_b / tot_t / 1e9
    cores = oracle.default_threads()
    line = {
        "impl": "reference",
        "metric": "decode-attn KV-read HBM GB/s (and us/layer)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": describe_sample(items, calls)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# How the timed GPU steps treat L2 (both arms print the same config)
L2_POLICY = "GPU steps: L2 flushed between timed steps by a write larger than L2"


def workload_config(wl):
    if wl.rings:
        geo = [dict(layer=wl.layers[0], **dict(inputs.geometry(wl.layers[0]), window=w), ring=w)
               for w in wl.rings]
    else:
        geo = [dict(layer=l, **{k: v for k, v in inputs.geometry(l).items()}) for l in wl.layers]
    cfg = {"workload": wl.name, "description": wl.description, "B": wl.B, "S": wl.S,
           "seed": wl.seed, "paged": wl.paged, "page_size": 16 if wl.paged else None,
           "geometry": geo}
    if wl.step:
        cfg["producer"] = "q/k/v norms, rope and the ring append run ahead of each attention call"
    cfg["l2"] = L2_POLICY
    return cfg


def run_ours(args, wl):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    import decode_attention_gb300 as gqa
    gqa.load_library()
    dev = torch.device("cuda", local)

    seed = rank_seed(wl.seed, rank)
    calls, lens = build_calls(wl, seed)
    torch.cuda.synchronize()

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # one untimed pass to load the kernels and check the status word
    for c in calls:
        c.launch(gqa)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0, "device status word raised during the first pass"

    # ---- warm-up, then the timed region, back to back on the device ----
    # The clock sampler starts first.  The W warm-up steps (with the same L2
    # flushes) run right before the K timed steps, so the GPU does not idle and
    # drop its clocks in between.  Everything is enqueued before one synchronize,
    # behind a ~1 ms spin on the GPU, so the host is ahead of the GPU from the first
    # step on and no host-side launch latency falls between a pair of events.
    events = {id(c): [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(args.steps)] for c in calls}
    sampler = ClockSampler(local)
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    torch.cuda._sleep(2_000_000)   # clock cycles
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        for c in calls:
            c.launch(gqa)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        for c in calls:
            ev = events[id(c)][i]
            ev[0].record(stream)
            c.launch(gqa)
            ev[1].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    for c in calls:
        c.times_ms = [a.elapsed_time(b) for a, b in events[id(c)]]
        print(f"[bench] {c.name} us per step: " + " ".join(f"{t * 1e3:.1f}" for t in c.times_ms),
              file=sys.stderr)
    barrier(world)
    time.sleep(0.1)
    clock_rows = sampler.stop()
    status = gqa.gqa_device_status()

    step_ms_rank = sum(sum(c.times_ms) for c in calls)
    bytes_rank = sum(c.bytes for c in calls) * args.steps
    t_max_ms = max_over_ranks(step_ms_rank, world, dev)
    bytes_all = sum_over_ranks(bytes_rank, world, dev)
    value = bytes_all / (t_max_ms * 1e-3) / 1e9

    # ---- the launch floor: an empty kernel timed the same way (after the same L2
    # flush, CUDA events on the same stream); no call can measure below it ----
    floor_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.warmup + args.steps)]
    torch.cuda._sleep(2_000_000)
    for i, (a, b) in enumerate(floor_ev):
        flush.fill_(i & 0xFF)
        a.record(stream)
        torch.cuda._sleep(0)
        b.record(stream)
    torch.cuda.synchronize()
    launch_floor_us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in floor_ev[args.warmup:])

    # ---- end to end through the public API: pinned host inputs in, o out ----
    # A decode call takes q and seq_lens from the host and returns o.  In a step
    # workload the producer takes the raw projections and seq_lens from the host
    # and writes q (and the new cache row) on the device; the decode call behind it
    # reads that q and returns o.
    h2d = d2h = 0
    plans = []
    for ci, c in enumerate(calls):
        fed = ci > 0 and calls[ci - 1].raw is not None   # q comes from the producer
        host = {}
        if c.raw is not None:
            for key in ("q_raw", "k_raw", "v_raw"):
                host[key] = (c.raw[key].cpu().pin_memory(), torch.empty_like(c.raw[key]))
        elif not fed:
            host["q"] = (c.case["q"].cpu().pin_memory(), torch.empty_like(c.case["q"]))
        if not fed:
            host["seq_lens"] = (c.case["seq_lens"].cpu().pin_memory(),
                                torch.empty_like(c.case["seq_lens"]))
        for h, _ in host.values():
            h2d += h.numel() * h.element_size()
        ho = None
        if c.raw is None:
            ho = torch.empty(c.out.shape, dtype=c.out.dtype).pin_memory()
            d2h += ho.numel() * ho.element_size()
        plans.append((c, host, ho))
    n_e2e = args.warmup + args.steps
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_e2e)]
    for i in range(n_e2e):
        flush.fill_(i & 0xFF)
        e2e_ev[i][0].record(stream)
        lens_dev = None
        for c, host, ho in plans:
            for h, d in host.values():
                d.copy_(h, non_blocking=True)
            if "seq_lens" in host:
                lens_dev = host["seq_lens"][1]
            if c.raw is not None:
                r = {k: host[k][1] for k in ("q_raw", "k_raw", "v_raw")}
                gqa.gqa_prepare_decode(r["q_raw"], r["k_raw"], r["v_raw"], c.raw["w_q"],
                                       c.raw["w_k"], lens_dev, c.case["q"], c.case["k"],
                                       c.case["v"], ring=c.ring > 0)
            else:
                q_in = host["q"][1] if "q" in host else c.case["q"]
                c.launch(gqa, q=q_in, seq_lens=lens_dev)
                ho.copy_(c.out, non_blocking=True)
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_ev[args.warmup:])
    e2e_max = max_over_ranks(e2e_ms, world, dev)
    e2e_value = bytes_all / (e2e_max * 1e-3) / 1e9

    # ---- roofline of the dominant kernel (the call moving the most bytes) ----
    dom = max(calls, key=lambda c: c.bytes)
    dom_ms = statistics.mean(dom.times_ms)
    achieved = dom.bytes / (dom_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    kernel = main_kernel(gqa, dom)
    roofline = {"bound": "hbm", "kernel": f"{kernel}<{dom.name}>",
                "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_kind,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": recorded_traffic(wl.name, dom.layer, kernel),
                "algorithmic_bytes_per_launch": dom.bytes}

    us_per_layer = {c.name: round(statistics.median(c.times_ms) * 1e3, 2) for c in calls}
    if wl.rings:
        us_per_layer["block_of_ring_calls"] = round(sum(us_per_layer[c.name] for c in calls), 2)
    if len(calls) == 2 and {c.layer for c in calls} == {"sliding", "global"}:
        us_per_layer["weighted_50_sliding_10_global"] = round(
            (50 * us_per_layer["sliding"] + 10 * us_per_layer["global"]) / 60, 2)
    pct = {c.name: [round(float(np.percentile(c.times_ms, p)) * 1e3, 2) for p in (10, 50, 90)]
           for c in calls}

    if rank != 0:
        return 0
    line = {
        "metric": "decode-attn KV-read HBM GB/s (and us/layer)",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "storage_dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl),
        "l2_flush": {"bytes": flush.numel(), "l2_bytes": l2},
        "us_per_layer": us_per_layer, "us_p10_p50_p90": pct,
        "launch_floor_us": round(launch_floor_us, 2),
        "kv_bytes_per_step": sum(c.bytes for c in calls),
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * sum(launches_per_call(gqa, c) for c in calls),
        "clocks": clock_summary(clock_rows, t_wall0, t_wall1),
        "device_status": status,
    }
    if not args.no_cpu_baseline and world == 1:
        items = oracle_sample(calls, budget_s=args.cpu_budget)
        nb, dt = run_oracle_items(items)
        reps = 1
        # repeat the sample until about cpu_budget seconds of oracle work are timed
        while dt < args.cpu_budget and reps < 100000:
            nb2, dt2 = run_oracle_items(items)
            nb, dt, reps = nb + nb2, dt + dt2, reps + 1
        import oracle
        line["cpu_baseline"] = {"value": round(nb / dt / 1e9, 4), "unit": "GB/s",
                                "cores": oracle.default_threads(), "kind": "oracle",
                                "sample": describe_sample(items, calls, reps),
                                "seconds": round(dt, 2)}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline leg")
    args = ap.parse_args(argv)
    wl = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
