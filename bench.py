#!/usr/bin/env python3
"""Benchmark of the CP token-layout and owner-gradient-return hot path.

One step = one pass of the whole path over one batch at the pages' training
shape (CP=4, S=262144 tokens as one causal document, 20 heads x 128, bf16;
"Add stream-ordered CP gradient return primitive", TransformerEngine PR 3235,
"Validation"):
  1. plan: ownership map l2g/g2l and rank-local metadata (2 kernels),
  2. partition: Q, K and V [S,20,128] into rank-local order (1 kernel),
  3. grad_return: P=4 writers' global dK and dV [4,S,20,128] summed into the
     owners' [4,S/4,20,128] in one fused launch (1 kernel).
Inputs are resident in HBM when the timed region starts; a step touches
~21.5 GB, far above the 129 MB L2, so no flush is needed between steps.

value = algorithmic bytes of all steps of all ranks / max-over-ranks time.
Prints ONE JSON line on rank 0. ``--impl reference`` times the CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "grad_return effective HBM GB/s and % of peak (S=262144,P=4); partition tok/s"
P, D = 4, 128
S, H = 262144, 20  # the pages' shape; --tokens / --heads select a smaller case
FALLBACK_HBM_GBS = 6800.0


def workload() -> str:
    return (f"{'pages-shaped ' if (S, H) == (262144, 20) else ''}CP=4 step: S={S} single causal "
            f"document, {H}x{D} bf16, DualChunkSwap")


# Algorithmic bytes (what the method must move), per unit:
#   grad_return, per owner token (both tensors): 2 x (P reads + 1 write) rows
#     + 2 int32 index reads
#   partition, per token (three tensors): 3 x (1 read + 1 write) rows
#     + 3 int32 index reads
#   plan, per token: l2g and g2l int32 writes
def row_bytes() -> int:
    return H * D * 2


PATH = "fused"


def gr_bytes_per_token() -> int:
    if PATH == "staged":
        # per token and tensor: P writers read and write their row into a slot,
        # then the owner reads P slot rows and writes one; plus P index reads
        return 2 * ((3 * P + 1) * row_bytes() + P * 4)
    return 2 * (P + 1) * row_bytes() + 2 * 4


def part_bytes_per_token() -> int:
    return 3 * 2 * row_bytes() + 3 * 4


PLAN_BYTES_PER_TOKEN = 2 * 4


def step_bytes(tokens: int) -> int:
    return tokens * (gr_bytes_per_token() + part_bytes_per_token() + PLAN_BYTES_PER_TOKEN)


def host_mem_available():
    """MemAvailable of this host in bytes, or None where /proc/meminfo is absent."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _device_code(text: str) -> str:
    """The parts of a .cu file that decide what its kernels do: every
    `constexpr` line and every `__global__` function (from its template line
    through its closing brace). Host launch code is left out, so an edit
    there does not invalidate a traffic record."""
    import re

    parts = [line for line in text.splitlines() if line.lstrip().startswith("constexpr ")]
    for m in re.finditer(r"(?m)^(template <[^\n]*>\n)?__global__", text):
        start = m.start()
        i = text.index("{", m.end())
        depth = 0
        for j in range(i, len(text)):
            if text[j] == "{":
                depth += 1
            elif text[j] == "}":
                depth -= 1
                if depth == 0:
                    parts.append(text[start:j + 1])
                    break
    return "\n".join(parts)


def kernel_source_hash() -> str:
    """Hash of the gradient-return kernels' device code (all of
    cpt_device.cuh, the kernels and constants of grad_return.cu)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "context_attention_token_gb300", "csrc")
    with open(os.path.join(csrc, "cpt_device.cuh")) as f:
        h.update(f.read().encode())
    with open(os.path.join(csrc, "grad_return.cu")) as f:
        h.update(_device_code(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, units: int):
    """(DRAM bytes per launch, how they were obtained), scaled from the
    committed ncu summary by the units the launch processes; (None, reason)
    when the summary is missing or was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    k, v = line.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_hash") != kernel_source_hash():
            return None, "kernel source changed since the ncu capture"
        per_unit = float(kv["dram_bytes_per_unit"])
        note = (f"ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch at "
                f"{kv.get('captured_at', 'the recorded case')}, {per_unit:.1f} B per {kv.get('unit', 'unit')}, "
                f"x {units} units")
        return int(per_unit * units), note
    except (OSError, KeyError, ValueError):
        return None, "no ncu record"


# ---------------------------------------------------------------- ranks

def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks of the default process group (the value
    itself without one). Timing uses it so that the slowest replica sets the
    whole-job time."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """GB/s of the whole job: every replica's bytes over the slowest replica's time."""
    return bytes_per_step * steps * world / (max_ms / 1e3) / 1e9


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []  # (t, sm, smmax, reasons set)
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smmax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = []
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                "sw_power_cap"), parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.append(name)
            self.samples.append((time.time(), sm, smmax, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        used = inside if inside else self.samples
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({r for s in used for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in used),
                "sm_max_mhz": max(s[2] for s in used), "reasons": reasons,
                "samples": len(used), "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------- oracle arm

def oracle_sample_step_factory(tokens: int):
    """One oracle pass of the whole path on `tokens` tokens of the workload
    (same P, heads, head_dim and layout; a single causal document)."""
    import numpy as np

    import oracle
    from context_attention_token_gb300 import synth

    cu = np.array([0, tokens], np.int32)
    qkv = [synth.normal_bf16(synth.rng_for(3, t), (tokens, H, D)) for t in range(3)]
    dk = [synth.normal_bf16(synth.rng_for(3, 10 + w), (tokens, H, D), 0.02) for w in range(P)]
    dv = [synth.normal_bf16(synth.rng_for(3, 20 + w), (tokens, H, D), 0.02) for w in range(P)]

    def step():
        l2g, _g2l = oracle.index_map(oracle.LAYOUT_DSC, P, cu, tokens)
        oracle.thd_metadata(oracle.LAYOUT_DSC, P, cu, tokens)
        for x in qkv:
            oracle.partition(l2g, x)
        oracle.grad_return(l2g, dk, oracle.BF16)
        oracle.grad_return(l2g, dv, oracle.BF16)

    return step


def _oracle_replica(tokens, heads, mode, count, budget_s, barrier, results):
    """One process of the all-cores oracle timing (spawned; module globals
    are the defaults there, so the head count comes in as an argument).

    mode "budget": after the common start, run passes until budget_s has
    passed and report (passes, seconds). mode "steps": run `count` passes,
    each started by a barrier that the parent also joins, so the parent
    times whole steps across all replicas."""
    global H
    H = heads
    step = oracle_sample_step_factory(tokens)
    step()  # page in the inputs
    if mode == "budget":
        barrier.wait()
        reps, t0 = 0, time.perf_counter()
        while True:
            step()
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s:
                break
        results.put((reps, dt))
    else:
        for _ in range(count):
            barrier.wait(timeout=600)
            step()
        barrier.wait(timeout=600)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def replica_count(tokens: int, want: int) -> int:
    """Cores to use, capped so that the replicas' inputs and outputs (about
    16 rows of every token each) stay under a quarter of host memory."""
    per = 16 * tokens * row_bytes()
    try:
        mem = os.sysconf("SC_PHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        mem = 0
    cap = max(1, int(0.25 * mem // per)) if mem else 1
    return max(1, min(want, cap))


def _spawn_replicas(n, tokens, mode, count, budget_s, parties):
    import multiprocessing as mp

    import oracle

    oracle.build()  # once here, not in every replica
    ctx = mp.get_context("spawn")  # never fork a process that holds a CUDA context
    barrier = ctx.Barrier(parties)
    results = ctx.Queue()
    procs = [ctx.Process(target=_oracle_replica, args=(tokens, H, mode, count, budget_s, barrier, results),
                         daemon=True) for _ in range(n)]
    for pr in procs:
        pr.start()
    return procs, barrier, results


def oracle_all_cores(tokens: int, budget_s: float, cores: int):
    """The unmodified oracle on `cores` host cores at once: independent
    single-threaded replicas of the same sample, each in its own process.
    value = bytes of all passes of all replicas / the longest replica time."""
    procs, _barrier, results = _spawn_replicas(cores, tokens, "budget", 0, budget_s, cores)
    # (_barrier stays bound until the replicas are joined, for the same reason)
    got = [results.get(timeout=600) for _ in procs]
    for pr in procs:
        pr.join(timeout=60)
    reps = sum(r for r, _ in got)
    dt = max(t for _, t in got)
    return {"value": step_bytes(tokens) * reps / dt / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": (f"{cores} single-threaded oracle replicas in parallel, {reps} passes in all "
                       f"of the whole path over {tokens} of {S} tokens (same P=4, {H}x{D} bf16 "
                       f"single document), {dt:.1f} s")}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cores = args.reference_cores or host_cores()
    tokens = args.sample_tokens
    if not args.fixed_sample:
        # size the sample so the whole run takes about args.reference_budget
        # seconds: time one pass on a small slice, scale per token, round
        # down to a power of two (a multiple of 2P, as the layout requires)
        probe = 2048
        probe_step = oracle_sample_step_factory(probe)
        probe_step()
        t0 = time.perf_counter()
        probe_step()
        per_token = (time.perf_counter() - t0) / probe
        fit = args.reference_budget / ((args.steps + args.warmup) * per_token)
        tokens = 256
        while tokens * 2 <= min(fit, args.sample_tokens):
            tokens *= 2
    cores = replica_count(tokens, cores)
    # every step: each of `cores` replicas makes one oracle pass over its
    # sample; the parent joins the barrier that starts each step
    # keep the queue bound: collecting it unlinks semaphores the children still need
    procs, barrier, _results = _spawn_replicas(cores, tokens, "steps", args.warmup + args.steps,
                                               0.0, cores + 1)
    for _ in range(args.warmup):
        barrier.wait(timeout=600)
    barrier.wait(timeout=600)
    t0 = time.perf_counter()
    for _ in range(args.steps - 1):
        barrier.wait(timeout=600)
    barrier.wait(timeout=600)
    dt = time.perf_counter() - t0
    for pr in procs:
        pr.join(timeout=60)
    value = step_bytes(tokens) * cores * args.steps / dt / 1e9
    sample = (f"{cores} x {tokens} of {S} tokens per step: {cores} single-threaded oracle replicas "
              f"in parallel, each over the same P=4, {H}x{D} bf16 single document; whole path: "
              f"maps, metadata, 3-tensor partition, dK+dV grad_return")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload(), "P": P, "S": S, "H": H, "D": D, "sample_tokens": tokens,
                   "replicas": cores},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def cpu_baseline(tokens: int, budget_s: float, cores: int = 0):
    """The oracle on one core, then (cores > 1) on `cores` cores at once.
    The all-cores figure is the line's baseline; the one-core one rides along."""
    step = oracle_sample_step_factory(tokens)
    step()  # warm caches and page in the inputs
    reps, t0 = 0, time.perf_counter()
    while True:
        step()
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    one = {"value": step_bytes(tokens) * reps / dt / 1e9, "unit": "GB/s", "cores": 1,
           "kind": "oracle",
           "sample": (f"{reps} oracle passes of the whole path over {tokens} of {S} tokens "
                      f"(same P=4, {H}x{D} bf16 single document), {dt:.1f} s single-threaded")}
    cores = replica_count(tokens, cores)
    if cores <= 1:
        return one
    out = oracle_all_cores(tokens, budget_s, cores)
    out["single_core"] = one
    return out


# ---------------------------------------------------------------- GPU arm

def copy_ceiling_gbs(dev, stream) -> float:
    """A plain device-to-device copy timed in the same run, as a practical
    ceiling beside the recorded peak: 1 Gi bf16 elements (2 GiB read + 2 GiB
    written), CUDA events on the launching stream, best of 10 after 3."""
    import torch

    a = torch.ones(1 << 30, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    best = float("inf")
    for i in range(13):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        b.copy_(a)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            best = min(best, e0.elapsed_time(e1))
    del a, b
    return 2 * (1 << 30) * 2 / (best / 1e3) / 1e9


def _events_ms(fn, stream, reps, warm, before=None):
    """Median CUDA-event time of fn() on `stream` over `reps` launches after
    `warm`; `before` (e.g. an L2 flush) runs outside each timed interval."""
    import torch

    for _ in range(warm):
        if before is not None:
            before()
        fn()
    evs = []
    for _ in range(reps):
        if before is not None:
            before()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


# Shapes tried for each mix ceiling: (block bytes, stages, CTAs per SM).
CEILING_SHAPES = {
    "read4_write1": [(10240, 4, 1), (8192, 4, 1), (12288, 4, 1), (5120, 4, 2), (5120, 8, 1), (16384, 3, 1)],
    "read1_write1": [(32768, 4, 1), (40960, 4, 1), (16384, 4, 2), (8192, 4, 2), (32768, 3, 1), (24576, 8, 1)],
    "read8_write1": [(4096, 4, 1), (8192, 3, 1), (4096, 6, 1), (2048, 4, 2), (3072, 8, 1)],
}


def mix_ceilings(cpt, srcs4, dst4, src1, dst1, stream, reps=10, warm=3):
    """The fastest of a few bulk-copy shapes that move each call's read/write
    mix with no arithmetic (cpt_stream_ceiling): 4 reads : 1 write (the
    gradient return at P=4) and 1 : 1 (the row gather). GB/s counts read +
    written bytes, like the kernels' algorithmic bytes."""
    out = {}
    for name, srcs, dst in (("read4_write1", srcs4, dst4), ("read1_write1", [src1], dst1)):
        nbytes = dst.numel() * dst.element_size()
        moved = (len(srcs) + 1) * nbytes
        tried = []
        for blk, stages, ctas in CEILING_SHAPES[name]:
            ms = _events_ms(lambda: cpt.cpt_stream_ceiling(srcs, dst, blk, stages, ctas), stream, reps, warm)
            tried.append((moved / (ms / 1e3) / 1e9, ms, blk, stages, ctas))
        best = max(tried)
        out[name] = {"gbs": best[0], "ms": best[1], "bytes": moved,
                     "shape": {"block_bytes": best[2], "stages": best[3], "ctas_per_sm": best[4]},
                     "tried_gbs": [round(t[0], 1) for t in tried]}
    return out


def staged_grad_return(cpt, plan, ep, dkw, dvw, dko, dvo, slots_k, slots_v, wstreams, ostreams, stream):
    """The staged flow on 2P streams: P writer streams scatter their global
    dK/dV into owner-major slots [owner][writer] and publish the epoch; P
    owner streams wait for all writers and reduce their P slots in writer
    order. The main stream waits for all of them."""
    import torch

    Pn = len(wstreams)
    cpt.cpt_epoch_advance(ep)
    start = torch.cuda.Event()
    start.record(stream)
    for w in range(Pn):
        ws_ = wstreams[w]
        ws_.wait_event(start)
        cpt.cpt_grad_scatter(plan, w, dkw[w], [slots_k[o, w] for o in range(Pn)], slots_k[w, w], stream=ws_)
        cpt.cpt_grad_scatter(plan, w, dvw[w], [slots_v[o, w] for o in range(Pn)], slots_v[w, w], stream=ws_)
        cpt.cpt_epoch_publish(ep, w, stream=ws_)
    for o in range(Pn):
        os_ = ostreams[o]
        os_.wait_event(start)
        cpt.cpt_epoch_wait(ep, o, 1_000_000_000, cpt.CPT_WAIT_BOUNDED, stream=os_)
        cpt.cpt_slot_reduce(slots_k[o], dko[o], ep.status_ptr(o), stream=os_)
        cpt.cpt_slot_reduce(slots_v[o], dvo[o], ep.status_ptr(o), stream=os_)
    for st in wstreams + ostreams:
        stream.wait_stream(st)


CONFIG_ROWS = ("single_doc", "lognormal_partition", "lognormal_grad_return", "slot_reduce", "pages_extras")


def run_config_rows(cpt, synth, stream, dev, peak, names, reps=20, warm=3, big=None):
    """Every configuration of the workload table besides the headline step,
    timed with CUDA events on `stream` in this run. Each row gives time,
    algorithmic bytes, GB/s, the fraction of the HBM peak and the kernel the
    measured rule picked. `big` holds the pages-shaped step's tensors for the
    restore, accumulate, allocation-free and staged rows."""
    import torch

    out = {}
    BF = cpt.CPT_BF16

    def kernel_of(call, Pk, in_dt, out_dt, acc, row_b, rows):
        k = cpt.cpt_kernel_path_of(call, Pk, in_dt, out_dt, acc, row_b, rows)
        return "bulk" if k == cpt.CPT_KERNEL_BULK else "loads"

    def row(ms, nbytes, **extra):
        gbs = nbytes / (ms / 1e3) / 1e9
        return {"ms": ms, "bytes": nbytes, "gbs": gbs, "frac_of_peak": gbs / peak, **extra}

    if "single_doc" in names:
        # P=4, S=32768 one document, 8x128 bf16 N(0,1): 0.67 GB per launch,
        # close to the 129 MB L2 in reach, so a 512 MB write flushes L2 first
        Tg, Hg = 32768, 8
        rb = Hg * D * 2
        plan = cpt.cpt_plan_create(0, P, [0, Tg], Tg)
        wk = synth.device_normal_bf16((P, Tg, Hg, D), 7001, 1.0, dev)
        wv = synth.device_normal_bf16((P, Tg, Hg, D), 7002, 1.0, dev)
        ok = torch.empty((P, Tg // P, Hg, D), dtype=torch.bfloat16, device=dev)
        ov = torch.empty_like(ok)
        flush = torch.zeros(512 << 20, dtype=torch.uint8, device=dev)
        sink = torch.empty((), dtype=torch.int64, device=dev)
        nbytes = Tg * (2 * (P + 1) * rb + 2 * 4)
        ms = _events_ms(lambda: cpt.cpt_grad_return(plan, wk, wv, ok, ov), stream, reps, warm,
                        before=flush.zero_)
        # the same after a flush that reads the 512 MB instead: L2 is then full
        # of clean lines, and the launch pays no write-back of someone else's
        ms_read = _events_ms(lambda: cpt.cpt_grad_return(plan, wk, wv, ok, ov), stream, reps, warm,
                             before=lambda: torch.sum(flush.view(torch.int64), dim=0, out=sink))
        gbs_read = nbytes / (ms_read / 1e3) / 1e9
        out["single_doc_grad_return_P4_S32768_8x128"] = row(
            ms, nbytes, l2="flushed before each launch by writing 512 MB",
            kernel=kernel_of(cpt.CPT_CALL_GRAD_RETURN, P, BF, BF, 0, rb, 2 * Tg),
            read_flush={"ms": ms_read, "gbs": gbs_read, "frac_of_peak": gbs_read / peak,
                        "l2": "flushed before each launch by reading 512 MB"})
        del wk, wv, ok, ov, flush, sink, plan

    if "lognormal_partition" in names or "lognormal_grad_return" in names:
        # T=131072 from lognormal document lengths, 16x128 bf16: per-document
        # DualChunkSwap on lengths rounded to multiples of 8, packed-contiguous
        # on the raw lengths; the Q/K/V partition and the dK+dV gradient return
        Tl, Hl = 131072, 16
        rb = Hl * D * 2
        if "lognormal_partition" in names:
            qkv = [synth.device_normal_bf16((Tl, Hl, D), 7100 + t, 1.0, dev) for t in range(3)]
            loc = [torch.empty((P, Tl // P, Hl, D), dtype=torch.bfloat16, device=dev) for _ in range(3)]
        if "lognormal_grad_return" in names:
            wk = synth.device_normal_bf16((P, Tl, Hl, D), 7110, 1.0, dev)
            wv = synth.device_normal_bf16((P, Tl, Hl, D), 7111, 1.0, dev)
            ok = torch.empty((P, Tl // P, Hl, D), dtype=torch.bfloat16, device=dev)
            ov = torch.empty_like(ok)
        for name, layout, mult in (("per_document_dual_chunk_swap", 0, 8), ("packed_contiguous", 1, 1)):
            lens = synth.lognormal_doc_lengths(Tl, synth.rng_for(2, 0), multiple=mult)
            plan = cpt.cpt_plan_create(layout, P, synth.cu_from_lengths(lens), Tl)
            if "lognormal_partition" in names:
                ms = _events_ms(lambda: cpt.cpt_partition(plan, qkv, loc), stream, reps, warm)
                out[f"lognormal_T131072_16x128_partition_{name}"] = row(
                    ms, Tl * (3 * 2 * rb + 3 * 4), tok_s=Tl / (ms / 1e3), docs=len(lens),
                    kernel="bulk" if cpt.cpt_kernel_path_of(cpt.CPT_CALL_ROW_GATHER, P, BF, BF, 0, rb,
                                                            3 * Tl) == cpt.CPT_KERNEL_BULK else "loads")
            if "lognormal_grad_return" in names:
                ms = _events_ms(lambda: cpt.cpt_grad_return(plan, wk, wv, ok, ov), stream, reps, warm)
                out[f"lognormal_T131072_16x128_grad_return_{name}"] = row(
                    ms, Tl * (2 * (P + 1) * rb + 2 * 4), docs=len(lens),
                    kernel=kernel_of(cpt.CPT_CALL_GRAD_RETURN, P, BF, BF, 0, rb, 2 * Tl))
            del plan
        if "lognormal_partition" in names:
            del qkv, loc
        if "lognormal_grad_return" in names:
            del wk, wv, ok, ov

    if "slot_reduce" in names:
        # 8 slots, uniform[-1,1]: 1 KB and 1 MB per slot as latency (launched
        # back to back from Python, and as replays of a graph of such calls),
        # 1 GB per slot as bandwidth over 9 GB read + written
        n_slots = 8
        for dtype, tag, code in ((torch.float32, "f32", cpt.CPT_F32), (torch.bfloat16, "bf16", BF)):
            esz = 4 if dtype == torch.float32 else 2
            for label, nbytes in (("1KB", 1 << 10), ("1MB", 1 << 20), ("1GB", 1 << 30)):
                n = nbytes // esz
                gen = torch.Generator(device=dev)
                gen.manual_seed(7200 + esz)
                slots = [(torch.rand(n, device=dev, generator=gen) * 2 - 1).to(dtype) for _ in range(n_slots)]
                dst = torch.empty(n, dtype=dtype, device=dev)
                kern = kernel_of(cpt.CPT_CALL_SLOT_REDUCE, n_slots, code, code, 0, nbytes, 0)
                if nbytes >= 1 << 30:
                    ms = _events_ms(lambda: cpt.cpt_slot_reduce(slots, dst), stream, 10, warm)
                    r = row(ms, (n_slots + 1) * nbytes, kernel=kern)
                    # the ceiling with the same 8 reads : 1 write, once per run
                    if "read8_write1" not in out.setdefault("_ceilings", {}):
                        tried = []
                        for blk, stages, ctas in CEILING_SHAPES["read8_write1"]:
                            c_ms = _events_ms(lambda: cpt.cpt_stream_ceiling(slots, dst, blk, stages, ctas),
                                              stream, 10, warm)
                            tried.append(((n_slots + 1) * nbytes / (c_ms / 1e3) / 1e9, blk, stages, ctas))
                        best = max(tried)
                        out["_ceilings"]["read8_write1"] = {
                            "gbs": best[0], "shape": {"block_bytes": best[1], "stages": best[2],
                                                      "ctas_per_sm": best[3]},
                            "tried_gbs": [round(t[0], 1) for t in tried]}
                    r["frac_mix"] = r["gbs"] / out["_ceilings"]["read8_write1"]["gbs"]
                    out[f"slot_reduce_8x{label}_{tag}"] = r
                else:
                    iters = 200
                    launched = _events_ms(lambda: [cpt.cpt_slot_reduce(slots, dst) for _ in range(iters)],
                                          stream, 3, 1) * 1e3 / iters
                    # the same call straight through the C ABI with its arguments
                    # built once, as a C or C++ caller makes it: the library's
                    # own host cost (checks and launch) without the binding's
                    arr = (ctypes.c_void_p * n_slots)(*[x.data_ptr() for x in slots])
                    c_args = (ctypes.cast(arr, ctypes.c_void_p), n_slots, n, code, code,
                              ctypes.c_void_p(dst.data_ptr()), None, ctypes.c_void_p(stream.cuda_stream))
                    if cpt._lib.cpt_slot_reduce(*c_args) != cpt.CPT_OK:
                        raise RuntimeError(cpt.cpt_last_error_string())
                    c_abi = _events_ms(lambda: [cpt._lib.cpt_slot_reduce(*c_args) for _ in range(iters)],
                                       stream, 3, 1) * 1e3 / iters
                    side = torch.cuda.Stream(device=dev)
                    side.wait_stream(stream)
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
                        for _ in range(iters):
                            cpt.cpt_slot_reduce(slots, dst, stream=side)
                    stream.wait_stream(side)
                    graph_us = _events_ms(g.replay, stream, 3, 1) * 1e3 / iters
                    out[f"slot_reduce_8x{label}_{tag}"] = {
                        "us_per_call_launched": launched, "us_per_call_c_abi": c_abi,
                        "us_per_call_graph": graph_us,
                        "bytes": (n_slots + 1) * nbytes, "kernel": kern,
                        "note": ("latency, L2-resident, back-to-back calls: launched = through the "
                                 "Python binding; c_abi = the C entry point with prebuilt arguments; "
                                 "graph = replays of a CUDA graph of such calls")}
                    del g
                del slots, dst

    if "pages_extras" in names and big is not None:
        # the widened rows at the pages' shape, on the step's own tensors
        plan, qkv, part, dkw, dvw, dko, dvo = big
        rb = H * D * 2
        back = [torch.empty((S, H, D), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        ms = _events_ms(lambda: cpt.cpt_restore(plan, part[1:], back), stream, reps, warm)
        out["pages_restore_kv"] = row(ms, S * (2 * 2 * rb + 2 * 4), tok_s=S / (ms / 1e3),
                                      kernel="bulk" if cpt.cpt_kernel_path_of(
                                          cpt.CPT_CALL_ROW_GATHER, P, BF, BF, 0, rb, 2 * S)
                                      == cpt.CPT_KERNEL_BULK else "loads")
        del back
        ms = _events_ms(lambda: cpt.cpt_grad_return_accumulate(plan, dkw, dvw, dko, dvo), stream, reps, warm)
        out["pages_grad_return_accumulate"] = row(ms, S * (2 * (P + 2) * rb + 2 * 4),
                                                  kernel=kernel_of(cpt.CPT_CALL_GRAD_RETURN, P, BF, BF, 1,
                                                                   rb, 2 * S))
        ms = _events_ms(lambda: cpt.cpt_grad_return_noalloc(0, P, [0, S], S, dkw, dvw, dko, dvo), stream,
                        reps, warm)
        out["pages_grad_return_noalloc"] = row(ms, S * (2 * (P + 1) * rb + 2 * 4) + S * 4,
                                               kernel=kernel_of(cpt.CPT_CALL_GRAD_RETURN, P, BF, BF, 0,
                                                                rb, 2 * S),
                                               note="includes its own map build each call")
        slots_k = torch.empty((P, P, S // P, H, D), dtype=torch.bfloat16, device=dev)
        slots_v = torch.empty_like(slots_k)
        ep = cpt.cpt_epoch_create(P)
        wst = [torch.cuda.Stream(device=dev) for _ in range(P)]
        ost = [torch.cuda.Stream(device=dev) for _ in range(P)]
        ms = _events_ms(lambda: staged_grad_return(cpt, plan, ep, dkw, dvw, dko, dvo, slots_k, slots_v,
                                                   wst, ost, stream), stream, 10, warm)
        out["pages_grad_return_staged"] = row(ms, S * 2 * ((3 * P + 1) * rb + P * 4), streams=2 * P,
                                              note="scatter + publish + bounded wait + slot reduce")
        del slots_k, slots_v
    torch.cuda.synchronize()
    return out


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from context_attention_token_gb300 import build as cpt_build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    if rank == 0 or world == 1:
        cpt_build.build()
    if world > 1:
        dist.barrier()
    from context_attention_token_gb300 import cpt, synth

    cpt.cpt_set_kernel_path({"auto": cpt.CPT_KERNEL_AUTO, "loads": cpt.CPT_KERNEL_LOADS,
                                    "bulk": cpt.CPT_KERNEL_BULK}[args.kernel_path])
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()

    # inputs resident in HBM (seeded device draws)
    qkv = [synth.device_normal_bf16((S, H, D), 3000 + t, 1.0, dev) for t in range(3)]
    dkw = synth.device_normal_bf16((P, S, H, D), 3010, 0.02, dev)
    dvw = synth.device_normal_bf16((P, S, H, D), 3011, 0.02, dev)
    part = [torch.empty((P, S // P, H, D), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    dko = torch.empty((P, S // P, H, D), dtype=torch.bfloat16, device=dev)
    dvo = torch.empty_like(dko)
    cu = [0, S]
    ws = torch.empty(cpt.cpt_plan_workspace_bytes(0, P, 1, S), dtype=torch.uint8, device=dev)
    kernels_per_step = 4

    ev_gr = []
    ev_part = []

    def step(record=False):
        plan = cpt.cpt_plan_create(cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP, P, cu, S, workspace=ws)
        if record:
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
        cpt.cpt_partition(plan, qkv, part)
        if record:
            e1.record(stream)
        if args.path == "staged":
            grad_return_staged(plan)
        else:
            cpt.cpt_grad_return(plan, dkw, dvw, dko, dvo)
        if record:
            e2.record(stream)
            ev_part.append((e0, e1))
            ev_gr.append((e1, e2))
        cpt.cpt_plan_destroy(plan)

    if args.path == "staged":
        slots_k = torch.empty((P, P, S // P, H, D), dtype=torch.bfloat16, device=dev)
        slots_v = torch.empty_like(slots_k)
        ep = cpt.cpt_epoch_create(P)
        wstreams = [torch.cuda.Stream() for _ in range(P)]
        ostreams = [torch.cuda.Stream() for _ in range(P)]
        kernels_per_step = 2 + 1 + P * 2 + P * 3  # plan, partition, scatters, checks + reduces

    def grad_return_staged(plan):
        staged_grad_return(cpt, plan, ep, dkw, dvw, dko, dvo, slots_k, slots_v, wstreams, ostreams, stream)

    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not gpu_uuid.startswith("GPU-"):
            gpu_uuid = "GPU-" + gpu_uuid
    except Exception:
        gpu_uuid = str(local)
    sampler = ClockSampler(gpu_uuid)
    sampler.start()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    start.record(stream)
    for _ in range(args.steps):
        step(record=True)
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    sampler.stop()
    elapsed_ms = start.elapsed_time(end)
    gr_ms = [a.elapsed_time(b) for a, b in ev_gr]
    part_ms = [a.elapsed_time(b) for a, b in ev_part]

    max_ms = max_over_ranks(elapsed_ms, dev)
    copy_gbs = copy_ceiling_gbs(dev, stream)

    # ---- end to end through the public API with host buffers
    e2e = None
    e2e_skip = None
    if not args.no_e2e:
        # every rank on this node pins its own host copy of the step's inputs
        # and outputs; leave the e2e leg out (with the reason) rather than
        # exhaust host memory
        need = sum(x.numel() * x.element_size() for x in qkv + [dkw, dvw] + part + [dko, dvo])
        local_world = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
        avail = host_mem_available()
        if avail is not None and need * local_world > 0.8 * avail:
            e2e_skip = (f"needs {need * local_world / 1e9:.1f} GB of pinned host memory for "
                        f"{local_world} rank(s), {avail / 1e9:.1f} GB available")
    if not args.no_e2e and e2e_skip is None:
        try:
            host_in = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in qkv + [dkw, dvw]]
            host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in part + [dko, dvo]]
        except RuntimeError as err:  # pinned allocation refused
            e2e_skip = f"pinned host allocation failed: {str(err).splitlines()[0]}"
    if not args.no_e2e and world > 1:
        # the e2e leg holds collectives: every rank runs it or none does
        ok = torch.tensor([0 if e2e_skip else 1], dtype=torch.int32, device=dev)
        dist.all_reduce(ok, op=dist.ReduceOp.MIN)
        if int(ok.item()) == 0 and e2e_skip is None:
            e2e_skip = "another rank could not pin its host buffers"
            del host_in, host_out
    if not args.no_e2e and e2e_skip is None:
        for h, d in zip(host_in, qkv + [dkw, dvw]):
            h.copy_(d)
        h2d = sum(x.numel() * x.element_size() for x in host_in)
        d2h = sum(x.numel() * x.element_size() for x in host_out)

        h_qkv, h_dkw, h_dvw = host_in[:3], host_in[3], host_in[4]
        h_part, h_dko, h_dvo = host_out[:3], host_out[3], host_out[4]

        # Each global chunk of the DualChunkSwap map (2P chunks of m tokens)
        # feeds one contiguous range of local rows; read the map back once
        # (outside the timed region) to find those ranges.
        m = S // (2 * P)
        probe = cpt.cpt_plan_create(cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP, P, cu, S, workspace=ws)
        g2l_dev = torch.empty(S, dtype=torch.int32, device=dev)
        l2g_dev = torch.empty(S, dtype=torch.int32, device=dev)
        cpt.cpt_index_map(probe, l2g_dev, g2l_dev)
        g2l = g2l_dev.cpu()
        chunks = []
        for k in range(2 * P):
            qs = g2l[k * m:(k + 1) * m]
            q0 = int(qs[0])
            if not bool((qs == torch.arange(q0, q0 + m, dtype=qs.dtype)).all()):
                raise RuntimeError("chunk of the map is not a contiguous local range")
            chunks.append((k * m, q0))
        del probe, g2l_dev, l2g_dev
        flat = lambda t: t.view(S, H, D)  # noqa: E731  rank-major local tensor as [S, H, D]

        # Pieces: every global chunk of m tokens cut into `pieces` runs of
        # local rows, so the last piece's copy out (the pipeline's tail) is short.
        pieces = []
        for g0, q0 in chunks:
            cut = [m * i // args.e2e_pieces for i in range(args.e2e_pieces + 1)]
            pieces += [(g0 + a, q0 + a, b - a) for a, b in zip(cut, cut[1:]) if b > a]
        h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()

        # Two device buffer sets, used by alternate steps, so that a step's
        # copies in can run while the previous step's results are still being
        # copied out: the host link carries both directions at once, and its
        # host-to-device side never waits for a step boundary.
        sets = [(qkv, dkw, dvw, part, dko, dvo),
                ([torch.empty_like(x) for x in qkv], torch.empty_like(dkw), torch.empty_like(dvw),
                 [torch.empty_like(x) for x in part], torch.empty_like(dko), torch.empty_like(dvo))]
        kernels_done = [None, None]   # per set: the last kernel of the step that used it
        outputs_out = [None, None]    # per set: the last copy out of the step that used it

        def e2e_step(i):
            # Three streams, one per resource: copies in of every piece back to
            # back on h2d_stream, the kernels of a piece on the main stream once
            # its rows are in, its rows out on d2h_stream once its kernels are
            # done. A set's inputs are overwritten only after the kernels that
            # read them (two steps back) are done, and its outputs only after
            # they were copied out.
            s_qkv, s_dkw, s_dvw, s_part, s_dko, s_dvo = sets[i % 2]
            t_host = time.perf_counter()
            plan = cpt.cpt_plan_create(cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP, P, cu, S, workspace=ws)
            if kernels_done[i % 2] is not None:
                h2d_stream.wait_event(kernels_done[i % 2])
            if outputs_out[i % 2] is not None:
                stream.wait_event(outputs_out[i % 2])
            # diagnostics: when this step's copies in start and end, and when
            # its copies out end, on their own streams
            marks = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            marks[0].record(h2d_stream)
            for g0, q0, c in pieces:
                with torch.cuda.stream(h2d_stream):
                    for d, h in zip(s_qkv, h_qkv):
                        d[g0:g0 + c].copy_(h[g0:g0 + c], non_blocking=True)
                    qkv_in = torch.cuda.Event()
                    qkv_in.record(h2d_stream)
                    for w in range(P):
                        s_dkw[w, g0:g0 + c].copy_(h_dkw[w, g0:g0 + c], non_blocking=True)
                        s_dvw[w, g0:g0 + c].copy_(h_dvw[w, g0:g0 + c], non_blocking=True)
                    grads_in = torch.cuda.Event()
                    grads_in.record(h2d_stream)
                stream.wait_event(qkv_in)
                cpt.cpt_partition_rows(plan, s_qkv, s_part, q0, c)
                part_done = torch.cuda.Event()
                part_done.record(stream)
                stream.wait_event(grads_in)
                cpt.cpt_grad_return_rows(plan, s_dkw, s_dvw, s_dko, s_dvo, q0, c)
                grads_done = torch.cuda.Event()
                grads_done.record(stream)
                with torch.cuda.stream(d2h_stream):
                    d2h_stream.wait_event(part_done)
                    for h, d in zip(h_part, s_part):
                        flat(h)[q0:q0 + c].copy_(flat(d)[q0:q0 + c], non_blocking=True)
                    d2h_stream.wait_event(grads_done)
                    flat(h_dko)[q0:q0 + c].copy_(flat(s_dko)[q0:q0 + c], non_blocking=True)
                    flat(h_dvo)[q0:q0 + c].copy_(flat(s_dvo)[q0:q0 + c], non_blocking=True)
            marks[1].record(h2d_stream)
            marks[2].record(d2h_stream)
            kernels_done[i % 2] = torch.cuda.Event()
            kernels_done[i % 2].record(stream)
            outputs_out[i % 2] = torch.cuda.Event()
            outputs_out[i % 2].record(d2h_stream)
            cpt.cpt_plan_destroy(plan)
            step_marks.append((marks, (time.perf_counter() - t_host) * 1e3))

        step_marks = []

        def join():
            stream.wait_stream(h2d_stream)
            stream.wait_stream(d2h_stream)

        # The host link's floor for one step, measured on the step's own
        # pinned buffers before the e2e leg: every input copied in alone,
        # every output copied out alone, and both at once on two streams.
        dev_in, dev_out = qkv + [dkw, dvw], part + [dko, dvo]

        def copies(inp, outp):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            h2d_stream.wait_stream(stream)
            d2h_stream.wait_stream(stream)
            if inp:
                with torch.cuda.stream(h2d_stream):
                    for d, h in zip(dev_in, host_in):
                        d.copy_(h, non_blocking=True)
            if outp:
                with torch.cuda.stream(d2h_stream):
                    for h, d in zip(host_out, dev_out):
                        h.copy_(d, non_blocking=True)
            stream.wait_stream(h2d_stream)
            stream.wait_stream(d2h_stream)
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b)

        link = {}
        for key, inp, outp in (("h2d_ms", True, False), ("d2h_ms", False, True), ("both_ms", True, True)):
            copies(inp, outp)
            link[key] = min(copies(inp, outp) for _ in range(2))
        r_in = h2d / (link["h2d_ms"] / 1e3)
        r_out = d2h / (link["d2h_ms"] / 1e3)

        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        for i in range(2):  # warm-up: one step on each buffer set
            e2e_step(i)
        join()
        torch.cuda.synchronize()
        step_marks.clear()
        if world > 1:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h2d_stream.wait_stream(stream)
        d2h_stream.wait_stream(stream)
        for i in range(e2e_steps):
            e2e_step(i)
        join()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b), dev) / e2e_steps
        # per step: copies-in span, idle time of the copy-in stream before the
        # step's first copy, lag of the last copy out behind the last copy in,
        # and host time to enqueue the step (large when the host had to wait)
        spans = [m[0].elapsed_time(m[1]) for m, _ in step_marks]
        gaps = [step_marks[k - 1][0][1].elapsed_time(step_marks[k][0][0]) for k in range(1, len(step_marks))]
        lags = [m[1].elapsed_time(m[2]) for m, _ in step_marks]
        host = [h for _, h in step_marks]
        diag = {"h2d_span_ms": [round(x, 2) for x in spans], "h2d_idle_before_ms": [round(x, 2) for x in gaps],
                "d2h_lag_ms": [round(x, 2) for x in lags], "host_enqueue_ms": [round(x, 2) for x in host]}
        # the results that came back equal the device-resident step's, on
        # sampled rows of every output (both sets computed the same inputs)
        g = torch.Generator().manual_seed(7)
        rows_chk = torch.randint(0, S, (4096,), generator=g)
        for h, d in zip(h_part + [h_dko, h_dvo], part + [dko, dvo]):
            if not torch.equal(flat(h)[rows_chk], flat(d)[rows_chk.to(dev)].cpu()):
                raise RuntimeError("e2e results differ from the device-resident step")
        # the same copies-only probe right after the leg (and its check): a
        # link that was slow during the leg shows here too, a pipeline stall
        # does not
        both_after_ms = min(copies(True, True) for _ in range(2))
        # the floor of one step: all of its copies in and out at once, with
        # nothing else on the link or the GPU, at the better of the two probes
        # (the link's rate changes from outside the process; diag shows when)
        link_floor_ms = min(link["both_ms"], both_after_ms)
        del sets
        e2e = {"value": whole_job_gbs(step_bytes(S), 1, world, e2e_ms), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": e2e_steps,
               "pipeline": (f"copies in, kernels, copies out on 3 streams over {len(pieces)} pieces, "
                            "two buffer sets so consecutive steps overlap"),
               "diag": diag,
               "link_floor_ms": link_floor_ms,
               "vs_link_floor": e2e_ms / link_floor_ms,
               "link": {"h2d_gbs": r_in / 1e9, "d2h_gbs": r_out / 1e9,
                        "h2d_alone_ms": link["h2d_ms"], "d2h_alone_ms": link["d2h_ms"],
                        "copies_only_ms": link["both_ms"],
                        "copies_only_after_ms": both_after_ms,
                        "how": ("the step's own pinned buffers copied in alone, out alone, and all "
                                "in and out at once on two streams (best of 2, CUDA events), just "
                                "before the e2e leg and again after it; link_floor_ms = the "
                                "better of the two all-at-once times")}}
        del host_in, host_out

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    peak, peak_src = load_peak()
    # mix-matched ceilings, into scratch buffers (the step's outputs stay as
    # they are): P of the writer tensors -> one owner-sized buffer, and Q ->
    # one local-sized buffer
    scratch4 = torch.empty_like(dko)
    scratch1 = torch.empty_like(part[0])
    ceil = mix_ceilings(cpt, [dkw[w] for w in range(P)], scratch4, qkv[0], scratch1, stream)
    del scratch4, scratch1
    configs = {}
    if args.configs != "none":
        names = CONFIG_ROWS if args.configs == "all" else tuple(args.configs.split(","))
        if (S, H) != (262144, 20):
            names = tuple(n for n in names if n != "pages_extras")
        plan_big = cpt.cpt_plan_create(cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP, P, cu, S, workspace=ws)
        configs = run_config_rows(cpt, synth, stream, dev, peak, names, reps=args.config_reps,
                                  warm=args.config_warmup,
                                  big=(plan_big, qkv, part, dkw, dvw, dko, dvo))
        cpt.cpt_plan_destroy(plan_big)
    timeouts = cpt.cpt_kernel_wait_timeouts()
    traffic, traffic_note = profiled_traffic("grad_return", S)
    gr_bytes = S * gr_bytes_per_token()
    gr_mean_ms = statistics.mean(gr_ms)
    gr_gbs = gr_bytes / (gr_mean_ms / 1e3) / 1e9
    part_bytes = S * part_bytes_per_token()
    part_mean_ms = statistics.mean(part_ms)
    part_gbs = part_bytes / (part_mean_ms / 1e3) / 1e9
    value = whole_job_gbs(step_bytes(S), args.steps, world, max_ms)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded device N(0,1) Q/K/V, N(0,0.02) dK/dV)",
        "config": {"workload": workload(), "P": P, "S": S, "H": H, "D": D,
                   "layout": "dual_chunk_swap", "grad_return_path": PATH,
                   "kernel_path": args.kernel_path,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (21.5 GB touched per step), no flush",
                   "step_bytes": step_bytes(S)},
        "grad_return": {"gbs": gr_gbs, "frac_of_peak": gr_gbs / peak, "ms": gr_mean_ms,
                        "bytes_per_launch": gr_bytes},
        "partition": {"tok_s": S / (part_mean_ms / 1e3), "gbs": part_gbs,
                      "frac_of_peak": part_gbs / peak, "ms": part_mean_ms,
                      "frac_mix": part_gbs / ceil["read1_write1"]["gbs"]},
        "roofline": {"kernel": "grad_return", "bound": "hbm", "achieved": gr_gbs, "peak": peak,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6800 GB/s", "unit": "GB/s", "frac": gr_gbs / peak,
                     "frac_mix": gr_gbs / ceil["read4_write1"]["gbs"],
                     "peak_mix": ceil["read4_write1"]["gbs"],
                     "traffic": traffic if PATH == "fused" else None,
                     "traffic_source": traffic_note if PATH == "fused" else None},
        "ceilings": {**ceil, **configs.pop("_ceilings", {}),
                     "how": ("cpt_stream_ceiling: the read/write mix of the call with no "
                                     "arithmetic, bulk copies through shared memory; the fastest of "
                                     "the shapes tried, CUDA events, median of 10 after 3")},
        "configs": configs,
        "wait_timeouts": timeouts,
        "copy_ceiling": {"gbs": copy_gbs, "grad_return_frac": gr_gbs / copy_gbs,
                         "partition_frac": part_gbs / copy_gbs,
                         "how": "torch copy_ of 1 Gi bf16 elements in this run, read+write bytes, "
                                "best of 10 after 3, CUDA events"},
        "clocks": sampler.summary(t_wall0, t_wall1),
        "kernels": {
            "partition": "bulk-copy row blocks" if cpt.cpt_kernel_path_of(
                cpt.CPT_CALL_ROW_GATHER, P, cpt.CPT_BF16, cpt.CPT_BF16, False, row_bytes(), 3 * S)
            == cpt.CPT_KERNEL_BULK else "16-byte loads",
            "grad_return": "bulk-copy row pipelines" if cpt.cpt_kernel_path_of(
                cpt.CPT_CALL_GRAD_RETURN, P, cpt.CPT_BF16, cpt.CPT_BF16, False, row_bytes(), 2 * S)
            == cpt.CPT_KERNEL_BULK else "16-byte loads",
            "path": args.kernel_path},
        "gpu_launches": kernels_per_step * args.steps,
        "e2e": e2e if e2e is not None else ({"value": None, "unit": "GB/s", "skipped": e2e_skip}
                                            if e2e_skip else None),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.sample_tokens, args.cpu_budget,
                                            args.cpu_cores or host_cores())
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- next rows

def _median_launch_ms(fn, stream, reps=20, warm=3):
    import torch

    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    evs = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def run_next_rows(args):
    """One JSON line per widened row, each at the pages' shape unless noted:
    restore (all-gather inverse reorder), accumulate-into grad_return, the
    P=2/8 grad_return sweep, the allocation-free grad_return, and a
    matched-input comparison of the partition policies on the lognormal
    packed-THD batch (T=131072, 16x128)."""
    import numpy as np
    import torch

    from context_attention_token_gb300 import build as cpt_build

    cpt_build.build()
    from context_attention_token_gb300 import cpt, synth

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    peak, peak_src = load_peak()
    row = H * D * 2

    def emit(name, ms, nbytes, **extra):
        gbs = nbytes / (ms / 1e3) / 1e9
        line = {"next_row": name, "ms": ms, "bytes": nbytes, "gbs": gbs, "frac_of_peak": gbs / peak,
                "peak": peak, "peak_source": peak_src, **extra}
        print(json.dumps(line), flush=True)

    # integer metadata: launch-bound, reported as latency. Per configuration:
    # the plan (cu_seqlens copy + map and metadata kernels) as host wall time
    # of the call and as device time between events; the stand-alone map and
    # metadata calls as device time; both as CUDA-graph replays per pair.
    lat_cases = (
        ("tiny_T64_P2_dsc", 0, 2, [16, 24, 24]),
        ("tiny_T64_P2_packed", 1, 2, [16, 24, 24]),
        ("single_doc_S32768_P4", 0, P, [32768]),
        ("lognormal_T131072_P4_dsc", 0, P,
         synth.lognormal_doc_lengths(131072, synth.rng_for(2, 0), multiple=8)),
        ("lognormal_T131072_P4_packed", 1, P, synth.lognormal_doc_lengths(131072, synth.rng_for(2, 0))),
        ("lognormal_T131072_P4_padded", 3, P, synth.lognormal_doc_lengths(131072, synth.rng_for(2, 0))),
        ("pages_S262144_P4", 0, P, [S]),
    )
    for name, layout, Pl, lens_l in lat_cases:
        cu_l = synth.cu_from_lengths(lens_l)
        T_l, n_l = int(cu_l[-1]), len(lens_l)
        ws_l = torch.empty(cpt.cpt_plan_workspace_bytes(layout, Pl, n_l, T_l), dtype=torch.uint8,
                           device="cuda")
        host_us, dev_ms = [], []
        for it in range(23):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            t0 = time.perf_counter()
            pl = cpt.cpt_plan_create(layout, Pl, cu_l, T_l, workspace=ws_l)
            t1 = time.perf_counter()
            b.record(stream)
            torch.cuda.synchronize()
            cpt.cpt_plan_destroy(pl)
            if it >= 3:
                host_us.append((t1 - t0) * 1e6)
                dev_ms.append(a.elapsed_time(b))
        pl = cpt.cpt_plan_create(layout, Pl, cu_l, T_l, workspace=ws_l)
        Tp_l = pl.padded_tokens
        l2g_l = torch.empty(Tp_l, dtype=torch.int32, device="cuda")
        g2l_l = torch.empty(Tp_l, dtype=torch.int32, device="cuda")
        meta = (torch.empty(Pl, dtype=torch.int32, device="cuda"),
                torch.empty(Pl, dtype=torch.int32, device="cuda"),
                torch.empty((Pl, n_l + 1), dtype=torch.int32, device="cuda"),
                torch.empty(Pl + 1, dtype=torch.int32, device="cuda"))
        map_ms = _median_launch_ms(lambda: cpt.cpt_index_map(pl, l2g_l, g2l_l), stream)
        meta_ms = _median_launch_ms(lambda: cpt.cpt_thd_metadata(pl, *meta), stream)
        side = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        reps = 20
        with torch.cuda.stream(side):
            cpt.cpt_index_map(pl, l2g_l, g2l_l, stream=side)
            cpt.cpt_thd_metadata(pl, *meta, stream=side)
            side.synchronize()
            with torch.cuda.graph(graph, stream=side):
                for _ in range(reps):
                    cpt.cpt_index_map(pl, l2g_l, g2l_l, stream=side)
                    cpt.cpt_thd_metadata(pl, *meta, stream=side)
        graph.replay()
        torch.cuda.synchronize()
        graph_ms = _median_launch_ms(graph.replay, stream, reps=10)
        print(json.dumps({"metadata_latency": name, "layout": layout, "P": Pl, "T": T_l,
                          "T_padded": Tp_l, "docs": n_l,
                          "plan_create_host_us": statistics.median(host_us),
                          "plan_create_device_us": statistics.median(dev_ms) * 1e3,
                          "index_map_device_us": map_ms * 1e3,
                          "thd_metadata_device_us": meta_ms * 1e3,
                          "map_plus_metadata_graph_us": graph_ms * 1e3 / reps}), flush=True)
        cpt.cpt_plan_destroy(pl)
        del graph, ws_l, l2g_l, g2l_l, meta

    # the Q/K/V partition at the pages' shape under each gather kernel
    plan = cpt.cpt_plan_create(0, P, [0, S], S)
    qkv_p = [synth.device_normal_bf16((S, H, D), 5900 + t, 1.0, "cuda") for t in range(3)]
    out_p = [torch.empty((P, S // P, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    for kname, kcode in (("", cpt.CPT_KERNEL_AUTO), ("_loads_kernel", cpt.CPT_KERNEL_LOADS),
                         ("_bulk_kernel", cpt.CPT_KERNEL_BULK)):
        cpt.cpt_set_kernel_path(kcode)
        ms = _median_launch_ms(lambda: cpt.cpt_partition(plan, qkv_p, out_p), stream)
        emit("partition_pages_shape" + kname, ms, S * (3 * 2 * row + 3 * 4), S=S, P=P,
             tok_s=S / (ms / 1e3), kernel=kname.strip("_").replace("_kernel", "") or "auto")
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)
    del qkv_p, out_p

    # f1: restore K and V from rank-local back to global order
    kv = [synth.device_normal_bf16((P, S // P, H, D), 6000 + t, 1.0, "cuda") for t in range(2)]
    back = [torch.empty((S, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ms = _median_launch_ms(lambda: cpt.cpt_restore(plan, kv, back), stream)
    emit("restore_kv", ms, S * (2 * 2 * row + 2 * 4), tensors=2, S=S, P=P,
         tok_s=S / (ms / 1e3))
    del kv, back

    # f4: accumulate-into grad_return, and the P sweep of the plain one
    for Pw in (2, 4, 8):
        planp = cpt.cpt_plan_create(0, Pw, [0, S], S)
        dkw = synth.device_normal_bf16((Pw, S, H, D), 6100 + Pw, 0.02, "cuda")
        dvw = synth.device_normal_bf16((Pw, S, H, D), 6200 + Pw, 0.02, "cuda")
        dko = torch.zeros((Pw, S // Pw, H, D), dtype=torch.bfloat16, device="cuda")
        dvo = torch.zeros_like(dko)
        ms = _median_launch_ms(lambda: cpt.cpt_grad_return(planp, dkw, dvw, dko, dvo), stream)
        emit(f"grad_return_P{Pw}", ms, S * (2 * (Pw + 1) * row + 2 * 4), P=Pw, S=S)
        if Pw == P:
            ms = _median_launch_ms(
                lambda: cpt.cpt_grad_return_accumulate(planp, dkw, dvw, dko, dvo), stream)
            emit("grad_return_accumulate_P4", ms, S * (2 * (Pw + 2) * row + 2 * 4), P=Pw, S=S)
            for kname, kcode in (("loads", cpt.CPT_KERNEL_LOADS), ("bulk", cpt.CPT_KERNEL_BULK)):
                cpt.cpt_set_kernel_path(kcode)
                ms = _median_launch_ms(
                    lambda: cpt.cpt_grad_return_accumulate(planp, dkw, dvw, dko, dvo), stream)
                emit(f"grad_return_accumulate_P4_{kname}_kernel", ms, S * (2 * (Pw + 2) * row + 2 * 4),
                     P=Pw, S=S, kernel=kname)
            cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)
            ms = _median_launch_ms(
                lambda: cpt.cpt_grad_return_noalloc(0, Pw, [0, S], S, dkw, dvw, dko, dvo), stream)
            emit("grad_return_noalloc_P4", ms, S * (2 * (Pw + 1) * row + 2 * 4) + S * 4, P=Pw, S=S,
                 note="includes its own map build (index-map kernel) each call")
            for kname, kcode in (("loads", cpt.CPT_KERNEL_LOADS), ("bulk", cpt.CPT_KERNEL_BULK)):
                cpt.cpt_set_kernel_path(kcode)
                ms = _median_launch_ms(lambda: cpt.cpt_grad_return(planp, dkw, dvw, dko, dvo), stream)
                emit(f"grad_return_P4_{kname}_kernel", ms, S * (2 * (Pw + 1) * row + 2 * 4), P=Pw, S=S,
                     kernel=kname)
            cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)
        del dkw, dvw, dko, dvo
        torch.cuda.empty_cache()

    # the other grad_return configurations: the
    # single-document case (S=32768, 8x128; its 0.67 GB are close to L2 size,
    # so each launch is preceded by a 512 MB write that flushes L2) and the
    # lognormal packed batch (T=131072, 16x128) under both layouts
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for name, Tg, Hg, lens_g in (("grad_return_single_doc_S32768_8x128", 32768, 8, [32768]),
                                 ("grad_return_lognormal_T131072_16x128_dsc", 131072, 16,
                                  synth.lognormal_doc_lengths(131072, synth.rng_for(2, 0), multiple=8)),
                                 ("grad_return_lognormal_T131072_16x128_packed", 131072, 16,
                                  synth.lognormal_doc_lengths(131072, synth.rng_for(2, 0)))):
        layout_g = 1 if name.endswith("packed") else 0
        plg = cpt.cpt_plan_create(layout_g, P, synth.cu_from_lengths(lens_g), Tg)
        wk = synth.device_normal_bf16((P, Tg, Hg, D), 6400, 1.0, "cuda")
        wv = synth.device_normal_bf16((P, Tg, Hg, D), 6401, 1.0, "cuda")
        ok = torch.empty((P, Tg // P, Hg, D), dtype=torch.bfloat16, device="cuda")
        ov = torch.empty_like(ok)
        for kname, kcode in (("", cpt.CPT_KERNEL_AUTO), ("_loads_kernel", cpt.CPT_KERNEL_LOADS),
                             ("_bulk_kernel", cpt.CPT_KERNEL_BULK)):
            cpt.cpt_set_kernel_path(kcode)
            evs = []
            for it in range(23):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                cpt.cpt_grad_return(plg, wk, wv, ok, ov)
                b.record(stream)
                if it >= 3:
                    evs.append((a, b))
            torch.cuda.synchronize()
            ms = statistics.median(x.elapsed_time(y) for x, y in evs)
            emit(name + kname, ms, Tg * (2 * (P + 1) * Hg * D * 2 + 2 * 4), P=P, T=Tg, docs=len(lens_g),
                 l2="flushed before each launch", kernel=kname.strip("_").replace("_kernel", "") or "auto")
        cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)
        del wk, wv, ok, ov
        torch.cuda.empty_cache()
    del flush

    # f3 / matched inputs: one lognormal batch (lengths multiples of 8 so all
    # three policies accept it), Q/K/V [T,16,128]
    T, Hq = 131072, 16
    lens = synth.lognormal_doc_lengths(T, synth.rng_for(2, 0), multiple=8)
    cu = synth.cu_from_lengths(lens)
    qkv = [synth.device_normal_bf16((T, Hq, D), 6300 + t, 1.0, "cuda") for t in range(3)]
    out = [torch.empty((P, T // P, Hq, D), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    for name, layout, cuu in (("per_document_dual_chunk_swap", 0, cu),
                              ("packed_contiguous", 1, cu),
                              ("mirrored_super_sequence_as_dsc_over_[0,T]", 0, np.array([0, T], np.int32))):
        pl = cpt.cpt_plan_create(layout, P, cuu, T)
        ms = _median_launch_ms(lambda: cpt.cpt_partition(pl, qkv, out), stream)
        emit(f"partition_policy:{name}", ms, T * (3 * 2 * Hq * D * 2 + 3 * 4), T=T, P=P,
             docs=len(lens), tok_s=T / (ms / 1e3))

    # f2: documents of raw (uneven) lengths: the padded per-document layout
    # pads on the fly; packed-contiguous needs no padding. Same raw batch.
    raw = synth.lognormal_doc_lengths(T, synth.rng_for(2, 0), multiple=1)
    cur = synth.cu_from_lengths(raw)
    for name, layout in (("per_document_padded", 3), ("packed_contiguous", 1)):
        pl = cpt.cpt_plan_create(layout, P, cur, T)
        Tpad = pl.padded_tokens
        outp = [torch.empty((P, Tpad // P, Hq, D), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
        ms = _median_launch_ms(lambda: cpt.cpt_partition(pl, qkv, outp), stream)
        emit(f"raw_lengths_partition:{name}", ms, 3 * ((T + Tpad) * Hq * D * 2 + Tpad * 4), T=T,
             T_padded=Tpad, P=P, docs=len(raw), tok_s=T / (ms / 1e3))
        del outp
    return 0


# ---------------------------------------------------------------- slot-reduce sweep

def run_host_link_sweep(args):
    """The host link under the e2e step: 2 GiB between pinned host memory and
    HBM by cudaMemcpyAsync, one direction at a time and both at once on two
    streams, best of 5 after a warm-up. One JSON line."""
    import torch

    torch.cuda.set_device(0)
    nbytes = 2 << 30
    h_src = torch.ones(nbytes, dtype=torch.uint8, pin_memory=True)
    h_dst = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_src = torch.ones(nbytes, dtype=torch.uint8, device="cuda")
    d_dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    main = torch.cuda.current_stream()

    def best_ms(fn):
        ms = []
        for i in range(6):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(main)
            s_in.wait_stream(main)
            s_out.wait_stream(main)
            fn()
            main.wait_stream(s_in)
            main.wait_stream(s_out)
            e1.record(main)
            torch.cuda.synchronize()
            if i:
                ms.append(e0.elapsed_time(e1))
        return min(ms)

    def h2d():
        with torch.cuda.stream(s_in):
            d_dst.copy_(h_src, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_out):
            h_dst.copy_(d_src, non_blocking=True)

    def both():
        h2d()
        d2h()

    gbs = lambda n, ms: n / (ms / 1e3) / 1e9  # noqa: E731
    line = {"sweep": "host_link", "bytes_per_direction": nbytes, "unit": "GB/s",
            "h2d": gbs(nbytes, best_ms(h2d)), "d2h": gbs(nbytes, best_ms(d2h)),
            "both_total": gbs(2 * nbytes, best_ms(both)),
            "how": "cudaMemcpyAsync between pinned host memory and HBM, CUDA events, best of 5"}
    print(json.dumps(line), flush=True)
    return 0


def run_grad_return_size_sweep(args):
    """The fused gradient return at P=4 with 2 KB rows (8x128 bf16, the
    single-document configuration's rows) over launches of 0.17 to 5.4 GB,
    each launch after an L2 flush (a 512 MB write), under the measured rule
    and with each kernel forced. One JSON line per (kernel, size), then one
    per kernel with a least-squares fit t = t0 + bytes / bw over the sizes,
    which separates a fixed per-launch cost from the streaming rate."""
    import torch

    from context_attention_token_gb300 import build as cpt_build

    cpt_build.build()
    from context_attention_token_gb300 import cpt, synth

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    peak, peak_src = load_peak()
    Hs = args.heads if args.heads != 20 else 8
    rb = Hs * D * 2
    flush = torch.zeros(512 << 20, dtype=torch.uint8, device="cuda")
    sink = torch.empty((), dtype=torch.int64, device="cuda")
    # "write" overwrites 512 MB (the flush the timing rules name), which leaves
    # L2 full of dirty lines the next kernel has to write back; "read" sums the
    # same 512 MB, which leaves it full of clean lines
    do_flush = flush.zero_ if args.flush == "write" else (lambda: torch.sum(flush.view(torch.int64), dim=0, out=sink))
    sizes = (8192, 16384, 32768, 65536, 131072, 262144)
    data = {name: [] for name in ("auto", "loads", "bulk")}
    for Ts in sizes:
        plan = cpt.cpt_plan_create(0, P, [0, Ts], Ts)
        wk = synth.device_normal_bf16((P, Ts, Hs, D), 7301, 1.0, "cuda")
        wv = synth.device_normal_bf16((P, Ts, Hs, D), 7302, 1.0, "cuda")
        ok = torch.empty((P, Ts // P, Hs, D), dtype=torch.bfloat16, device="cuda")
        ov = torch.empty_like(ok)
        nbytes = Ts * (2 * (P + 1) * rb + 2 * 4)
        for name, code in (("auto", cpt.CPT_KERNEL_AUTO), ("loads", cpt.CPT_KERNEL_LOADS),
                           ("bulk", cpt.CPT_KERNEL_BULK)):
            cpt.cpt_set_kernel_path(code)
            ms = _events_ms(lambda: cpt.cpt_grad_return(plan, wk, wv, ok, ov), stream, 20, 3,
                            before=do_flush)
            data[name].append((nbytes, ms))
            gbs = nbytes / (ms / 1e3) / 1e9
            print(json.dumps({"sweep": "grad_return_launch_size", "kernel": name, "P": P, "S": Ts,
                              "row_bytes": rb, "bytes": nbytes, "ms": ms, "gbs": gbs,
                              "frac_of_peak": gbs / peak,
                              "l2": f"flushed before each launch by a 512 MB {args.flush}"}), flush=True)
        cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)
        del wk, wv, ok, ov, plan
        torch.cuda.empty_cache()
    for name, pts in data.items():
        n = len(pts)
        mx = sum(b for b, _ in pts) / n
        my = sum(t for _, t in pts) / n
        sxx = sum((b - mx) ** 2 for b, _ in pts)
        slope = sum((b - mx) * (t - my) for b, t in pts) / sxx  # ms per byte
        t0 = my - slope * mx
        print(json.dumps({"sweep": "grad_return_launch_size_fit", "kernel": name, "flush": args.flush,
                          "t0_us": t0 * 1e3,
                          "streaming_gbs": 1 / (slope / 1e3) / 1e9,
                          "streaming_frac_of_peak": 1 / (slope / 1e3) / 1e9 / peak,
                          "peak": peak, "peak_source": peak_src,
                          "fit": "least squares of ms on bytes over all sizes"}), flush=True)
    return 0


def run_slot_reduce_sweep(args):
    """P slot buffers (--slots, default 8) of N bytes each, N = 1 KB x 4^k up to 1 GB, float32 and
    bf16: one ordered sum per launch. One JSON line per (dtype, N), with the
    launch latency (back-to-back C-ABI calls, and replays of a CUDA graph of
    such calls) and the effective bandwidth over (P+1)N algorithmic bytes."""
    import torch

    from context_attention_token_gb300 import build as cpt_build

    cpt_build.build()
    from context_attention_token_gb300 import cpt

    torch.cuda.set_device(0)
    cpt.cpt_set_kernel_path({"auto": cpt.CPT_KERNEL_AUTO, "loads": cpt.CPT_KERNEL_LOADS,
                            "bulk": cpt.CPT_KERNEL_BULK}[args.kernel_path])
    peak, peak_src = load_peak()
    stream = torch.cuda.Stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    n_slots = args.slots
    for dtype in (torch.float32, torch.bfloat16):
        esz = torch.tensor([], dtype=dtype).element_size()
        for k in range(11):
            nbytes = 1024 * 4**k
            n = nbytes // esz
            gen = torch.Generator(device="cuda")
            gen.manual_seed(5000 + k)
            slots = [(torch.rand(n, device="cuda", generator=gen) * 2 - 1).to(dtype) for _ in range(n_slots)]
            dst = torch.empty(n, dtype=dtype, device="cuda")
            iters = max(3, min(2000, int(2e9 // ((n_slots + 1) * nbytes))))
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                for _ in range(3):
                    cpt.cpt_slot_reduce(slots, dst, stream=stream)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(iters):
                    cpt.cpt_slot_reduce(slots, dst, stream=stream)
                b.record(stream)
            torch.cuda.synchronize()
            call_us = a.elapsed_time(b) * 1e3 / iters
            # the same call straight through the C ABI, arguments built once
            arr = (ctypes.c_void_p * n_slots)(*[x.data_ptr() for x in slots])
            code = cpt.CPT_F32 if dtype == torch.float32 else cpt.CPT_BF16
            c_args = (arr, n_slots, n, code, code, ctypes.c_void_p(dst.data_ptr()), None,
                      ctypes.c_void_p(stream.cuda_stream))
            if cpt._lib.cpt_slot_reduce(*c_args) != cpt.CPT_OK:
                raise RuntimeError(cpt.cpt_last_error_string())
            with torch.cuda.stream(stream):
                a1, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a1.record(stream)
                for _ in range(iters):
                    cpt._lib.cpt_slot_reduce(*c_args)
                b1.record(stream)
            torch.cuda.synchronize()
            c_abi_us = a1.elapsed_time(b1) * 1e3 / iters
            # the same calls captured once into a graph and replayed
            graph_us = None
            g_iters = min(iters, 200)
            try:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                    for _ in range(g_iters):
                        cpt.cpt_slot_reduce(slots, dst, stream=torch.cuda.current_stream())
                g.replay()
                torch.cuda.synchronize()
                a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    a2.record(stream)
                    g.replay()
                    b2.record(stream)
                torch.cuda.synchronize()
                graph_us = a2.elapsed_time(b2) * 1e3 / g_iters
                del g
            except Exception as e:  # capture refused: report the plain number only
                graph_us = f"capture failed: {e}"
            # each call alone after an L2 flush (a 512 MB write): DRAM-honest
            cold = []
            with torch.cuda.stream(stream):
                for _ in range(min(iters, 20)):
                    flush.zero_()
                    a3, b3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a3.record(stream)
                    cpt.cpt_slot_reduce(slots, dst, stream=stream)
                    b3.record(stream)
                    cold.append((a3, b3))
            torch.cuda.synchronize()
            cold_us = statistics.median(a3.elapsed_time(b3) for a3, b3 in cold) * 1e3
            gbs = (n_slots + 1) * nbytes / (cold_us * 1e-6) / 1e9
            line = {"sweep": "slot_reduce", "metric": "slot_reduce latency and effective GB/s",
                    "dtype": "f32" if dtype == torch.float32 else "bf16", "slots": n_slots,
                    "kernel_path": args.kernel_path,
                    "bytes_per_slot": nbytes, "iters": iters,
                    "us_per_call_launched": call_us, "us_per_call_c_abi": c_abi_us,
                    "us_per_call_graph": graph_us,
                    "us_per_call_cold_l2": cold_us,
                    "l2_resident_when_repeated": (n_slots + 1) * nbytes < 129 * 2**20,
                    "gbs": gbs, "frac_of_peak": gbs / peak, "peak": peak, "peak_source": peak_src}
            print(json.dumps(line), flush=True)
            del slots, dst
            torch.cuda.empty_cache()
    return 0


def main():
    global S, H, PATH
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-pieces", type=int, default=2,
                    help="pieces each of the 2P global chunks is cut into for the e2e pipeline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sample-tokens", type=int, default=16384,
                    help="tokens of the workload the CPU oracle processes per pass")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work, for each of the one-core and all-cores legs")
    ap.add_argument("--cpu-cores", type=int, default=0,
                    help="host cores for the all-cores oracle leg (0 = every core this process may use)")
    ap.add_argument("--reference-cores", type=int, default=0,
                    help="--impl reference: parallel oracle replicas (0 = every core)")
    ap.add_argument("--reference-budget", type=float, default=120.0,
                    help="target seconds for a whole --impl reference run")
    ap.add_argument("--fixed-sample", action="store_true",
                    help="--impl reference: use --sample-tokens as given")
    ap.add_argument("--path", choices=["fused", "staged"], default="fused",
                    help="gradient return as one fused launch (default) or as the staged "
                         "scatter / publish / wait / reduce flow on 2P streams")
    ap.add_argument("--next-rows", action="store_true",
                    help="instead of the step: restore, accumulate, P sweep, no-alloc and "
                         "partition-policy lines")
    ap.add_argument("--sweep", choices=["slot_reduce", "host_link", "grad_return_sizes"], default=None,
                    help="instead of the step: the slot-reduce message-size sweep, or the "
                         "host link's copy rates")
    ap.add_argument("--kernel-path", choices=["auto", "loads", "bulk"], default="auto",
                    help="kernel of the gradient return and the slot reduce: the measured rule "
                         "(default), or one forced")
    ap.add_argument("--slots", type=int, default=8, help="--sweep slot_reduce: number of slots (1..8)")
    ap.add_argument("--flush", choices=["write", "read"], default="write",
                    help="--sweep grad_return_sizes: flush L2 by writing or by reading 512 MB")
    ap.add_argument("--configs", default="all",
                    help="configuration rows timed after the step: all, none, or a comma list of "
                         + ", ".join(CONFIG_ROWS))
    ap.add_argument("--config-reps", type=int, default=20, help="timed launches per configuration row")
    ap.add_argument("--config-warmup", type=int, default=3, help="untimed launches per configuration row")
    ap.add_argument("--tokens", type=int, default=S, help="S (multiple of 2P)")
    ap.add_argument("--heads", type=int, default=H)
    args = ap.parse_args()
    S, H = args.tokens, args.heads
    PATH = args.path
    if S % (2 * P) or S <= 0 or H <= 0:
        ap.error("--tokens must be a positive multiple of 8, --heads positive")
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep == "slot_reduce":
        return run_slot_reduce_sweep(args)
    if args.sweep == "host_link":
        return run_host_link_sweep(args)
    if args.sweep == "grad_return_sizes":
        return run_grad_return_size_sweep(args)
    if args.next_rows:
        return run_next_rows(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
