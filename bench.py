#!/usr/bin/env python3
"""Benchmark: one decode step (reshape_and_cache + paged decode attention) of a
synthetic batch, timed on the GPU with CUDA events.

Default workload: the GQA 8B-shaped batch (256 sequences, 32 query / 8 kv
heads, head_dim 128, bf16, block size 16, context lengths lognormal with
median 1000 clipped to [16, 8192]).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 0-4]
                  [--split P] [--impl ours|reference] [--no-cpu-baseline]

Under torchrun (N > 1) each rank runs its own independently seeded batch
(replicas: sequences are independent, no data exchange); rank 0 prints the
aggregate over all ranks with the time of the slowest rank.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_230_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2, help="0 tiny, 1 mha7b, 2 gqa8b, 3 long_split, 4 prefix_fp8")
    ap.add_argument("--split", type=int, default=-1, help="partition size (0 = single pass; -1 = workload default)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-flush", action="store_true",
                    help="never flush L2 between steps (steady state; the shared-prefix workload reads from L2)")
    ap.add_argument("--separate", action="store_true",
                    help="time the scatter and the decode as two launches instead of pa_cache_and_decode")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--seqs", type=int, default=0, help="keep only the first N sequences (profiling runs)")
    ap.add_argument("--qlen", type=int, default=1, help="new query tokens per sequence (multi-token decode)")
    ap.add_argument("--block-size", type=int, default=16, help="KV block size of the prefill workload (8, 16, 32)")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"], help="cache dtype of the prefill workload")
    ap.add_argument("--head-dim", type=int, default=128, choices=[64, 128], help="head_dim of the prefill workload")
    ap.add_argument("--op", default="decode", choices=["decode", "blocks", "prefill", "l2read"],
                    help="blocks: time copy-on-write block copies and swap-out/in through pinned host memory; "
                         "l2read: measure the rate at which the SMs read an L2-resident buffer")
    ap.add_argument("--ref-budget", type=float, default=0.0,
                    help="reference arm: seconds of oracle work per step (default min(20, 120 / steps))")
    return ap.parse_args()


# --------------------------------------------------------------------------
# distributed plumbing (barrier and max over ranks only)
# --------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if _has_cuda() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def _has_cuda():
    import torch
    return torch.cuda.is_available()


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float, device=None) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, x: float, device=None) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t)
    return float(t.item())


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "25"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, begin: bool):
        """Brackets the timed region: only samples that arrive inside it count."""
        if begin:
            self.t0 = time.perf_counter()
        else:
            self.t1 = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons, watts = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t0", None), getattr(self, "t1", None)
        lines = [ln for t, ln in self.lines if t0 is None or t1 is None or t0 <= t <= t1 + 0.05]
        if not lines and self.lines:  # a region shorter than the sampling period: the nearest sample after it began
            later = [ln for t, ln in self.lines if t0 is None or t >= t0]
            lines = later[:1] if later else [self.lines[-1][1]]
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            try:
                watts.append(float(f[2]))
            except ValueError:
                pass
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w": statistics.median(watts) if watts else None}


# --------------------------------------------------------------------------
# roofline helpers
# --------------------------------------------------------------------------

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


DECODE_SOURCES = ("pa_decode.cuh", "pa_ptx.cuh", "pa_internal.h", "pa_decode_f16.cu", "pa_decode_bf16.cu",
                  "pa_decode_fp8.cu")


TC_SOURCES = ("pa_attn_tc.cu", "pa_attn_tc.h", "pa_tcgen05.cuh", "pa_ptx.cuh")


PREFILL_SOURCES = ("pa_prefill.cu", "pa_prefill_pair.cu", "pa_prefill.h", "pa_widen.cu", "pa_widen.h", "pa_tcgen05.cuh",
                   "pa_ptx.cuh")


def kernel_source_hash(sources=DECODE_SOURCES) -> str:
    """Hash of the sources a kernel is compiled from (the decode kernel's by default)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_230_gb300", "csrc")
    for name in sources:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def _profile_values(name: str, sources) -> dict:
    """The key: value lines of profiles/<name>.txt, or {} when the file is
    missing or was captured from other kernel sources than the current ones."""
    try:
        text = open(os.path.join(ROOT, "profiles", name + ".txt")).read()
    except OSError:
        return {}
    vals = {}
    for ln in text.splitlines():
        if ":" in ln:
            k, v = ln.split(":", 1)
            v = v.split()
            vals[k.strip()] = v[0] if v else ""
    return vals if vals.get("kernel_source_hash") == kernel_source_hash(sources) else {}


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch recorded by an ncu capture under profiles/, valid
    only while the kernel sources hash to the value recorded with it."""
    try:
        sources = TC_SOURCES if kernel.startswith("attn_tc") else DECODE_SOURCES
        return float(_profile_values("%s_%s" % (kernel, workload), sources)["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


def recorded_prefill_traffic(name: str, chunk: int, seqs: int, sources=PREFILL_SOURCES):
    """DRAM bytes of one prefill launch over `seqs` sequences with a `chunk`-token
    chunk at context 2 x chunk: the captured bytes per sequence (every
    sequence reads its own q, K and V and writes its own output) times seqs."""
    try:
        per_seq = float(_profile_values("%s_chunk%d" % (name, chunk), sources)["dram_bytes_per_sequence"])
    except (KeyError, ValueError):
        return None
    return per_seq * seqs


# --------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline object)
# --------------------------------------------------------------------------

def oracle_sample_time(wl: W.Workload, budget_s: float = 20.0, threads: int = 0):
    """Times the oracle (scatter + decode, on `threads` host threads, 0 = all)
    on a bounded sample of the batch: whole sequences in order until about
    `budget_s` of wall time has been spent; returns (seconds, kv_bytes, seqs,
    threads)."""
    import oracle
    threads = threads if threads > 0 else oracle.max_threads()
    if wl.kv_dtype == W.FP8:
        kc = np.zeros(wl.cache_shape(), np.uint8)
        vc = np.zeros(wl.cache_shape(), np.uint8)
        oracle.reshape_and_cache(wl.prefill_key, wl.prefill_value, wl.q_dtype, kc, vc, "fp8", wl.prefill_slots,
                                 wl.kv_scale)
    else:
        kc, vc = wl.k_cache, wl.v_cache
    total_t, total_b, nseq = 0.0, 0, 0
    chunk = max(1, wl.S // 16)
    i = 0
    while total_t < budget_s:  # passes over the batch, in order, until the budget is spent
        sel = np.arange(i, min(wl.S, i + chunk))
        sub = W.subset(wl, sel)
        t0 = time.perf_counter()
        oracle.reshape_and_cache(sub.key, sub.value, sub.q_dtype, kc, vc, sub.kv_dtype, sub.slot_mapping,
                                 sub.kv_scale)
        if sub.qlen == 1:
            oracle.decode(sub.q, sub.q_dtype, kc, vc, sub.kv_dtype, sub.block_tables, sub.context_lens, sub.scale,
                          sub.kv_scale, partition_size=sub.partition_size, num_threads=threads)
        else:
            # new token j of k attends causally to the prefix ending at its
            # position L - k + j: the oracle decodes it as its own query
            k = sub.qlen
            L = (sub.context_lens[:, None] - k + 1 + np.arange(k)[None, :]).reshape(-1)
            oracle.decode(sub.q.reshape(sub.S * k, sub.Hq, sub.D), sub.q_dtype, kc, vc, sub.kv_dtype,
                          np.repeat(sub.block_tables, k, axis=0), np.maximum(L, 0).astype(np.int32), sub.scale,
                          sub.kv_scale, partition_size=sub.partition_size, num_threads=threads)
        total_t += time.perf_counter() - t0
        total_b += sub.kv_bytes()
        nseq += len(sel)
        i = (i + chunk) % wl.S
    return total_t, total_b, nseq, threads


def unique_kv_bytes(wl: W.Workload) -> int:
    """KV bytes of the distinct physical blocks the batch reads."""
    return int(wl.notes.get("unique_blocks", 0)) * wl.Hkv * wl.bs * wl.D * 2 * W.ELEM_BYTES[wl.kv_dtype]


def workload_config(wl: W.Workload, P: int, world: int, fused: bool, no_flush: bool) -> dict:
    """The `config` object of a decode bench line, the same for both arms."""
    small = unique_kv_bytes(wl) < 4 * L2_BYTES
    return {"workload": wl.name, "num_seqs": wl.S, "q_heads": wl.Hq, "kv_heads": wl.Hkv,
            "head_dim": wl.D, "block_size": wl.bs, "kv_dtype": wl.kv_dtype, "new_tokens_per_seq": wl.qlen,
            "context_tokens": int(wl.context_lens.sum()), "max_context": wl.max_context_len,
            "kv_bytes_per_step": wl.kv_bytes(), "partition_size": P,
            "l2": ("no flush (steady state)" if small and no_flush else
                   "256 MiB L2 flush between steps" if small else "inputs larger than L2"),
            "parallelism": "replicas" if world > 1 else "single",
            "step": ("pa_cache_and_decode: scatter fused into the decode launch" if fused
                     else "pa_reshape_and_cache, then the decode call")}


def run_reference(args, wl, world, rank, pg):
    if rank != 0:
        return
    steps = max(1, args.steps)
    per_step = args.ref_budget if args.ref_budget > 0 else min(20.0, 120.0 / steps)
    secs, byts, nseq = 0.0, 0, 0
    threads = 1
    for _ in range(max(0, min(args.warmup, 1))):
        oracle_sample_time(wl, budget_s=min(0.5, per_step))
    for _ in range(steps):
        t, b, n, threads = oracle_sample_time(wl, budget_s=per_step)
        secs += t
        byts += b
        nseq += n
    gbs = byts / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, wl.partition_size if args.split < 0 else args.split, world,
                                  not args.separate, args.no_flush),
        "decode_tokens_per_s": nseq / secs,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": "fp64 C oracle (scatter + decode) over leading sequences of the batch, "
                                   "about %.0f s per step, %d sequences in total" % (per_step, nseq)},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def run_ours(args, wl, world, rank, local, pg):
    import torch
    from paged_kv_cache_230_gb300 import build as _build
    _build.build()
    from paged_kv_cache_230_gb300 import pagedattn as pa
    from paged_kv_cache_230_gb300.device import DeviceBatch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    P = wl.partition_size if args.split < 0 else args.split
    fused = not args.separate
    b = DeviceBatch(wl, dev, partition_size=P, fused=fused)
    stream = torch.cuda.current_stream(dev)
    kv_bytes = wl.kv_bytes()
    # the fused kernel also reads the new rows and writes them into the pool
    alg_bytes = wl.algorithmic_bytes() + (wl.scatter_bytes() if fused else 0)
    flush = None
    if unique_kv_bytes(wl) < 4 * L2_BYTES and not args.no_flush:
        flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)

    for _ in range(max(3, args.warmup)):
        b.step()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local) if not args.no_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(pg)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    if sampler:
        sampler.mark(True)
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 0xFF)
        e0, e1, e2 = ev[i]
        e0.record(stream)
        if fused:  # one launch
            b.step()
        else:
            b.scatter()
            e1.record(stream)
            b.decode()
        e2.record(stream)
    torch.cuda.synchronize(dev)
    barrier(pg)
    wall = time.perf_counter() - t_wall
    if sampler:
        sampler.mark(False)
    clocks = sampler.stop() if sampler else None
    step_ms = [e0.elapsed_time(e2) for e0, _, e2 in ev]
    dec_ms = [(e0 if fused else e1).elapsed_time(e2) for e0, e1, e2 in ev]
    sc_ms = None if fused else [e0.elapsed_time(e1) for e0, e1, _ in ev]
    total_ms = sum(step_ms)
    total_ms_max = max_over_ranks(pg, total_ms, dev)
    units = sum_over_ranks(pg, float(kv_bytes), dev)
    seqs = sum_over_ranks(pg, float(wl.S), dev)
    ms_per_step = total_ms_max / K
    value = units / (ms_per_step * 1e-3) / 1e9
    dec_avg = sum(dec_ms) / K
    peak, peak_kind = measured_hbm_peak()
    achieved = alg_bytes / (dec_avg * 1e-3) / 1e9
    kernel_name = ("decode_multi_split" if P else "decode_multi") if wl.qlen > 1 else ("decode_split" if P else "decode")
    if b.tensor_core_path():
        kernel_name = "attn_tc_split" if P else "attn_tc"
    elif fused:
        kernel_name = "cache_and_" + kernel_name
    traffic = recorded_traffic(wl.name, kernel_name)

    e2e = None
    if not args.no_e2e:
        e2e = e2e_measure(b, wl, dev, K=min(K, 200), warm=3, pg=pg)

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        t, byts, nseq, threads = oracle_sample_time(wl, budget_s=10.0)
        t1, byts1, nseq1, _ = oracle_sample_time(wl, budget_s=3.0, threads=1)
        cpu = {"value": byts / t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": "fp64 C oracle (scatter + decode) over %d sequences of the same %d-sequence batch, in "
                         "order with wrap-around (%.2f GB of KV), %.1f s" % (nseq, wl.S, byts / 1e9, t),
               "single_thread": {"value": byts1 / t1 / 1e9, "unit": "GB/s", "cores": 1,
                                 "sample": "%d sequences, %.2f GB of KV, %.1f s" % (nseq1, byts1 / 1e9, t1)}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if wl.q_dtype == "bf16" and wl.kv_dtype != W.FP8 else
                     ("e4m3-kv/bf16" if wl.kv_dtype == W.FP8 else "f16"),
            "data": "synthetic",
            "config": workload_config(wl, P, world, fused, args.no_flush),
            "decode_tokens_per_s": seqs / (ms_per_step * 1e-3),
            "pct_of_hbm_peak": 100.0 * value / peak,
            "decode_kernel_us": 1e3 * dec_avg,
            "decode_kernel_us_median": 1e3 * statistics.median(dec_ms),
            "decode_kernel_us_p10_p90": [1e3 * pct(dec_ms, 10), 1e3 * pct(dec_ms, 90)],
            "scatter_us": None if sc_ms is None else 1e3 * sum(sc_ms) / K,
            "scatter_gbs": None if sc_ms is None else wl.scatter_bytes() / (sum(sc_ms) / K * 1e-3) / 1e9,
            "wall_s": wall,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_source": peak_kind,
                         "kernel": "pa_" + kernel_name, "algorithmic_bytes_per_launch": alg_bytes},
            "gpu_launches": K * b.launches_per_step(),
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def pct(xs, q):
    """q-th percentile (nearest rank) of a list."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, int(round(q / 100.0 * (len(ys) - 1)))))]


def e2e_measure(b, wl, dev, K, warm, pg):
    """Same step through the public API with inputs in pinned host memory: the
    host->device copies of this step's q, new K/V rows, block tables, context
    lengths and slot ids, the scatter + decode, and the device->host copy of
    the output are all inside the timed region.  Steps are pipelined over two
    sets of device input/output buffers: a copy stream moves step i+1's inputs
    in and step i-1's output out while step i's kernels run (events order
    every buffer's reuse), so the copies overlap the kernels of other steps."""
    import torch
    names = ("q", "key", "value", "block_tables", "context_lens", "slot_mapping")
    sets = [b.io_set(), b.spare_io_set()]
    host = {n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype, pin_memory=True).copy_(sets[0][n])
            for n in names}
    outs_h = [torch.empty(sets[0]["out"].shape, dtype=sets[0]["out"].dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    compute = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in comp_done + d2h_done:
        e.record(compute)

    def run(n):
        with torch.cuda.stream(copy):  # inputs of step 0
            for name in names:
                sets[0][name].copy_(host[name], non_blocking=True)
            h2d_done[0].record(copy)
        for i in range(n):
            j = i % 2
            compute.wait_event(h2d_done[j])
            compute.wait_event(d2h_done[j])  # step i - 2's output has left this buffer
            b.bind(sets[j])
            b.step()
            comp_done[j].record(compute)
            with torch.cuda.stream(copy):
                if i + 1 < n:  # step i + 1's inputs, once step i - 1 is done with that set
                    nj = (i + 1) % 2
                    copy.wait_event(comp_done[nj])
                    for name in names:
                        sets[nj][name].copy_(host[name], non_blocking=True)
                    h2d_done[nj].record(copy)
                copy.wait_event(comp_done[j])
                outs_h[j].copy_(sets[j]["out"], non_blocking=True)
                d2h_done[j].record(copy)
        compute.wait_stream(copy)
        b.bind(sets[0])

    run(warm)
    torch.cuda.synchronize(dev)
    barrier(pg)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    run(K)
    e1.record(compute)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(pg, e0.elapsed_time(e1), dev) / K
    units = sum_over_ranks(pg, float(wl.kv_bytes()), dev)
    return {"value": units / (ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms,
            "pipelining": "two buffer sets; copies on a second stream overlap other steps' kernels"}


def run_l2read(args, local):
    """The L2 -> SM read rate: a 64 MiB buffer (half of L2) read once, then
    timed over launches of pa_probe_l2_read with plain 16-byte loads (mode 0)
    and with the 2 KB TMA boxes the attention kernels load K/V with (mode 1).
    Median and best of 7 launches of about 12 GB each; no setting changed."""
    import torch
    from paged_kv_cache_230_gb300 import build as _build
    _build.build()
    from paged_kv_cache_230_gb300 import pagedattn as pa
    torch.cuda.set_device(local)
    nbytes = 64 << 20
    buf = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(16, dtype=torch.uint8, device="cuda")
    nsm = torch.cuda.get_device_properties(local).multi_processor_count
    sampler = ClockSampler(local) if not args.no_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
        sampler.mark(True)
    res = {}
    for mode, iters in ((0, 192), (1, max(1, int(12e9 / (nsm * 32768))))):
        for _ in range(2):
            pa.probe_l2_read(buf, mode, iters, sink)
        torch.cuda.synchronize()
        rates = []
        for _ in range(7):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            nread = pa.probe_l2_read(buf, mode, iters, sink)
            e1.record()
            torch.cuda.synchronize()
            rates.append(nread / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        res[mode] = (statistics.median(rates), max(rates), nread)
    if sampler:
        sampler.mark(False)
    clocks = sampler.stop() if sampler else None
    assert pa.get_device_error() == 0
    line = {"metric": "L2 -> SM read bandwidth", "value": res[0][0], "unit": "GB/s", "n_gpus": 1, "steps": 7,
            "higher_is_better": True, "dtype": "u8", "data": "synthetic",
            "config": {"workload": "l2_resident_buffer", "buffer_bytes": nbytes, "bytes_per_launch_plain": res[0][2],
                       "bytes_per_launch_tma": res[1][2]},
            "plain_loads_gbs": {"median": res[0][0], "best": res[0][1]},
            "tma_boxes_gbs": {"median": res[1][0], "best": res[1][1]},
            "clocks": clocks, "gpu_launches": 14}
    print(json.dumps(line), flush=True)


def run_blocks(args, local):
    """Whole-block moves on the gqa8b pool shape (8 kv heads x 16 tokens x 128
    channels, bf16: 32 KiB per block per cache): pa_copy_blocks of 4096
    disjoint (src, dst) pairs, then pa_gather_blocks into pinned host memory
    and pa_scatter_blocks back from it for 4096 blocks.  GB/s counts bytes
    read plus bytes written."""
    import torch
    from paged_kv_cache_230_gb300 import build as _build
    _build.build()
    from paged_kv_cache_230_gb300 import pagedattn as pa
    torch.cuda.set_device(local)
    NB, Hkv, bs, D, n = 16384, 8, 16, 128, 4096
    kc = torch.randn((NB, Hkv, bs, D), device="cuda").to(torch.bfloat16)
    vc = torch.randn_like(kc)
    perm = torch.randperm(NB, device="cuda")
    pairs = torch.stack([perm[:n], perm[n:2 * n]], dim=1).contiguous()
    ids = perm[2 * n:3 * n].contiguous()
    host = torch.empty((n, 2, Hkv, bs, D), dtype=torch.bfloat16, pin_memory=True)
    block = Hkv * bs * D * 2
    moved = 2 * n * block  # K and V blocks per call
    res = {}
    sampler = ClockSampler(local) if not args.no_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
        sampler.mark(True)
    for name, fn in (("copy_blocks", lambda: pa.copy_blocks(kc, vc, pairs)),
                     ("gather_to_host", lambda: pa.gather_blocks(host, kc, vc, ids)),
                     ("scatter_from_host", lambda: pa.scatter_blocks(kc, vc, host, ids))):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        K = max(1, min(args.steps, 200))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            fn()
        e1.record()
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / K
        res[name] = {"us": us, "gbs": 2 * moved / (us * 1e-6) / 1e9}
    if sampler:
        sampler.mark(False)
    clocks = sampler.stop() if sampler else None
    # KV fragmentation of the host block manager on the gqa8b length mix:
    # unused tail slots over all slots of the blocks the sequences hold
    lens = W.config_lengths(2, 2)
    bm = pa.BlockManager(int(sum(-(-int(x) // bs) for x in lens)), bs)
    for sid, x in enumerate(lens):
        bm.add_sequence(sid, int(x))
    res["fragmentation_gqa8b"] = bm.tail_waste() / ((bm.num_blocks - bm.num_free_blocks()) * bs)
    peak, kind = measured_hbm_peak()
    line = {"metric": "block copy GB/s (read + write)", "value": res["copy_blocks"]["gbs"], "unit": "GB/s",
            "n_gpus": 1, "steps": min(args.steps, 200), "warmup": args.warmup, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "blocks_gqa8b_pool", "blocks_per_call": n, "block_bytes_per_cache": block},
            "ops": res, "clocks": clocks,
            "roofline": {"bound": "hbm", "achieved": res["copy_blocks"]["gbs"], "peak": peak, "unit": "GB/s",
                         "frac": res["copy_blocks"]["gbs"] / peak, "peak_source": kind, "kernel": "pa_copy_blocks"}}
    print(json.dumps(line), flush=True)


def measured_tensor_peak(sustained: bool = False):
    """bf16 tensor peak: the burst figure, or the sustained one (a seconds-long
    loop under the power cap) for kernels timed inside a long loop."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        if sustained and "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured (sustained)"
        return float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return (1700.0, "fallback (sustained)") if sustained else (1900.0, "fallback")


def run_prefill(args, local):
    """Chunked prefill of a GQA 8B-shaped batch through pa_prefill: by default
    16 sequences, each with a chunk of 2048 new tokens at the end of a
    4096-token context (32/8 heads, head_dim 128, bf16, block size 16);
    --seqs and --qlen change the batch and the chunk (context = 2 x chunk),
    --kv-dtype fp8 stores the caches in E4M3 (per-tensor scale) and
    --head-dim 64 halves the head.  TFLOP/s counts the causal work only:
    4 * D * Hq * sum over query rows of (position + 1)."""
    import torch
    from paged_kv_cache_230_gb300 import build as _build
    _build.build()
    from paged_kv_cache_230_gb300 import pagedattn as pa
    from paged_kv_cache_230_gb300.device import DeviceBatch
    torch.cuda.set_device(local)
    S = args.seqs if args.seqs > 0 else 16
    C = args.qlen if args.qlen > 1 else 2048
    L = 2 * C
    bs = getattr(args, "block_size", 16)
    kv = W.FP8 if getattr(args, "kv_dtype", "bf16") == "fp8" else W.BF16
    wl = W.make_prefill_workload(S=S, C=C, bs=bs, kv_dtype=kv, D=getattr(args, "head_dim", 128))
    b = DeviceBatch(wl, "cuda")
    pos = np.arange(L - C, L, dtype=np.float64)
    flops = 4.0 * wl.D * wl.Hq * S * float((pos + 1).sum())
    # an even group goes to the head-pair kernel (head_dim 64 or 128; E4M3
    # caches widened to the q dtype first), an odd one to the one-head kernel
    # (16-bit, head_dim 128) or the tensor-core kernel with the GQA heads
    # packed in rows
    even = (wl.Hq // wl.Hkv) % 2 == 0
    per_head = even or (kv != W.FP8 and wl.D == 128)
    if even:
        kernel = "pa_prefill (widen_kv_kernel, prefill_pair_kernel)" if kv == W.FP8 else "pa_prefill (prefill_pair_kernel)"
    elif per_head:
        kernel = "pa_prefill (prefill_kernel)"
    else:
        kernel = "pa_prefill (attn_tc_kernel)"
    sources = PREFILL_SOURCES if per_head else TC_SOURCES

    # the E4M3 widening's workspace, allocated once outside the timed region
    need = pa.prefill_workspace_size(S, b.block_tables.shape[1], b.k_cache)
    ws = torch.empty(need, dtype=torch.uint8, device=b.k_cache.device) if need > 0 else None

    def run():
        pa.prefill(b.out, b.q, b.k_cache, b.v_cache, b.block_tables, b.context_lens, wl.scale, wl.kv_scale,
                   workspace=ws)

    for _ in range(max(3, args.warmup)):
        run()
    torch.cuda.synchronize()
    # time enough launches to fill about two seconds, so that the clock
    # sampler sees the kernel under load for many periods
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        run()
    e1.record()
    torch.cuda.synchronize()
    est_ms = max(1e-3, e0.elapsed_time(e1) / 3)
    K = max(1, args.steps) if args.no_clocks else max(1, args.steps, min(20000, int(2000.0 / est_ms)))
    sampler = ClockSampler(local) if not args.no_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
        sampler.mark(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        run()
    e1.record()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(False)
    clocks = sampler.stop() if sampler else None
    us = 1e3 * e0.elapsed_time(e1) / K
    tflops = flops / (us * 1e-6) / 1e12
    # the timed region is about two seconds of back-to-back launches under
    # the power cap, so the sustained peak is the denominator; the burst
    # fraction is reported beside it
    peak, kind = measured_tensor_peak(sustained=True)
    burst, _ = measured_tensor_peak()
    line = {"metric": "paged prefill attention TFLOP/s (causal FLOPs)", "value": tflops, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": K, "warmup": args.warmup, "higher_is_better": True,
            # E4M3 blocks are widened exactly to the q dtype (bf16) for the
            # head-pair kernel; the packed-group kernel widens them to f16
            "dtype": "bf16" if (even or kv != W.FP8) else "f16",
            "data": "synthetic", "config": {"workload": wl.name, "num_seqs": S, "chunk": C, "context": L,
                                            "q_heads": 32, "kv_heads": 8, "head_dim": wl.D, "block_size": bs,
                                            "kv_dtype": wl.kv_dtype},
            "prefill_us": us, "tokens_per_s": S * C / (us * 1e-6), "clocks": clocks,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "peak_source": kind, "frac_of_burst_peak": tflops / burst,
                         "traffic": recorded_prefill_traffic(wl.name, C, S, sources), "kernel": kernel}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local, pg = dist_setup()
    if args.op in ("blocks", "prefill", "l2read"):
        if rank == 0:
            {"blocks": run_blocks, "prefill": run_prefill, "l2read": run_l2read}[args.op](args, local)
        return
    if args.impl == "reference" and rank != 0:
        return
    seed = args.config + 1000 * rank  # replicas draw independent batches
    wl = W.make_config(args.config, seed=seed, qlen=args.qlen)
    if args.seqs and args.seqs < wl.S:
        name = "%s_first%d" % (wl.name, args.seqs)
        wl = W.subset(wl, np.arange(args.seqs))
        wl.name = name
    if args.impl == "reference":
        run_reference(args, wl, world, rank, pg)
    else:
        run_ours(args, wl, world, rank, local, pg)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
