#!/usr/bin/env python3
"""Benchmark of paged GQA decode attention on GB300.

One step = one decode_attn_paged call (split kernel + combine kernel) over the whole batch
of the large ragged workload: B=128 sequences, Hq=32, Hkv=8, D=128, kv_len ~ U{256..4096},
page_size 16, pages assigned by a seeded shuffle of a 2x pool.  Inputs are resident in HBM
before the timed region; two (or more) independent copies of every input are rotated so
that the bytes touched between two reads of the same copy exceed 2x L2 (cold KV).

Printed (rank 0, one JSON line): achieved HBM GB/s of algorithmic bytes (K/V rows inside
seq_lens, q, out, the block-table entries used, seq_lens) per step time, with the split
kernel's own roofline, an end-to-end figure through host buffers, the fp64 oracle on a
bounded sample of the same workload on the host cores, and the SM clocks seen meanwhile.

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference] [--workload W]

With N > 1 (torchrun, one process per GPU) every rank runs an independent replica (the
path has no cross-GPU exchange); value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

FALLBACK_HBM_GBS = 6800.0


# ---- helpers -----------------------------------------------------------------------------

def rank_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class ClockSampler:
    """nvidia-smi samples (20 ms) of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"dap_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.idx), "-lms", "20"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 9:
                    continue
                try:
                    sm.append(float(c[1]))
                    mx = float(c[2])
                except ValueError:
                    continue
                for n, v in zip(names, c[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


KERNEL_SOURCES = {"split_kernel": ("dap_decode.cu", "dap_tile.cuh", "dap_device.cuh", "dap_internal.h"),
                  "multi_kernel": ("dap_multi.cu", "dap_tile.cuh", "dap_device.cuh", "dap_internal.h"),
                  "fp8kv_kernel": ("dap_fp8kv.cu", "dap_tile.cuh", "dap_device.cuh", "dap_internal.h"),
                  "swa_kernel": ("dap_fp8.cu", "dap_device.cuh", "dap_internal.h")}


def kernel_source_sha(kernel: str) -> str:
    """Hash of the sources a kernel is built from (a recorded ncu figure is only reported
    while they are unchanged)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_298_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    kernel source for this workload; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(kernel, {}).get(workload_key)
        if e and e.get("source_sha") == kernel_source_sha(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def workload_key(args) -> str:
    """Key of the workload in the recorded-traffic table (the batch size when not the default)."""
    return args.workload if not getattr(args, "batch", 0) else f"{args.workload}_b{args.batch}"


def job_throughput(ms_list, nbytes_per_rank, world, device):
    """Whole-job GB/s for each timing in ms_list: every rank processed nbytes_per_rank, and
    the job took as long as its slowest rank (max over ranks of each timing).  Returns
    [(GB/s, max ms), ...].  With world > 1 it needs an initialised process group."""
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in ms_list], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [(world * nbytes_per_rank / (m * 1e-3) / 1e9, m) for m in t.tolist()]


# ---- workloads ---------------------------------------------------------------------------

def make_workload(name: str, device, batch=None):
    from paged_kv_cache_298_gb300 import inputs
    if name == "ragged":
        return inputs.ragged_paged(device=device, B=batch or 128)
    if name == "llama":
        return inputs.llama_paged(device=device)
    if name in ("long1", "long4"):
        return inputs.long_paged(B=int(name[-1]), device=device)
    raise SystemExit(f"unknown workload {name}")


def algorithmic_bytes(case, rows=None) -> int:
    """K/V rows inside seq_lens + q + out + block-table entries used + seq_lens.
    `rows`: restrict to these sequences (for a CPU sample)."""
    lens = case.seq_lens.cpu().to(torch.int64)
    if rows is not None:
        lens = lens[rows]
    B = lens.numel()
    kv = int(lens.sum()) * case.Hkv * case.D * 2 * 2
    qo = 2 * B * case.Hq * case.D * 2
    pages = int(((lens + case.page_size - 1) // case.page_size).sum()) * 4
    return kv + qo + pages + B * 4


def workload_config(case, S, copies, footprint):
    lens = case.seq_lens.cpu()
    return {"workload": case.name, "B": case.B, "Hq": case.Hq, "Hkv": case.Hkv, "D": case.D,
            "page_size": case.page_size, "kv_len_min": int(lens.min()), "kv_len_max": int(lens.max()),
            "total_kv": int(lens.to(torch.int64).sum()), "num_splits": S, "kv_dtype": "bf16",
            "cold_kv": f"{copies} rotated input copies of {footprint / 1e9:.2f} GB each (> 2x L2)"}


# ---- the CPU oracle (reference arm and cpu_baseline) -------------------------------------

class OracleRunner:
    def __init__(self, case):
        import oracle
        self.oracle = oracle
        self.case = case
        self.q = bits(case.q)
        self.k = bits(case.k_cache)
        self.v = bits(case.v_cache)
        self.table = case.block_table.cpu().numpy()
        self.lens = case.seq_lens.cpu().numpy()

    def run(self, rows):
        """Oracle on the sequences `rows` (all heads).  Returns seconds."""
        c = self.case
        q = np.ascontiguousarray(self.q[rows])
        t0 = time.perf_counter()
        self.oracle.decode_paged(q, self.k, self.v, np.ascontiguousarray(self.table[rows]),
                                 np.ascontiguousarray(self.lens[rows]), c.scale)
        return time.perf_counter() - t0

    def sample_rows(self, target_s: float):
        """A prefix of the batch sized for about target_s seconds of oracle time."""
        n = 1
        dt = self.run(np.arange(1))
        B = self.case.B
        n = int(max(1, min(B, target_s / max(dt, 1e-4))))
        return np.arange(n)


def repeat_for(run, target_s=10.0):
    """Call run() (which returns its own seconds) until about target_s seconds of CPU work
    have accumulated; returns (mean seconds per pass, passes)."""
    total, n = 0.0, 0
    while n == 0 or total < target_s:
        total += run()
        n += 1
    return total / n, n


def cpu_baseline(case, target_s=10.0, single_s=3.0):
    """The oracle on the host cores (OpenMP over all of them), plus the same oracle on one
    thread over a smaller sample."""
    r = OracleRunner(case)
    rows = r.sample_rows(target_s)
    dt, passes = repeat_for(lambda: r.run(rows), target_s)
    nbytes = algorithmic_bytes(case, torch.as_tensor(rows))
    cores = r.oracle.num_threads()
    r.oracle.set_num_threads(1)
    try:
        rows1 = r.sample_rows(single_s)
        dt1, passes1 = repeat_for(lambda: r.run(rows1), single_s)
    finally:
        r.oracle.set_num_threads(cores)
    nbytes1 = algorithmic_bytes(case, torch.as_tensor(rows1))
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle (OpenMP) on sequences 0..{len(rows) - 1} of {case.B} (all heads), "
                      f"{passes} passes of {dt:.2f} s",
            "single_thread": {"value": nbytes1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"sequences 0..{len(rows1) - 1}, {passes1} passes of {dt1:.2f} s"}}


# ---- our arm -----------------------------------------------------------------------------

def run_ours(args):
    from paged_kv_cache_298_gb300 import binding
    import torch.distributed as dist

    rank, local, world = rank_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    binding.load()
    case = make_workload(args.workload, dev, args.batch)
    hbm_peak, peak_src = peaks()
    sms = binding.device_sm_count()
    S = args.splits if args.splits >= 0 else binding.plan_splits(
        sms, case.B, case.Hq, case.Hkv, case.D, case.page_size, case.max_kv_len, case.total_kv)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    footprint = sum(t.numel() * t.element_size() for t in (case.q, case.k_cache, case.v_cache,
                                                           case.block_table, case.seq_lens))
    copies = 1 + max(1, math.ceil(2 * l2 / footprint))
    sets = [case] + [type(case)(case.q.clone(), case.k_cache.clone(), case.v_cache.clone(),
                                case.block_table.clone(), case.seq_lens.clone(), case.page_size, case.scale,
                                case.name) for _ in range(copies - 1)]
    ws = [torch.empty(max(1, binding.workspace_bytes(case.B, case.Hq, case.Hkv, case.D, S)), dtype=torch.uint8,
                      device=dev)
          for _ in sets]
    outs = [torch.empty_like(case.q) for _ in sets]
    maxlen = case.max_kv_len
    stream = torch.cuda.current_stream()

    def step(i):
        c = sets[i % copies]
        binding.decode_attn_paged(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens, max_kv_len=maxlen,
                                  scale=c.scale, num_splits=S, workspace=ws[i % copies], out=outs[i % copies])

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if binding.get_device_errors(clear=True):
        raise SystemExit("device error word set during warm-up")

    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start.record(stream)
    for i in range(K):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = t_start.elapsed_time(t_end) / K

    # the split kernel's own duration: events around each launch (a separate loop, because an
    # event between the two kernels stops the combine from overlapping the split kernel's tail)
    KT = min(K, 50)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(KT)]
    for e in ev:   # torch creates the CUDA event on first record; the trace hook needs the handle
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    for i in range(KT):
        binding.set_trace_events(*ev[i])
        step(i)
    torch.cuda.synchronize()
    binding.set_trace_events()
    split_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    combine_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    errs = binding.get_device_errors(clear=True)

    # end to end through host buffers: q, block table and seq_lens in, out back, every step
    from paged_kv_cache_298_gb300 import binding as b2
    hq = case.q.cpu().pin_memory()
    ht = case.block_table.cpu().pin_memory()
    hl = case.seq_lens.cpu().pin_memory()
    ho = torch.empty(case.q.shape, dtype=torch.bfloat16).pin_memory()
    dq = [s.q for s in sets]
    dt_ = [s.block_table for s in sets]
    dl = [s.seq_lens for s in sets]

    def h2d(i):
        j = i % copies
        dq[j].copy_(hq, non_blocking=True)
        dt_[j].copy_(ht, non_blocking=True)
        dl[j].copy_(hl, non_blocking=True)

    def call(i):
        j = i % copies
        c = sets[j]
        b2.decode_attn_paged(dq[j], c.k_cache, c.v_cache, dt_[j], dl[j], max_kv_len=maxlen, scale=c.scale,
                             num_splits=S, workspace=ws[j], out=outs[j])

    def d2h(i):
        ho.copy_(outs[i % copies], non_blocking=True)

    e2e_ms, e2e_sched = time_e2e(h2d, call, d2h, K, args.warmup, copies, stream, world)

    nbytes = algorithmic_bytes(case)
    (value, ms), (e2e_value, e2e_ms) = job_throughput([ms, e2e_ms], nbytes, world, dev)
    achieved = nbytes / (split_ms * 1e-3) / 1e9
    line = {
        "metric": "paged decode attention achieved HBM GB/s (algorithmic bytes), cold KV",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "us_per_call": round(ms * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(case, S, copies, footprint),
        "pct_of_peak": round(100 * value / world / hbm_peak, 1),
        "roofline": {"bound": "hbm", "kernel": "split_kernel", "achieved": round(achieved, 1),
                     "peak": hbm_peak, "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "split_kernel_ms": round(split_ms, 5),
                     "combine_ms": round(combine_ms, 5), "algorithmic_bytes_per_launch": nbytes,
                     "traffic": recorded_traffic("split_kernel", workload_key(args))},
        "e2e": {"schedule": e2e_sched, "value": round(e2e_value, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": hq.numel() * 2 + ht.numel() * 4 + hl.numel() * 4,
                "d2h_bytes_per_step": ho.numel() * 2},
        "gpu_launches": K * (2 if S != 1 else 1),
        "device_errors": errs,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---- fp8 sliding-window latent decode -----------------------------------------------------

def fp8_counts(case):
    """Participating rows per token (j < min(len, W), slot >= 0), from the inputs."""
    idx = case.indices.cpu()
    lens = case.lens.cpu().clamp(min=0, max=case.W)
    j = torch.arange(case.W)[None, :]
    return ((j < lens[:, None]) & (idx >= 0)).sum(dim=1)


def fp8_algorithmic(case):
    """Bytes: q + out + every participating fp8 row and its bf16 inverse scale + the slot
    table + lens.  Flops: QK^T and PV, 2 * 2 * NH * rows * HD per token."""
    n = fp8_counts(case)
    rows = int(n.sum())
    nbytes = 2 * case.T * case.NH * case.HD * 2 + rows * (case.HD + 2) + case.T * case.W * 8 + case.T * 8
    flops = 4 * case.NH * case.HD * rows
    return nbytes, flops, rows


def run_fp8(args):
    from paged_kv_cache_298_gb300 import binding, inputs
    rank, local, world = rank_info()
    import torch.distributed as dist
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    binding.load()
    case = inputs.fp8_swa(device=dev)
    hbm_peak, peak_src = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    parts = (case.q, case.kv_cache, case.inv_scale, case.indices, case.lens)
    footprint = sum(t.numel() * t.element_size() for t in parts) + case.q.numel() * 2
    copies = 1 + max(1, math.ceil(2 * l2 / footprint))
    sets = [parts] + [tuple(t.clone() for t in parts) for _ in range(copies - 1)]
    outs = [torch.empty_like(case.q) for _ in sets]
    stream = torch.cuda.current_stream()

    def step(i):
        q, kv, inv, idx, ln = sets[i % copies]
        binding.decode_attn_paged_fp8(q, kv, inv, idx, ln, scale=case.scale, out=outs[i % copies])

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0.record(stream)
    for i in range(K):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / K
    # the kernel's own time: one launch per call, so a CUDA graph of 50 calls replayed gives
    # the device time per launch without the Python binding's host cost between launches
    per = 50
    graph = torch.cuda.CUDAGraph()
    gs = torch.cuda.Stream()
    gs.wait_stream(stream)
    with torch.cuda.stream(gs):
        with torch.cuda.graph(graph, stream=gs):
            for i in range(per):
                step(i)
    stream.wait_stream(gs)
    graph.replay()
    torch.cuda.synchronize()
    reps = max(1, K // per)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(reps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    kern_ms = g0.elapsed_time(g1) / (reps * per)
    errs = binding.get_device_errors(clear=True)
    nbytes, flops, rows = fp8_algorithmic(case)

    # end to end: q, the slot table and the lengths in from pinned host memory, out back
    hq = case.q.cpu().pin_memory()
    hidx = case.indices.cpu().pin_memory()
    hln = case.lens.cpu().pin_memory()
    ho = torch.empty(case.q.shape, dtype=torch.bfloat16).pin_memory()

    def h2d(i):
        q, kv, inv, idx, ln = sets[i % copies]
        q.copy_(hq, non_blocking=True)
        idx.copy_(hidx, non_blocking=True)
        ln.copy_(hln, non_blocking=True)

    def call(i):
        j = i % copies
        q, kv, inv, idx, ln = sets[j]
        binding.decode_attn_paged_fp8(q, kv, inv, idx, ln, scale=case.scale, out=outs[j])

    def d2h(i):
        ho.copy_(outs[i % copies], non_blocking=True)

    e2e_ms, e2e_sched = time_e2e(h2d, call, d2h, K, args.warmup, copies, stream, world)
    if world > 1:
        dist.barrier()
    (value, ms), (e2e_value, e2e_ms) = job_throughput([ms, e2e_ms], nbytes, world, dev)
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    line = {
        "metric": "fp8 sliding-window latent decode achieved HBM GB/s (algorithmic bytes), cold inputs",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "us_per_call": round(ms * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": case.name, "T": case.T, "NH": case.NH, "HD": case.HD, "W": case.W,
                   "num_blocks": case.num_blocks, "block_size": case.block_size, "rows": rows,
                   "kv_dtype": "fp8-e4m3", "cold": f"{copies} rotated input copies of {footprint / 1e6:.1f} MB"},
        "roofline": {"bound": "hbm", "kernel": "swa_kernel", "achieved": round(achieved, 1), "peak": hbm_peak,
                     "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "kernel_ms": round(kern_ms, 5), "kernel_timing": "CUDA graph of 50 calls, replayed",
                     "algorithmic_bytes_per_launch": nbytes,
                     "tflops": round(flops / (kern_ms * 1e-3) / 1e12, 2),
                     "traffic": recorded_traffic("swa_kernel", "fp8")},
        "e2e": {"schedule": e2e_sched, "value": round(e2e_value, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": hq.numel() * 2 + hidx.numel() * 8 + hln.numel() * 8,
                "d2h_bytes_per_step": ho.numel() * 2},
        "gpu_launches": K, "device_errors": errs, "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        cq, ckv, cinv, cidx, cln = (t.cpu() for t in parts)
        a = (bits(cq), ckv.numpy(), bits(cinv), cidx.numpy(), cln.numpy(), case.block_size, case.scale)
        passes, tt = 0, time.perf_counter()
        while True:   # whole passes over all tokens until about 10 s of CPU work
            oracle.fp8_swa(*a)
            passes += 1
            if time.perf_counter() - tt > 10.0:
                break
        dt = (time.perf_counter() - tt) / passes
        line["cpu_baseline"] = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
                                "kind": "oracle", "sample": f"fp64 oracle (OpenMP), all {case.T} tokens, "
                                                            f"{passes} passes, {dt * 1e3:.1f} ms each"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---- cache appends (the step before decode) ----------------------------------------------

def run_append(args):
    """Times the two append kernels on the decode step of the ragged batch (one new token
    per sequence: B=128 x Hkv=8 rows of D=128) and of the fp8 workload (T=64 latent rows of
    HD=512).  Bytes: new rows read + cache rows written + the indices they go through."""
    from paged_kv_cache_298_gb300 import binding, inputs
    dev = torch.device("cuda", 0)
    binding.load()
    case = inputs.ragged_paged(device=dev)
    g = torch.Generator(device=dev).manual_seed(298010)
    k_new = inputs.randn_bf16((case.B, case.Hkv, case.D), g, dev)
    v_new = inputs.randn_bf16((case.B, case.Hkv, case.D), g, dev)
    pos = case.seq_lens.clone()   # one past the end; every table has room (2x pool, full pages)
    pos = torch.minimum(pos, torch.tensor(case.max_pages * case.page_size - 1, device=dev, dtype=torch.int32))
    f = inputs.fp8_swa(device=dev)
    rows = inputs.randn_bf16((f.T, f.HD), g, dev)
    slots = torch.randperm(f.num_blocks * f.block_size, generator=torch.Generator().manual_seed(298011))[:f.T]
    slots = slots.to(torch.int64).to(dev)
    K, W = args.steps, args.warmup

    def timed(fn):
        """Device time per call: the calls are captured in a CUDA graph of 50 and replayed, so
        the Python binding's host cost (about 10 us a call) does not starve the GPU."""
        for _ in range(W):
            fn()
        torch.cuda.synchronize()
        graph, per = torch.cuda.CUDAGraph(), 50
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                for _ in range(per):
                    fn()
        torch.cuda.current_stream().wait_stream(s)
        graph.replay()
        torch.cuda.synchronize()
        reps = max(1, K // per)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * per)

    ms_paged = timed(lambda: binding.kv_append_paged(k_new, v_new, case.k_cache, case.v_cache, case.block_table, pos))
    ms_fp8 = timed(lambda: binding.kv_append_fp8(rows, f.kv_cache, f.inv_scale, slots))
    b_paged = 2 * 2 * k_new.numel() * 2 + case.B * 4 * 2
    b_fp8 = rows.numel() * 2 + rows.numel() + f.T * (2 + 8)
    hbm_peak, peak_src = peaks()
    print(json.dumps({
        "metric": "paged KV append achieved HBM GB/s (algorithmic bytes)",
        "value": round(b_paged / (ms_paged * 1e-3) / 1e9, 1), "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_step": round(ms_paged, 5), "us_per_call": round(ms_paged * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "append one decode token: ragged B=128 Hkv=8 D=128 page 16; fp8 T=64 HD=512",
                   "bytes_per_call": b_paged},
        "fp8_append": {"us_per_call": round(ms_fp8 * 1e3, 2), "bytes_per_call": b_fp8,
                       "GB/s": round(b_fp8 / (ms_fp8 * 1e-3) / 1e9, 1)},
        "roofline": {"bound": "latency", "peak": hbm_peak, "peak_source": f"{peak_src} hbm_gbs",
                     "note": "a 1 MB / 0.1 MB problem: launch and memory latency, not HBM bandwidth, set the time"},
        "timing": "CUDA graph of 50 calls, replayed",
        "gpu_launches": 2 * 50 * max(1, K // 50), "device_errors": binding.get_device_errors()}), flush=True)


# ---- end to end through host buffers ------------------------------------------------------

def time_e2e(h2d, compute, d2h, K, W, copies, stream, world=1):
    """Milliseconds per end-to-end step and the schedule that gave them.  Step i copies its
    inputs in from pinned host memory (`h2d(i)`), runs the library call (`compute(i)`, on
    `stream`) and copies its result back (`d2h(i)`); every step does all three inside the
    timed region.  Two schedules are timed and the faster is reported, as a serving loop
    would pick: "serial" (all three on `stream`, step after step: the fewest host calls,
    best when a step is host-bound) and "pipelined" (the copies in on one stream, the
    kernels on `stream`, the copies out on a third, so that step i + 1's inputs and step
    i - 1's result travel while step i computes; step i's kernels wait for its inputs, the
    device slot i % copies is refilled only after step i - copies has read it and its
    output overwritten only after that step's result was copied out)."""
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def events(n):  # created (torch does so on first record) before the timed region
        ev = [torch.cuda.Event(enable_timing=False) for _ in range(n)]
        for e in ev:
            e.record(stream)
        return ev

    def serial(n):
        for i in range(n):
            h2d(i)
            compute(i)
            d2h(i)

    def pipelined(n, ready, done, read, start):
        start.record(stream)
        up.wait_event(start)
        down.wait_event(start)
        for i in range(n):
            with torch.cuda.stream(up):
                if i >= copies:
                    up.wait_event(done[i - copies])
                h2d(i)
                ready[i].record(up)
            stream.wait_event(ready[i])
            if i >= copies:
                stream.wait_event(read[i - copies])
            compute(i)
            done[i].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(done[i])
                d2h(i)
                read[i].record(down)
        stream.wait_event(read[n - 1])

    def timed(fn, *ev):
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn(K, *ev)
        e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return e0.elapsed_time(e1) / K

    serial(W)
    pipelined(W, events(W), events(W), events(W), events(1)[0])
    res = {"serial": timed(serial),
           "pipelined": timed(pipelined, events(K), events(K), events(K), events(1)[0])}
    if world > 1:  # every rank reports the schedule rank 0 found faster
        pick = torch.tensor([0 if res["serial"] <= res["pipelined"] else 1], dtype=torch.int32,
                            device=torch.device("cuda", torch.cuda.current_device()))
        dist.broadcast(pick, 0)
        best = "serial" if int(pick.item()) == 0 else "pipelined"
    else:
        best = min(res, key=res.get)
    return res[best], best


# ---- shared single-GPU measurement of a decode step ------------------------------------------

def measure_step(binding, step, e2e, K, W, stream, copies):
    """Times `step(i)` (inputs resident, rotated copies chosen by the caller): K untraced steps
    bracketed by CUDA events with the clocks sampled meanwhile; then the library's own launch
    events around its attention kernel and its combine over min(K, 50) steps (a separate loop:
    an event between the two kernels stops their overlap); then the end-to-end step given as
    `e2e` = (copies in, call, copy out) over K steps (`time_e2e`).  Returns a dict of
    per-step milliseconds and the clocks."""
    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    if binding.get_device_errors(clear=True):
        raise SystemExit("device error word set during warm-up")
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(0)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0.record(stream)
    for i in range(K):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / K
    KT = min(K, 50)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(KT)]
    for e in ev:   # torch creates the CUDA event on first record; the trace hook needs the handle
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    for i in range(KT):
        binding.set_trace_events(*ev[i])
        step(i)
    torch.cuda.synchronize()
    binding.set_trace_events()
    kern_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    combine_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    errs = binding.get_device_errors(clear=True)
    e2e_ms, e2e_sched = time_e2e(*e2e, K, W, copies, stream)
    return {"ms": ms, "kern_ms": kern_ms, "combine_ms": combine_ms, "e2e_ms": e2e_ms, "e2e_schedule": e2e_sched,
            "errors": errs, "clocks": clk}


# ---- multi-token decode (speculative verification) ----------------------------------------

def multi_algorithmic(case, rows=None) -> int:
    """K/V rows each sequence's last new token attends (every tile of a sequence reads a
    prefix of them; with one tile per (sequence, kv head) each row is read once) + q + out +
    block-table entries + seq_lens + the work map.  `rows`: restrict to these sequences."""
    kv = case.kv
    lens = kv.seq_lens.cpu().to(torch.int64)
    ql = torch.as_tensor(case.q_lens, dtype=torch.int64)
    if rows is not None:
        lens, ql = lens[rows], ql[rows]
    B = lens.numel()
    nkv = int(lens.sum()) * kv.Hkv * kv.D * 2 * 2
    qo = 2 * int(ql.sum()) * kv.Hq * kv.D * 2
    pages = int(((lens + kv.page_size - 1) // kv.page_size).sum()) * 4
    return nkv + qo + pages + B * 4 + (B + 1) * 4 + 2 * 4 * B


class MultiOracle:
    def __init__(self, case):
        import oracle
        self.oracle = oracle
        self.case = case
        kv = case.kv
        self.q = bits(case.q)
        self.k = bits(kv.k_cache)
        self.v = bits(kv.v_cache)
        self.table = kv.block_table.cpu().numpy()
        self.lens = kv.seq_lens.cpu().numpy()
        self.qi = np.concatenate([[0], np.cumsum(case.q_lens)]).astype(np.int64)

    def run(self, seqs):
        qrows = np.concatenate([np.arange(self.qi[b], self.qi[b + 1]) for b in seqs])
        qi = np.concatenate([[0], np.cumsum([self.case.q_lens[b] for b in seqs])]).astype(np.int32)
        t0 = time.perf_counter()
        self.oracle.decode_paged_multi(np.ascontiguousarray(self.q[qrows]), self.k, self.v,
                                       np.ascontiguousarray(self.table[seqs]), np.ascontiguousarray(self.lens[seqs]),
                                       qi, self.case.kv.scale)
        return time.perf_counter() - t0

    def sample(self, target_s):
        dt = self.run(np.arange(1))
        return np.arange(int(max(1, min(len(self.case.q_lens), target_s / max(dt, 1e-4)))))


def run_multi(args):
    from paged_kv_cache_298_gb300 import binding, inputs
    dev = torch.device("cuda", 0)
    binding.load()
    case = inputs.spec_verify_paged(device=dev, B=args.batch or 128)
    kv = case.kv
    hbm_peak, peak_src = peaks()
    plan = binding.MultiPlan(case.q_lens, kv.Hq, kv.Hkv, dev)
    sms = binding.device_sm_count()
    S = args.splits if args.splits > 0 else binding.plan_splits(sms, plan.num_tiles, kv.Hq, kv.Hkv, kv.D,
                                                                kv.page_size, kv.max_kv_len, kv.total_kv)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    footprint = sum(t.numel() * t.element_size() for t in (case.q, kv.k_cache, kv.v_cache, kv.block_table,
                                                           kv.seq_lens))
    copies = 1 + max(1, math.ceil(2 * l2 / footprint))
    sets = [case] + [inputs.MultiCase(case.q.clone(), inputs.PagedCase(
        kv.q, kv.k_cache.clone(), kv.v_cache.clone(), kv.block_table.clone(), kv.seq_lens.clone(), kv.page_size,
        kv.scale, kv.name), case.q_lens) for _ in range(copies - 1)]
    ws = [torch.empty(max(1, binding.workspace_bytes_multi(case.total_q, kv.Hq, kv.D, S)), dtype=torch.uint8,
                      device=dev) for _ in sets]
    outs = [torch.empty_like(case.q) for _ in sets]
    maxlen = kv.max_kv_len
    stream = torch.cuda.current_stream()

    def step(i, pl=None):
        c = sets[i % copies]
        binding.decode_attn_paged_multi(c.q, c.kv.k_cache, c.kv.v_cache, c.kv.block_table, c.kv.seq_lens,
                                        plan if pl is None else pl, max_kv_len=maxlen, scale=kv.scale, num_splits=S,
                                        workspace=ws[i % copies], out=outs[i % copies])

    # end to end: q, block table, seq_lens and the work map in from pinned host memory, out back
    hq = case.q.cpu().pin_memory()
    ht = kv.block_table.cpu().pin_memory()
    hl = kv.seq_lens.cpu().pin_memory()
    hmap = [plan.qo_indptr.cpu().pin_memory(), plan.tile_batch.cpu().pin_memory(),
            plan.tile_index.cpu().pin_memory()]
    ho = torch.empty(case.q.shape, dtype=torch.bfloat16).pin_memory()
    plans = [binding.MultiPlan(case.q_lens, kv.Hq, kv.Hkv, dev) for _ in sets]

    def h2d(i):
        j = i % copies
        c = sets[j]
        c.q.copy_(hq, non_blocking=True)
        c.kv.block_table.copy_(ht, non_blocking=True)
        c.kv.seq_lens.copy_(hl, non_blocking=True)
        for d, h in zip((plans[j].qo_indptr, plans[j].tile_batch, plans[j].tile_index), hmap):
            d.copy_(h, non_blocking=True)

    def d2h(i):
        ho.copy_(outs[i % copies], non_blocking=True)

    r = measure_step(binding, step, (h2d, lambda i: step(i, pl=plans[i % copies]), d2h), args.steps, args.warmup,
                     stream, copies)
    K, ms, kern_ms, combine_ms, e2e_ms = args.steps, r["ms"], r["kern_ms"], r["combine_ms"], r["e2e_ms"]
    errs, clk = r["errors"], r["clocks"]

    nbytes = multi_algorithmic(case)
    lens = kv.seq_lens.cpu().tolist()
    flops = sum(4 * kv.Hq * kv.D * sum(L - ql + i + 1 for i in range(ql)) for L, ql in zip(lens, case.q_lens))
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    h2d = hq.numel() * 2 + ht.numel() * 4 + hl.numel() * 4 + sum(h.numel() * 4 for h in hmap)
    line = {
        "metric": "multi-token paged decode achieved HBM GB/s (algorithmic bytes), cold KV",
        "value": round(nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "us_per_call": round(ms * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": kv.name, "B": len(case.q_lens), "q_len": case.q_lens[0], "total_q": case.total_q,
                   "Hq": kv.Hq, "Hkv": kv.Hkv, "D": kv.D, "page_size": kv.page_size, "total_kv": kv.total_kv,
                   "num_tiles": plan.num_tiles, "num_splits": S, "kv_dtype": "bf16",
                   "cold_kv": f"{copies} rotated input copies of {footprint / 1e9:.2f} GB each (> 2x L2)"},
        "attention_tflops": round(flops / (ms * 1e-3) / 1e12, 2),
        "roofline": {"bound": "hbm", "kernel": "multi_kernel", "achieved": round(achieved, 1), "peak": hbm_peak,
                     "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "multi_kernel_ms": round(kern_ms, 5), "combine_ms": round(combine_ms, 5),
                     "algorithmic_bytes_per_launch": nbytes,
                     "traffic": recorded_traffic("multi_kernel", workload_key(args))},
        "e2e": {"schedule": r["e2e_schedule"], "value": round(nbytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": ho.numel() * 2},
        "gpu_launches": K * (2 if S > 1 else 1), "device_errors": errs, "clocks": clk,
    }
    if not args.no_cpu_baseline:
        r = MultiOracle(case)
        seqs = r.sample(10.0)
        dt, passes = repeat_for(lambda: r.run(seqs))
        line["cpu_baseline"] = {"value": multi_algorithmic(case, torch.as_tensor(seqs)) / dt / 1e9, "unit": "GB/s",
                                "cores": r.oracle.num_threads(), "kind": "oracle",
                                "sample": f"fp64 oracle (OpenMP) on sequences 0..{len(seqs) - 1} of "
                                          f"{len(case.q_lens)} (all new tokens and heads), {passes} passes of "
                                          f"{dt:.2f} s"}
    print(json.dumps(line), flush=True)


def run_reference_multi(args):
    from paged_kv_cache_298_gb300 import inputs
    case = inputs.spec_verify_paged()
    r = MultiOracle(case)
    seqs = r.sample(min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        r.run(seqs)
    dt = statistics.mean(r.run(seqs) for _ in range(args.steps))
    value = multi_algorithmic(case, torch.as_tensor(seqs)) / dt / 1e9
    print(json.dumps({
        "impl": "reference",
        "metric": "multi-token paged decode achieved HBM GB/s (algorithmic bytes), cold KV",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": {"workload": case.kv.name, "sample_sequences": len(seqs)},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": r.oracle.num_threads(), "kind": "oracle",
                         "sample": f"fp64 oracle (OpenMP) on sequences 0..{len(seqs) - 1} per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


# ---- GQA decode over an e4m3 cache --------------------------------------------------------

def fp8kv_algorithmic(case, rows=None) -> int:
    """e4m3 K/V codes of the rows inside seq_lens + their two bf16 factors per kv head + q +
    out + block-table entries + seq_lens.  `rows`: restrict to these sequences."""
    lens = case.seq_lens.cpu().to(torch.int64)
    if rows is not None:
        lens = lens[rows]
    B = lens.numel()
    kv = int(lens.sum()) * case.Hkv * (2 * case.D + 2 * 2)
    qo = 2 * B * case.Hq * case.D * 2
    pages = int(((lens + case.page_size - 1) // case.page_size).sum()) * 4
    return kv + qo + pages + B * 4


class Fp8KvOracle:
    def __init__(self, case):
        import oracle
        self.oracle = oracle
        self.case = case
        self.q = bits(case.q)
        self.kc = case.k_codes.cpu().numpy()
        self.vc = case.v_codes.cpu().numpy()
        self.ks = bits(case.k_scale)
        self.vs = bits(case.v_scale)
        self.table = case.block_table.cpu().numpy()
        self.lens = case.seq_lens.cpu().numpy()

    def run(self, rows):
        t0 = time.perf_counter()
        self.oracle.decode_paged_fp8kv(np.ascontiguousarray(self.q[rows]), self.kc, self.vc, self.ks, self.vs,
                                       np.ascontiguousarray(self.table[rows]), np.ascontiguousarray(self.lens[rows]),
                                       self.case.scale)
        return time.perf_counter() - t0

    def sample(self, target_s):
        dt = self.run(np.arange(1))
        return np.arange(int(max(1, min(self.case.B, target_s / max(dt, 1e-4)))))


def run_fp8kv(args):
    from paged_kv_cache_298_gb300 import binding, inputs
    dev = torch.device("cuda", 0)
    binding.load()
    case = inputs.ragged_fp8kv(device=dev, B=args.batch or 128)
    hbm_peak, peak_src = peaks()
    sms = binding.device_sm_count()
    S = args.splits if args.splits > 0 else binding.plan_splits(sms, case.B, case.Hq, case.Hkv, case.D,
                                                                case.page_size, case.max_kv_len, case.total_kv)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    parts = ("q", "k_codes", "v_codes", "k_scale", "v_scale", "block_table", "seq_lens")
    footprint = sum(getattr(case, n).numel() * getattr(case, n).element_size() for n in parts)
    copies = 1 + max(1, math.ceil(2 * l2 / footprint))
    sets = [case] + [inputs.Fp8KvCase(*[getattr(case, n).clone() for n in parts], case.page_size, case.scale,
                                      case.name) for _ in range(copies - 1)]
    ws = [torch.empty(max(1, binding.workspace_bytes(case.B, case.Hq, case.Hkv, case.D, S) if S > 1 else 1),
                      dtype=torch.uint8, device=dev) for _ in sets]
    outs = [torch.empty_like(case.q) for _ in sets]
    maxlen = case.max_kv_len
    stream = torch.cuda.current_stream()

    def step(i):
        j = i % copies
        c = sets[j]
        binding.decode_attn_paged_fp8kv(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.block_table, c.seq_lens,
                                        max_kv_len=maxlen, scale=c.scale, num_splits=S, workspace=ws[j], out=outs[j])

    # end to end: q, block table and seq_lens in from pinned host memory, out back
    hq = case.q.cpu().pin_memory()
    ht = case.block_table.cpu().pin_memory()
    hl = case.seq_lens.cpu().pin_memory()
    ho = torch.empty(case.q.shape, dtype=torch.bfloat16).pin_memory()

    def h2d(i):
        c = sets[i % copies]
        c.q.copy_(hq, non_blocking=True)
        c.block_table.copy_(ht, non_blocking=True)
        c.seq_lens.copy_(hl, non_blocking=True)

    def d2h(i):
        ho.copy_(outs[i % copies], non_blocking=True)

    r = measure_step(binding, step, (h2d, step, d2h), args.steps, args.warmup, stream, copies)
    K, ms, kern_ms, combine_ms, e2e_ms = args.steps, r["ms"], r["kern_ms"], r["combine_ms"], r["e2e_ms"]
    errs, clk = r["errors"], r["clocks"]

    nbytes = fp8kv_algorithmic(case)
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    lens = case.seq_lens.cpu()
    line = {
        "metric": "paged decode attention over an e4m3 KV cache, achieved HBM GB/s (algorithmic bytes), cold KV",
        "value": round(nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "us_per_call": round(ms * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": case.name, "B": case.B, "Hq": case.Hq, "Hkv": case.Hkv, "D": case.D,
                   "page_size": case.page_size, "kv_len_min": int(lens.min()), "kv_len_max": int(lens.max()),
                   "total_kv": case.total_kv, "num_splits": S, "kv_dtype": "e4m3 + bf16 factor per (slot, kv head)",
                   "cold_kv": f"{copies} rotated input copies of {footprint / 1e9:.2f} GB each (> 2x L2)"},
        "kv_tokens_per_s": round(case.total_kv / (ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": "fp8kv_kernel", "achieved": round(achieved, 1), "peak": hbm_peak,
                     "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "fp8kv_kernel_ms": round(kern_ms, 5), "combine_ms": round(combine_ms, 5),
                     "algorithmic_bytes_per_launch": nbytes,
                     "traffic": recorded_traffic("fp8kv_kernel", workload_key(args))},
        "e2e": {"schedule": r["e2e_schedule"], "value": round(nbytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": hq.numel() * 2 + ht.numel() * 4 + hl.numel() * 4,
                "d2h_bytes_per_step": ho.numel() * 2},
        "gpu_launches": K * (2 if S > 1 else 1), "device_errors": errs, "clocks": clk,
    }
    if not args.no_cpu_baseline:
        r = Fp8KvOracle(case)
        rows = r.sample(10.0)
        dt, passes = repeat_for(lambda: r.run(rows))
        line["cpu_baseline"] = {"value": fp8kv_algorithmic(case, torch.as_tensor(rows)) / dt / 1e9, "unit": "GB/s",
                                "cores": r.oracle.num_threads(), "kind": "oracle",
                                "sample": f"fp64 oracle (OpenMP) on sequences 0..{len(rows) - 1} of {case.B} "
                                          f"(all heads), {passes} passes of {dt:.2f} s"}
    print(json.dumps(line), flush=True)


def run_reference_fp8kv(args):
    from paged_kv_cache_298_gb300 import inputs
    case = inputs.ragged_fp8kv()
    r = Fp8KvOracle(case)
    rows = r.sample(min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        r.run(rows)
    dt = statistics.mean(r.run(rows) for _ in range(args.steps))
    value = fp8kv_algorithmic(case, torch.as_tensor(rows)) / dt / 1e9
    print(json.dumps({
        "impl": "reference",
        "metric": "paged decode attention over an e4m3 KV cache, achieved HBM GB/s (algorithmic bytes), cold KV",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": {"workload": case.name, "sample_sequences": len(rows)},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": r.oracle.num_threads(), "kind": "oracle",
                         "sample": f"fp64 oracle (OpenMP) on sequences 0..{len(rows) - 1} per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


# ---- masked decode --------------------------------------------------------------------------

def masked_inputs(device):
    """The ragged decode batch with a 2-D bool mask keeping each key with probability 0.9
    (seeded), rows padded to a multiple of 16 bytes."""
    from paged_kv_cache_298_gb300 import inputs
    case = inputs.ragged_paged(device=device)
    width = (case.max_kv_len + 15) // 16 * 16
    g = torch.Generator().manual_seed(298008)
    mask = (torch.rand((case.B, width), generator=g) < 0.9).to(torch.uint8).to(device)
    return case, mask


def masked_algorithmic(case, rows=None) -> int:
    """The bf16 decode's algorithmic bytes (every K/V row inside seq_lens is streamed; the
    mask drops keys from the softmax, not from the tiles) plus one mask byte per key."""
    lens = case.seq_lens.cpu().to(torch.int64)
    if rows is not None:
        lens = lens[rows]
    return algorithmic_bytes(case, rows) + int(lens.sum())


def run_masked(args):
    from paged_kv_cache_298_gb300 import binding
    dev = torch.device("cuda", 0)
    binding.load()
    case, mask = masked_inputs(dev)
    hbm_peak, peak_src = peaks()
    S = args.splits if args.splits > 0 else binding.plan_splits(binding.device_sm_count(), case.B, case.Hq, case.Hkv,
                                                                case.D, case.page_size, case.max_kv_len,
                                                                case.total_kv)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    footprint = sum(t.numel() * t.element_size() for t in (case.q, case.k_cache, case.v_cache, case.block_table,
                                                           case.seq_lens, mask))
    copies = 1 + max(1, math.ceil(2 * l2 / footprint))
    sets = [(case, mask)] + [(type(case)(case.q.clone(), case.k_cache.clone(), case.v_cache.clone(),
                                         case.block_table.clone(), case.seq_lens.clone(), case.page_size, case.scale,
                                         case.name), mask.clone()) for _ in range(copies - 1)]
    ws = [torch.empty(max(1, binding.workspace_bytes(case.B, case.Hq, case.Hkv, case.D, S) if S > 1 else 1),
                      dtype=torch.uint8, device=dev) for _ in sets]
    outs = [torch.empty_like(case.q) for _ in sets]
    maxlen = case.max_kv_len
    stream = torch.cuda.current_stream()

    def step(i):
        j = i % copies
        c, m = sets[j]
        binding.decode_attn_paged_masked(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens, m, max_kv_len=maxlen,
                                         scale=c.scale, num_splits=S, workspace=ws[j], out=outs[j])

    hq, ht, hl = (t.cpu().pin_memory() for t in (case.q, case.block_table, case.seq_lens))
    hm = mask.cpu().pin_memory()
    ho = torch.empty(case.q.shape, dtype=torch.bfloat16).pin_memory()

    def h2d(i):
        c, m = sets[i % copies]
        c.q.copy_(hq, non_blocking=True)
        c.block_table.copy_(ht, non_blocking=True)
        c.seq_lens.copy_(hl, non_blocking=True)
        m.copy_(hm, non_blocking=True)

    def d2h(i):
        ho.copy_(outs[i % copies], non_blocking=True)

    r = measure_step(binding, step, (h2d, step, d2h), args.steps, args.warmup, stream, copies)
    nbytes = masked_algorithmic(case)
    achieved = nbytes / (r["kern_ms"] * 1e-3) / 1e9
    line = {
        "metric": "masked paged decode achieved HBM GB/s (algorithmic bytes), cold KV",
        "value": round(nbytes / (r["ms"] * 1e-3) / 1e9, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(r["ms"], 5), "us_per_call": round(r["ms"] * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(case, S, copies, footprint) | {
            "workload": case.name + ", 2-D bool mask keeping 90% of keys", "mask": "uint8 [B, 4096], p(keep) = 0.9"},
        "roofline": {"bound": "hbm", "kernel": "multi_kernel (one token per sequence, masked)",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "peak_source": f"{peak_src} hbm_gbs",
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "kernel_ms": round(r["kern_ms"], 5),
                     "combine_ms": round(r["combine_ms"], 5), "algorithmic_bytes_per_launch": nbytes,
                     "traffic": recorded_traffic("multi_kernel", "masked")},
        "e2e": {"schedule": r["e2e_schedule"], "value": round(nbytes / (r["e2e_ms"] * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(r["e2e_ms"], 5),
                "h2d_bytes_per_step": hq.numel() * 2 + ht.numel() * 4 + hl.numel() * 4 + hm.numel(),
                "d2h_bytes_per_step": ho.numel() * 2},
        "gpu_launches": args.steps * (2 if S > 1 else 1), "device_errors": r["errors"], "clocks": r["clocks"],
    }
    if not args.no_cpu_baseline:
        import oracle
        cm = mask.cpu().numpy()
        q, k, v = bits(case.q), bits(case.k_cache), bits(case.v_cache)
        table, lens = case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy()
        def one(n):
            t0 = time.perf_counter()
            oracle.decode_paged_masked(q[:n], k, v, table[:n], lens[:n], cm[:n], case.scale)
            return time.perf_counter() - t0
        n = int(max(1, min(case.B, 10.0 / max(one(1), 1e-4))))   # a prefix within about 10 s a pass
        dt, passes = repeat_for(lambda: one(n))
        line["cpu_baseline"] = {"value": masked_algorithmic(case, torch.arange(n)) / dt / 1e9, "unit": "GB/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"fp64 oracle (OpenMP) on sequences 0..{n - 1} of {case.B} (all heads), "
                                          f"{passes} passes of {dt:.2f} s"}
    print(json.dumps(line), flush=True)


def run_reference_masked(args):
    import oracle
    case, mask = masked_inputs("cpu")
    q, k, v = bits(case.q), bits(case.k_cache), bits(case.v_cache)
    table, lens, cm = case.block_table.numpy(), case.seq_lens.numpy(), mask.numpy()
    budget = min(8.0, 150.0 / max(1, args.steps + args.warmup))
    t0 = time.perf_counter()
    oracle.decode_paged_masked(q[:1], k, v, table[:1], lens[:1], cm[:1], case.scale)
    n = int(max(1, min(case.B, budget / max(time.perf_counter() - t0, 1e-4))))
    for _ in range(args.warmup):
        oracle.decode_paged_masked(q[:n], k, v, table[:n], lens[:n], cm[:n], case.scale)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.decode_paged_masked(q[:n], k, v, table[:n], lens[:n], cm[:n], case.scale)
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    value = masked_algorithmic(case, torch.arange(n)) / dt / 1e9
    print(json.dumps({
        "impl": "reference", "metric": "masked paged decode achieved HBM GB/s (algorithmic bytes), cold KV",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": {"workload": case.name + ", 2-D bool mask keeping 90% of keys",
                                                        "sample_sequences": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"fp64 oracle (OpenMP) on sequences 0..{n - 1} per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


# ---- reference arm: the fp64 oracle on the host cores ----------------------------------

def run_reference_fp8(args):
    import oracle
    from paged_kv_cache_298_gb300 import inputs
    case = inputs.fp8_swa()
    nbytes, _, _ = fp8_algorithmic(case)
    a = (bits(case.q), case.kv_cache.numpy(), bits(case.inv_scale), case.indices.numpy(), case.lens.numpy())
    for _ in range(args.warmup):
        oracle.fp8_swa(*a, case.block_size, case.scale)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.fp8_swa(*a, case.block_size, case.scale)
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    value = nbytes / dt / 1e9
    print(json.dumps({
        "impl": "reference",
        "metric": "fp8 sliding-window latent decode achieved HBM GB/s (algorithmic bytes), cold inputs",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": {"workload": case.name},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"fp64 oracle (OpenMP), all {case.T} tokens per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


def run_reference(args):
    rank, _, world = rank_info()
    if rank != 0:
        return
    if args.workload == "fp8":
        return run_reference_fp8(args)
    if args.workload == "multi":
        return run_reference_multi(args)
    if args.workload == "fp8kv":
        return run_reference_fp8kv(args)
    if args.workload == "masked":
        return run_reference_masked(args)
    case = make_workload(args.workload, "cpu")
    r = OracleRunner(case)
    rows = r.sample_rows(target_s=min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        r.run(rows)
    times = [r.run(rows) for _ in range(args.steps)]
    dt = statistics.mean(times)
    nbytes = algorithmic_bytes(case, torch.as_tensor(rows))
    value = nbytes / dt / 1e9
    sample = (f"fp64 oracle (OpenMP) on sequences 0..{len(rows) - 1} of {case.B} (all heads) per step")
    line = {
        "impl": "reference",
        "metric": "paged decode attention achieved HBM GB/s (algorithmic bytes), cold KV",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(case, 0, 1, 0) | {"sample_sequences": len(rows),
                                                   "cold_kv": "host memory (oracle on the CPU cores)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": r.oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ragged", choices=["ragged", "llama", "long1", "long4", "fp8", "append", "multi", "fp8kv", "masked"])
    ap.add_argument("--splits", type=int, default=-1,
                    help="-1 = the planner's choice, 0 = balanced schedule, S > 0 = per-sequence splits")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="ragged / multi workloads: number of sequences (0 = the workload's own, 128); "
                         "smaller batches are for profiler captures")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "fp8":
        run_fp8(args)
    elif args.workload == "append":
        run_append(args)
    elif args.workload == "multi":
        run_multi(args)
    elif args.workload == "fp8kv":
        run_fp8kv(args)
    elif args.workload == "masked":
        run_masked(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
