#!/usr/bin/env python3
"""Benchmark of paged GQA decode attention on GB300.

Headline step = one decode_attn_paged call (split kernel + combine kernel) over the whole
batch of the large ragged workload: B=128 sequences, Hq=32, Hkv=8, D=128, kv_len ~
U{256..4096}, page_size 16, pages assigned by a seeded shuffle of a 2x pool.  Inputs are
resident in HBM before the timed region; independent copies of every input are rotated so
that the bytes touched between two reads of the same copy exceed 2x L2 (cold KV).

Printed (rank 0, one JSON line): achieved HBM GB/s of algorithmic bytes (K/V rows inside
seq_lens, q, out, the block-table entries used, seq_lens) per step time, with the attention
kernel's own roofline, an end-to-end figure through host buffers, the fp64 oracle on a
bounded sample of the same workload on the host cores, and the SM clocks seen meanwhile.
With no --workload the same line carries, under "workloads", a compact leg for every other
configuration (Llama paged and contiguous, long context B=1 and B=4, fp8 sliding window,
multi-token, e4m3 cache, masked), each timed the same way with its own oracle baseline.

Per-call times are medians over back-to-back calls with CUDA events at every call boundary
(the attention kernel's own time from events the library records around its launch); the
contract's ms_per_step is the K-step region bracketed by two events.

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference] [--workload W]

With N > 1 (torchrun, one process per GPU) every rank runs an independent replica of the
headline (the path has no cross-GPU exchange); value = all ranks' bytes / the slowest
rank's time.
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
import tempfile
import time
from dataclasses import dataclass, field
from typing import Callable

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
LEGS = ("llama", "llama_contig", "long1", "long4", "fp8", "multi", "multi_g8", "multi_g8_q8", "fp8kv", "masked")
WORKLOADS = ("ragged",) + LEGS + ("append",)


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
        self.path = os.path.join(tempfile.gettempdir(), f"dap_clocks_{os.getpid()}_{id(self)}.csv")

    def start(self):
        try:
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


KERNEL_SOURCES = {"split_kernel": ("dap_decode.cu", "dap_decode.cuh", "dap_tile.cuh", "dap_device.cuh",
                                    "dap_internal.h"),
                  "multi_kernel": ("dap_multi.cu", "dap_multi.cuh", "dap_tile.cuh", "dap_device.cuh",
                                   "dap_internal.h"),
                  "multi_tc_kernel": ("dap_multi_tc.cu", "dap_multi.cuh", "dap_tile.cuh", "dap_device.cuh",
                                      "dap_tc.cuh", "dap_internal.h"),
                  "fp8kv_kernel": ("dap_fp8kv.cu", "dap_tile.cuh", "dap_device.cuh", "dap_internal.h"),
                  "swa_kernel": ("dap_fp8.cu", "dap_device.cuh", "dap_tc.cuh", "dap_internal.h")}


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


def job_throughput(ms_list, nbytes_per_rank, world, device):
    """Whole-job GB/s for each timing in ms_list: every rank processed nbytes_per_rank, and
    the job took as long as its slowest rank (max over ranks of each timing).  Returns
    [(GB/s, max ms), ...].  With world > 1 it needs an initialised process group."""
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in ms_list], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [(world * nbytes_per_rank / (m * 1e-3) / 1e9, m) for m in t.tolist()]


def rotated(make_copy, footprint, l2, at_least=2):
    """Independent copies of a workload's inputs, enough that the bytes touched between two
    reads of one copy exceed 2x L2 (the first is the original)."""
    n = max(at_least, 1 + math.ceil(2 * l2 / max(1, footprint)))
    return [make_copy(i) for i in range(n)]


# ---- algorithmic bytes (what the method must move; K/V rows inside the lengths) -------------

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


def contig_bytes(case, rows=None) -> int:
    """The contiguous cache: K/V rows inside seq_lens + q + out + seq_lens (no table)."""
    lens = case.seq_lens.cpu().to(torch.int64)
    if rows is not None:
        lens = lens[rows]
    B = lens.numel()
    return int(lens.sum()) * case.Hkv * case.D * 2 * 2 + 2 * B * case.Hq * case.D * 2 + B * 4


def fp8_counts(case):
    """Participating rows per token (j < min(len, W), slot >= 0), from the inputs."""
    idx = case.indices.cpu()
    lens = case.lens.cpu().clamp(min=0, max=case.W)
    j = torch.arange(case.W)[None, :]
    return ((j < lens[:, None]) & (idx >= 0)).sum(dim=1)


def fp8_algorithmic(case, tokens=None):
    """Bytes: q + out + every participating fp8 row and its bf16 inverse scale + the slot
    table + lens.  Flops: QK^T and PV, 2 * 2 * NH * rows * HD per token."""
    n = fp8_counts(case)
    T = case.T
    if tokens is not None:
        n = n[:tokens]
        T = tokens
    rows = int(n.sum())
    nbytes = 2 * T * case.NH * case.HD * 2 + rows * (case.HD + 2) + T * case.W * 8 + T * 8
    flops = 4 * case.NH * case.HD * rows
    return nbytes, flops, rows


def multi_algorithmic(case, rows=None) -> int:
    """K/V rows each sequence's last new token attends, once per (sequence, kv head) + q +
    out + block-table entries + seq_lens + the work map.  `rows`: restrict to these
    sequences.  A kernel that reads a sequence's rows more than once (several q tiles of
    one sequence) pays for it in time, not in this count."""
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


def masked_algorithmic(case, rows=None) -> int:
    """The bf16 decode's algorithmic bytes (every K/V row inside seq_lens is streamed; the
    mask drops keys from the softmax, not from the tiles) plus one mask byte per key."""
    lens = case.seq_lens.cpu().to(torch.int64)
    if rows is not None:
        lens = lens[rows]
    return algorithmic_bytes(case, rows) + int(lens.sum())


# ---- workloads ---------------------------------------------------------------------------

def masked_inputs(device):
    """The ragged decode batch with a 2-D bool mask keeping each key with probability 0.9
    (seeded), rows padded to a multiple of 16 bytes."""
    from paged_kv_cache_298_gb300 import inputs
    case = inputs.ragged_paged(device=device)
    width = (case.max_kv_len + 15) // 16 * 16
    g = torch.Generator().manual_seed(298008)
    mask = (torch.rand((case.B, width), generator=g) < 0.9).to(torch.uint8).to(device)
    return case, mask


def make_case(key, device, batch=0):
    from paged_kv_cache_298_gb300 import inputs
    if key == "ragged":
        return inputs.ragged_paged(device=device, B=batch or 128)
    if key in ("llama", "llama_contig"):
        return inputs.llama_paged(device=device)
    if key in ("long1", "long4"):
        return inputs.long_paged(B=int(key[-1]), device=device)
    if key == "fp8":
        return inputs.fp8_swa(device=device)
    if key == "multi":
        return inputs.spec_verify_paged(device=device, B=batch or 128)
    if key in ("multi_g8", "multi_g8_q8"):   # G = 8: Hq=64, Hkv=8, 4 or 8 new tokens
        return inputs.spec_verify_paged(device=device, B=batch or 128, q_len=8 if key.endswith("q8") else 4, Hq=64)
    if key == "fp8kv":
        return inputs.ragged_fp8kv(device=device, B=batch or 128)
    if key == "masked":
        return masked_inputs(device)
    raise SystemExit(f"unknown workload {key}")


class OracleSample:
    """The fp64 oracle on the first n units (sequences or tokens) of a workload, on the host
    cores.  `run(n)` returns its seconds; `nbytes(n)` the algorithmic bytes of those units."""

    def __init__(self, units, run, nbytes, unit_name):
        import oracle
        self.oracle = oracle
        self.units, self.run, self.nbytes, self.unit_name = units, run, nbytes, unit_name

    def size_for(self, target_s):
        dt = self.run(1)
        return int(max(1, min(self.units, target_s / max(dt, 1e-4))))

    def measure(self, target_s):
        """Whole passes over a prefix sized for about target_s a pass, repeated until about
        target_s of CPU work: GB/s of the sample's algorithmic bytes."""
        n = self.size_for(target_s)
        total, passes = 0.0, 0
        while passes == 0 or total < target_s:
            total += self.run(n)
            passes += 1
        dt = total / passes
        return {"value": self.nbytes(n) / dt / 1e9, "unit": "GB/s", "cores": self.oracle.num_threads(),
                "kind": "oracle",
                "sample": f"fp64 oracle (OpenMP) on {self.unit_name} 0..{n - 1} of {self.units}, "
                          f"{passes} passes of {dt:.3f} s"}


def oracle_sample(key, case) -> OracleSample:
    """The oracle on a CPU copy of the workload's inputs."""
    import oracle

    def timed(fn):
        def run(n):
            t0 = time.perf_counter()
            fn(n)
            return time.perf_counter() - t0
        return run

    if key == "fp8":
        a = (bits(case.q), case.kv_cache.cpu().numpy(), bits(case.inv_scale), case.indices.cpu().numpy(),
             case.lens.cpu().numpy())
        return OracleSample(case.T, timed(lambda n: oracle.fp8_swa(*a, case.block_size, case.scale, tokens=(0, n))),
                            lambda n: fp8_algorithmic(case, n)[0], "tokens")
    if key.startswith("multi"):
        kv = case.kv
        q, k, v = bits(case.q), bits(kv.k_cache), bits(kv.v_cache)
        table, lens = kv.block_table.cpu().numpy(), kv.seq_lens.cpu().numpy()
        qi = np.concatenate([[0], np.cumsum(case.q_lens)]).astype(np.int32)
        return OracleSample(len(case.q_lens), timed(lambda n: oracle.decode_paged_multi(
            q[:qi[n]], k, v, table[:n], lens[:n], qi[:n + 1], kv.scale)),
            lambda n: multi_algorithmic(case, torch.arange(n)), "sequences")
    if key == "fp8kv":
        q, kc, vc = bits(case.q), case.k_codes.cpu().numpy(), case.v_codes.cpu().numpy()
        ks, vs = bits(case.k_scale), bits(case.v_scale)
        table, lens = case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy()
        return OracleSample(case.B, timed(lambda n: oracle.decode_paged_fp8kv(q[:n], kc, vc, ks, vs, table[:n],
                                                                             lens[:n], case.scale)),
                            lambda n: fp8kv_algorithmic(case, torch.arange(n)), "sequences")
    if key == "masked":
        c, m = case
        q, k, v = bits(c.q), bits(c.k_cache), bits(c.v_cache)
        table, lens, mk = c.block_table.cpu().numpy(), c.seq_lens.cpu().numpy(), m.cpu().numpy()
        return OracleSample(c.B, timed(lambda n: oracle.decode_paged_masked(q[:n], k, v, table[:n], lens[:n], mk[:n],
                                                                           c.scale)),
                            lambda n: masked_algorithmic(c, torch.arange(n)), "sequences")
    if key == "llama_contig":
        from paged_kv_cache_298_gb300 import inputs
        kl, vl = inputs.logical_kv(case)
        q, k, v, lens = bits(case.q), bits(kl), bits(vl), case.seq_lens.cpu().numpy()
        return OracleSample(case.B, timed(lambda n: oracle.decode_contig(q[:n], k[:n], v[:n], lens[:n], case.scale)),
                            lambda n: contig_bytes(case, torch.arange(n)), "sequences")
    q, k, v = bits(case.q), bits(case.k_cache), bits(case.v_cache)
    table, lens = case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy()
    return OracleSample(case.B, timed(lambda n: oracle.decode_paged(q[:n], k, v, table[:n], lens[:n], case.scale)),
                        lambda n: algorithmic_bytes(case, torch.arange(n)), "sequences")


@dataclass
class Leg:
    """One workload ready to time on the GPU."""
    key: str
    metric: str
    config: dict
    nbytes: int                          # algorithmic bytes per call
    kernel: str                          # the dominant kernel (its roofline is reported)
    step: Callable[[int], None]          # one library call on rotated input copy i
    e2e: tuple                           # (copies in, call, copy out) for step i
    h2d_bytes: int
    d2h_bytes: int
    launches: int                        # kernels per call
    copies: int
    trace: bool = True                   # the library records events around its kernel
    extra: dict = field(default_factory=dict)


def prepare_leg(key, case, dev, l2, splits=None, tpt=None) -> Leg:
    """Rotated device copies of the inputs, the step, the end-to-end copies and the bytes."""
    from paged_kv_cache_298_gb300 import binding, inputs
    sms = binding.device_sm_count()

    def plan(units, Hq, Hkv, D, ps, L, total):
        """The split count passed to the library: the planner's, made with the summed
        lengths the host knows (or --splits when given)."""
        if splits is not None:
            return splits
        return binding.resolve_splits(0, sms, units, Hq, Hkv, D, ps, L, total)

    if key in ("ragged", "llama", "long1", "long4", "llama_contig", "masked"):
        mask = None
        if key == "masked":
            case, mask = case
        contig = key == "llama_contig"
        S = plan(case.B, case.Hq, case.Hkv, case.D, case.page_size, case.max_kv_len, case.total_kv)
        run = binding.resolve_splits(S, sms, case.B, case.Hq, case.Hkv, case.D, case.page_size, case.max_kv_len)
        if contig:
            k0, v0 = inputs.logical_kv(case)
            parts = (case.q, k0, v0, case.seq_lens)
            nbytes = contig_bytes(case)
        else:
            parts = (case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens) + \
                ((mask,) if mask is not None else ())
            nbytes = masked_algorithmic(case) if mask is not None else algorithmic_bytes(case)
        footprint = sum(t.numel() * t.element_size() for t in parts)
        sets = rotated(lambda i: parts if i == 0 else tuple(t.clone() for t in parts), footprint, l2)
        ws = [torch.empty(max(1, binding.workspace_bytes(case.B, case.Hq, case.Hkv, case.D, run)),
                          dtype=torch.uint8, device=dev) for _ in sets]
        outs = [torch.empty_like(case.q) for _ in sets]
        maxlen, n = case.max_kv_len, len(sets)

        def call(i):
            j = i % n
            p = sets[j]
            if contig:
                binding.decode_attn_contig(p[0], p[1], p[2], p[3], max_kv_len=maxlen, scale=case.scale,
                                           num_splits=S, workspace=ws[j], out=outs[j])
            elif mask is not None:
                binding.decode_attn_paged_masked(*p[:5], p[5], max_kv_len=maxlen, scale=case.scale, num_splits=S,
                                                 workspace=ws[j], out=outs[j])
            else:
                binding.decode_attn_paged(*p, max_kv_len=maxlen, scale=case.scale, num_splits=S, workspace=ws[j],
                                          out=outs[j])

        # end to end: q, the table (or nothing for the contiguous cache), seq_lens and the
        # mask in from pinned host memory, out back; the K/V cache is resident state
        small = [0, 3] if contig else [0, 3, 4] + ([5] if mask is not None else [])
        host = {k: parts[k].cpu().pin_memory() for k in small}
        ho = torch.empty(case.q.shape, dtype=torch.bfloat16).pin_memory()

        def h2d(i):
            for k, h in host.items():
                sets[i % n][k].copy_(h, non_blocking=True)

        def d2h(i):
            ho.copy_(outs[i % n], non_blocking=True)

        lens = case.seq_lens.cpu()
        cfg = {"workload": case.name + (", contiguous cache" if contig else "") +
               (", 2-D bool mask keeping 90% of keys" if mask is not None else ""),
               "B": case.B, "Hq": case.Hq, "Hkv": case.Hkv, "D": case.D,
               "page_size": None if contig else case.page_size, "kv_len_min": int(lens.min()),
               "kv_len_max": int(lens.max()), "total_kv": case.total_kv, "num_splits": run, "kv_dtype": "bf16",
               "cold_kv": f"{n} rotated input copies of {footprint / 1e9:.2f} GB each (> 2x L2)"}
        metric = ("masked paged decode" if mask is not None else
                  "contiguous-cache decode" if contig else "paged decode attention")
        return Leg(key, f"{metric} achieved HBM GB/s (algorithmic bytes), cold KV", cfg, nbytes,
                   "multi_kernel" if mask is not None else "split_kernel", call, (h2d, call, d2h),
                   sum(h.numel() * h.element_size() for h in host.values()), ho.numel() * 2,
                   2 if run != 1 else 1, n)

    if key == "fp8":
        parts = (case.q, case.kv_cache, case.inv_scale, case.indices, case.lens)
        footprint = sum(t.numel() * t.element_size() for t in parts) + case.q.numel() * 2
        sets = rotated(lambda i: parts if i == 0 else tuple(t.clone() for t in parts), footprint, l2)
        outs = [torch.empty_like(case.q) for _ in sets]
        n = len(sets)

        def call(i):
            q, kv, inv, idx, ln = sets[i % n]
            binding.decode_attn_paged_fp8(q, kv, inv, idx, ln, scale=case.scale, out=outs[i % n])

        hq, hidx, hln = (case.q.cpu().pin_memory(), case.indices.cpu().pin_memory(), case.lens.cpu().pin_memory())
        ho = torch.empty(case.q.shape, dtype=torch.bfloat16).pin_memory()

        def h2d(i):
            q, kv, inv, idx, ln = sets[i % n]
            q.copy_(hq, non_blocking=True)
            idx.copy_(hidx, non_blocking=True)
            ln.copy_(hln, non_blocking=True)

        def d2h(i):
            ho.copy_(outs[i % n], non_blocking=True)

        nbytes, flops, rows = fp8_algorithmic(case)
        cfg = {"workload": case.name, "T": case.T, "NH": case.NH, "HD": case.HD, "W": case.W,
               "num_blocks": case.num_blocks, "block_size": case.block_size, "rows": rows, "kv_dtype": "fp8-e4m3",
               "cold": f"{n} rotated input copies of {footprint / 1e6:.1f} MB"}
        return Leg(key, "fp8 sliding-window latent decode achieved HBM GB/s (algorithmic bytes), cold inputs", cfg,
                   nbytes, "swa_kernel", call, (h2d, call, d2h), hq.numel() * 2 + hidx.numel() * 8 + hln.numel() * 8,
                   ho.numel() * 2, 1, n, trace=False, extra={"flops": flops})

    if key.startswith("multi"):
        kv = case.kv
        mplan = binding.MultiPlan(case.q_lens, kv.Hq, kv.Hkv, dev, tokens_per_tile=tpt, D=kv.D)
        # 128 query rows per tile: the tcgen05 consumer; 16 or 32 columns: the mma.sync one
        mkernel = "multi_tc_kernel" if mplan.tokens_per_tile * (kv.Hq // kv.Hkv) == 128 else "multi_kernel"
        S = plan(mplan.num_tiles, kv.Hq, kv.Hkv, kv.D, kv.page_size, kv.max_kv_len, kv.total_kv)
        run = binding.resolve_splits(S, sms, mplan.num_tiles, kv.Hq, kv.Hkv, kv.D, kv.page_size, kv.max_kv_len)
        parts = (case.q, kv.k_cache, kv.v_cache, kv.block_table, kv.seq_lens)
        footprint = sum(t.numel() * t.element_size() for t in parts)
        sets = rotated(lambda i: parts if i == 0 else tuple(t.clone() for t in parts), footprint, l2)
        n = len(sets)
        plans = [binding.MultiPlan(case.q_lens, kv.Hq, kv.Hkv, dev, tokens_per_tile=mplan.tokens_per_tile)
                 for _ in sets]
        ws = [torch.empty(max(1, binding.workspace_bytes_multi(case.total_q, kv.Hq, kv.D, run)), dtype=torch.uint8,
                          device=dev) for _ in sets]
        outs = [torch.empty_like(case.q) for _ in sets]

        maxlen = kv.max_kv_len   # host values only inside the step (no device read per call)

        def call(i):
            j = i % n
            binding.decode_attn_paged_multi(*sets[j], plans[j], max_kv_len=maxlen, scale=kv.scale,
                                            num_splits=S, workspace=ws[j], out=outs[j])

        host = [parts[k].cpu().pin_memory() for k in (0, 3, 4)]
        hmap = [mplan.qo_indptr.cpu().pin_memory(), mplan.tile_batch.cpu().pin_memory(),
                mplan.tile_index.cpu().pin_memory()]
        ho = torch.empty(case.q.shape, dtype=torch.bfloat16).pin_memory()

        def h2d(i):
            j = i % n
            for k, h in zip((0, 3, 4), host):
                sets[j][k].copy_(h, non_blocking=True)
            for d, h in zip((plans[j].qo_indptr, plans[j].tile_batch, plans[j].tile_index), hmap):
                d.copy_(h, non_blocking=True)

        def d2h(i):
            ho.copy_(outs[i % n], non_blocking=True)

        lens = kv.seq_lens.cpu().tolist()
        flops = sum(4 * kv.Hq * kv.D * sum(L - ql + i + 1 for i in range(ql)) for L, ql in zip(lens, case.q_lens))
        cfg = {"workload": kv.name, "B": len(case.q_lens), "q_len": case.q_lens[0], "total_q": case.total_q,
               "Hq": kv.Hq, "Hkv": kv.Hkv, "D": kv.D, "page_size": kv.page_size, "total_kv": kv.total_kv,
               "num_tiles": mplan.num_tiles, "tokens_per_tile": mplan.tokens_per_tile, "num_splits": run,
               "kv_dtype": "bf16",
               "cold_kv": f"{n} rotated input copies of {footprint / 1e9:.2f} GB each (> 2x L2)"}
        return Leg(key, "multi-token paged decode achieved HBM GB/s (algorithmic bytes), cold KV", cfg,
                   multi_algorithmic(case), mkernel, call, (h2d, call, d2h),
                   sum(h.numel() * h.element_size() for h in host + hmap), ho.numel() * 2, 2 if run != 1 else 1, n,
                   extra={"flops": flops})

    if key == "fp8kv":
        S = plan(case.B, case.Hq, case.Hkv, case.D, case.page_size, case.max_kv_len, case.total_kv)
        run = binding.resolve_splits(S, sms, case.B, case.Hq, case.Hkv, case.D, case.page_size, case.max_kv_len)
        names = ("q", "k_codes", "v_codes", "k_scale", "v_scale", "block_table", "seq_lens")
        parts = tuple(getattr(case, nm) for nm in names)
        footprint = sum(t.numel() * t.element_size() for t in parts)
        sets = rotated(lambda i: parts if i == 0 else tuple(t.clone() for t in parts), footprint, l2)
        n = len(sets)
        ws = [torch.empty(max(1, binding.workspace_bytes(case.B, case.Hq, case.Hkv, case.D, run)), dtype=torch.uint8,
                          device=dev) for _ in sets]
        outs = [torch.empty_like(case.q) for _ in sets]

        maxlen = case.max_kv_len   # host values only inside the step (no device read per call)

        def call(i):
            j = i % n
            binding.decode_attn_paged_fp8kv(*sets[j], max_kv_len=maxlen, scale=case.scale, num_splits=S,
                                            workspace=ws[j], out=outs[j])

        host = [parts[k].cpu().pin_memory() for k in (0, 5, 6)]
        ho = torch.empty(case.q.shape, dtype=torch.bfloat16).pin_memory()

        def h2d(i):
            for k, h in zip((0, 5, 6), host):
                sets[i % n][k].copy_(h, non_blocking=True)

        def d2h(i):
            ho.copy_(outs[i % n], non_blocking=True)

        lens = case.seq_lens.cpu()
        cfg = {"workload": case.name, "B": case.B, "Hq": case.Hq, "Hkv": case.Hkv, "D": case.D,
               "page_size": case.page_size, "kv_len_min": int(lens.min()), "kv_len_max": int(lens.max()),
               "total_kv": case.total_kv, "num_splits": run, "kv_dtype": "e4m3 + bf16 factor per (slot, kv head)",
               "cold_kv": f"{n} rotated input copies of {footprint / 1e9:.2f} GB each (> 2x L2)"}
        return Leg(key, "paged decode attention over an e4m3 KV cache, achieved HBM GB/s (algorithmic bytes), "
                        "cold KV", cfg, fp8kv_algorithmic(case), "fp8kv_kernel", call, (h2d, call, d2h),
                   sum(h.numel() * h.element_size() for h in host), ho.numel() * 2, 2 if run != 1 else 1, n)
    raise SystemExit(f"unknown workload {key}")


# ---- timing ------------------------------------------------------------------------------

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
    import torch.distributed as dist
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


def measure(leg: Leg, K, W, stream, world=1, clocks: ClockSampler | None = None):
    """Times `leg.step(i)` (inputs resident, rotated copies):
      - ms_loop: K back-to-back steps bracketed by two CUDA events (after a barrier and a
        synchronize on both sides), clocks sampled meanwhile when `clocks` is given;
      - us_per_call: median of K per-call times, events at every call boundary;
      - kernel_us: median of the attention kernel's own time per launch (events the library
        records around its launch, or, for a kernel without them, a CUDA graph of 50 calls
        replayed: the median replay time over 50);
      - e2e_ms: the end-to-end step through host buffers (time_e2e)."""
    import torch.distributed as dist
    from paged_kv_cache_298_gb300 import binding
    for i in range(W):
        leg.step(i)
    torch.cuda.synchronize()
    if binding.get_device_errors(clear=True):
        raise SystemExit(f"{leg.key}: device error word set during warm-up")
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clk = None
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        leg.step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms_loop = t0.elapsed_time(t1) / K

    # per-call times: an event at every call boundary
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    for e in ev:   # torch creates the CUDA event on first record
        e.record(stream)
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(K):
        leg.step(i)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    per_call = [ev[i].elapsed_time(ev[i + 1]) for i in range(K)]

    graph_ms = graph_time(leg.step, K, stream)
    combine_ms = None
    if leg.trace:
        tr = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for e in tr:
            for x in e:
                x.record(stream)
        torch.cuda.synchronize()
        for i in range(K):
            binding.set_trace_events(*tr[i])
            leg.step(i)
        torch.cuda.synchronize()
        binding.set_trace_events()
        kern = [e[0].elapsed_time(e[1]) for e in tr]
        combine_ms = statistics.median(e[1].elapsed_time(e[2]) for e in tr)
        kernel_timing = f"median of {K} launches, events around the launch"
    else:   # one kernel per call: the graph-replayed call is the kernel
        kern = [graph_ms]
        kernel_timing = f"CUDA graph of {max(K, 20)} calls, median of 5 replays"
    errs = binding.get_device_errors(clear=True)
    e2e_ms, sched = time_e2e(*leg.e2e, K, W, leg.copies, stream, world)
    return {"ms_loop": ms_loop, "call_ms": statistics.median(per_call), "kern_ms": statistics.median(kern),
            "graph_ms": graph_ms, "combine_ms": combine_ms, "kernel_timing": kernel_timing, "e2e_ms": e2e_ms,
            "e2e_schedule": sched, "errors": errs, "clocks": clk}


def graph_time(step, K, stream, reps=5):
    """Device milliseconds per call with the host out of the way: max(K, 20) calls (the same
    rotation of input copies) captured in one CUDA graph, replayed `reps` times; the median
    replay over the calls in it."""
    per = max(K, 20)
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
    res = []
    for _ in range(reps):
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        graph.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        res.append(g0.elapsed_time(g1) / per)
    return statistics.median(res)


def compact(leg: Leg, r, hbm_peak, cpu):
    """The `workloads` entry of one leg."""
    gbs = lambda ms: round(leg.nbytes / (ms * 1e-3) / 1e9, 1)
    out = {"metric": leg.metric, "config": leg.config, "algorithmic_bytes": leg.nbytes,
           "us_per_call": round(r["call_ms"] * 1e3, 2), "gb_s": gbs(r["call_ms"]),
           "frac": round(leg.nbytes / (r["call_ms"] * 1e-3) / 1e9 / hbm_peak, 4),
           "graph_us_per_call": round(r["graph_ms"] * 1e3, 2), "graph_gb_s": gbs(r["graph_ms"]),
           "graph_frac": round(leg.nbytes / (r["graph_ms"] * 1e-3) / 1e9 / hbm_peak, 4),
           "kernel": {"name": leg.kernel, "us": round(r["kern_ms"] * 1e3, 2), "gb_s": gbs(r["kern_ms"]),
                      "frac": round(leg.nbytes / (r["kern_ms"] * 1e-3) / 1e9 / hbm_peak, 4),
                      "timing": r["kernel_timing"],
                      "traffic": recorded_traffic(leg.kernel, leg.key) if leg.kernel in KERNEL_SOURCES else None},
           "loop_us_per_call": round(r["ms_loop"] * 1e3, 2),
           "e2e": {"schedule": r["e2e_schedule"], "gb_s": gbs(r["e2e_ms"]), "us_per_call": round(r["e2e_ms"] * 1e3, 2),
                   "h2d_bytes_per_step": leg.h2d_bytes, "d2h_bytes_per_step": leg.d2h_bytes},
           "device_errors": r["errors"], "cpu_baseline": cpu}
    if r["combine_ms"] is not None:
        out["kernel"]["combine_us"] = round(r["combine_ms"] * 1e3, 2)
    if "flops" in leg.extra:
        out["kernel"]["tflops"] = round(leg.extra["flops"] / (r["kern_ms"] * 1e-3) / 1e12, 2)
    return out


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
    hbm_peak, peak_src = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.current_stream()
    key = args.workload or "ragged"
    case = make_case(key, dev, args.batch)
    leg = prepare_leg(key, case, dev, l2, args.splits, args.tpt or None)
    K, W = args.steps, args.warmup
    clocks = ClockSampler(local)
    r = measure(leg, K, W, stream, world, clocks)
    (value, ms), (e2e_value, e2e_ms) = job_throughput([r["ms_loop"], r["e2e_ms"]], leg.nbytes, world, dev)
    achieved = leg.nbytes / (r["kern_ms"] * 1e-3) / 1e9
    wkey = key if not args.batch else f"{key}_b{args.batch}"
    line = {
        "metric": leg.metric, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms, 5), "us_per_call": round(r["call_ms"] * 1e3, 2),
        "graph_us_per_call": round(r["graph_ms"] * 1e3, 2),
        "graph_frac": round(leg.nbytes / (r["graph_ms"] * 1e-3) / 1e9 / hbm_peak, 4),
        "statistic": "value and ms_per_step: the K-step region bracketed by two CUDA events; us_per_call: median "
                     "of K per-call times (events at every call boundary, host binding included); "
                     "graph_us_per_call: the same calls replayed from a CUDA graph (device time per call)",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": leg.config, "pct_of_peak": round(100 * value / world / hbm_peak, 1),
        "roofline": {"bound": "hbm", "kernel": leg.kernel, "achieved": round(achieved, 1), "peak": hbm_peak,
                     "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "kernel_ms": round(r["kern_ms"], 5), "kernel_timing": r["kernel_timing"],
                     "combine_ms": None if r["combine_ms"] is None else round(r["combine_ms"], 5),
                     "algorithmic_bytes_per_launch": leg.nbytes,
                     "traffic": recorded_traffic(leg.kernel, wkey)},
        "e2e": {"schedule": r["e2e_schedule"], "value": round(e2e_value, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": leg.h2d_bytes,
                "d2h_bytes_per_step": leg.d2h_bytes},
        "gpu_launches": K * leg.launches, "device_errors": r["errors"], "clocks": r["clocks"],
    }
    if "flops" in leg.extra:
        line["roofline"]["tflops"] = round(leg.extra["flops"] / (r["kern_ms"] * 1e-3) / 1e12, 2)
    del leg
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = oracle_sample(key, case)
        line["cpu_baseline"] = s.measure(6.0)
        cores = s.oracle.num_threads()
        s.oracle.set_num_threads(1)
        try:
            one = s.measure(1.5)
        finally:
            s.oracle.set_num_threads(cores)
        line["cpu_baseline"]["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}
    del case
    torch.cuda.empty_cache()
    if world == 1 and args.workload is None and not args.no_legs:
        legs, clocks_all = {}, ClockSampler(local)
        clocks_all.start()
        for lk in LEGS:
            c = make_case(lk, dev)
            lg = prepare_leg(lk, c, dev, l2)
            lr = measure(lg, K, W, stream)
            cpu = None
            if not args.no_cpu_baseline:
                cpu = oracle_sample(lk, c).measure(0.8)
            legs[lk] = compact(lg, lr, hbm_peak, cpu)
            del lg, c
            torch.cuda.empty_cache()
        line["workloads"] = legs
        line["workloads_clocks"] = clocks_all.stop()
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
        the Python binding's host cost (about 10 us a call) does not starve the GPU; the
        median of the replays."""
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
        res = []
        for _ in range(max(5, K // per)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            res.append(e0.elapsed_time(e1) / per)
        return statistics.median(res)

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
        "gpu_launches": 2 * 50 * max(5, K // 50), "device_errors": binding.get_device_errors()}), flush=True)


# ---- reference arm: the fp64 oracle on the host cores ----------------------------------

def run_reference(args):
    """The oracle, as it stands, on the host cores, on the same workload and metric as our
    arm: each step one pass over a prefix of the workload sized so that the whole run ends
    within a few minutes."""
    rank, _, world = rank_info()
    if rank != 0:
        return
    key = args.workload or "ragged"
    if key == "append":
        print(json.dumps({"impl": "reference", "unavailable": "the append workload has no oracle timing leg"}))
        return
    case = make_case(key, "cpu")
    s = oracle_sample(key, case)
    n = s.size_for(min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        s.run(n)
    times = [s.run(n) for _ in range(args.steps)]
    dt = statistics.median(times)
    value = s.nbytes(n) / dt / 1e9
    sample = f"fp64 oracle (OpenMP) on {s.unit_name} 0..{n - 1} of {s.units} per step"
    c = case[0] if key == "masked" else case
    name = getattr(c, "name", "") or getattr(getattr(c, "kv", None), "name", key)
    metric = {"fp8": "fp8 sliding-window latent decode achieved HBM GB/s (algorithmic bytes), cold inputs",
              "multi": "multi-token paged decode achieved HBM GB/s (algorithmic bytes), cold KV",
              "multi_g8": "multi-token paged decode achieved HBM GB/s (algorithmic bytes), cold KV",
              "multi_g8_q8": "multi-token paged decode achieved HBM GB/s (algorithmic bytes), cold KV",
              "fp8kv": "paged decode attention over an e4m3 KV cache, achieved HBM GB/s (algorithmic bytes), cold KV",
              "masked": "masked paged decode achieved HBM GB/s (algorithmic bytes), cold KV",
              "llama_contig": "contiguous-cache decode achieved HBM GB/s (algorithmic bytes), cold KV"}.get(
        key, "paged decode attention achieved HBM GB/s (algorithmic bytes), cold KV")
    print(json.dumps({
        "impl": "reference", "metric": metric, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "statistic": "median of the steps", "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "sample_units": n, "cold_kv": "host memory (oracle on the CPU cores)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": s.oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, choices=WORKLOADS,
                    help="time this workload alone (default: the ragged headline plus every other "
                         "configuration under 'workloads')")
    ap.add_argument("--splits", type=int, default=None,
                    help="num_splits passed to the library (default: the planner's S made with the summed "
                         "lengths; 0 = the library's own plan; -1 = balanced schedule; S > 0 = per-sequence)")
    ap.add_argument("--tpt", type=int, default=0,
                    help="multi-token workloads: tokens per work-map tile (0 = the library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-legs", action="store_true", help="the headline only")
    ap.add_argument("--batch", type=int, default=0,
                    help="ragged / multi / e4m3 workloads: number of sequences (0 = the workload's own, 128); "
                         "smaller batches are for profiler captures")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "append":
        run_append(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
