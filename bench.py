#!/usr/bin/env python3
"""Throughput of the DSA indexer paged MQA-logits on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-configs] [--kernel-ms MS]

One step is one pass of the indexer over one batch of synthetic inputs.  The
default workload is the bf16 decode batch (B=64, W=2048, lengths
log-uniform 4K..128K: 635 MB per call), the largest configuration of the
five on one GPU.  Inputs are device-resident when the timed region starts; K
steps run as CUDA-graph replays, bracketed by a barrier and synchronisations
and timed with CUDA events on the launching stream.  Input and output buffers
rotate among enough copies that every step reads HBM, not L2.

Prints one JSON line (rank 0).  `value` is key positions scored per second
over all ranks (weak scaling: each rank runs the same per-GPU workload).
`roofline` is the dominant kernel's, from a separate region of back-to-back
launches at least --kernel-ms long.  `configs` holds one such record for
every configuration (1, both calls of 2, 3 at W=4097 and W=512, the short
lengths at W=4097 and W=32, 4 and 5), each against MEASURED_PEAKS.json.
`--impl reference` times the fp64 CPU oracle on the host cores instead.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_paged_gb300 import workloads as wl  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0

WORKLOAD_DESC = {
    "1": "decode fp8 B=1 W=8 L~U[1,512]",
    "2": "decode fp8 B=16 W=32 L~U[1,2048] + B=32 W=16 L~U[1,1024]",
    "2a": "decode fp8 B=16 W=32 L~U[1,2048]",
    "2b": "decode fp8 B=32 W=16 L~U[1,1024]",
    "3": "decode fp8 B=64 W=4097 L log-uniform 512..32768",
    "3ref": "decode fp8 B=64 W=512 L log-uniform 512..32768",
    "3short": "decode fp8 B=64 W=4097 L log-uniform 512..2048",
    "3short_capped": "decode fp8 B=64 W=32 L log-uniform 512..2048",
    "4": "decode bf16 B=64 W=2048 L log-uniform 4096..131072",
    "4s": "decode bf16 B=64 W=512 L log-uniform 1024..32768 (config 4's kernel, profile-sized)",
    "5": "prefill bf16 n_q=4096 W=352 causal limit 18432+i",
    "6": "prefill bf16, 4 requests (query tokens, context) = (256, 6144), (512, 12288), "
         "(128, 3072), (1024, 20480), per-query table rows",
    "6v": "prefill bf16, the same 4 requests, one table row per request (all requests' query "
          "tiles in one launch)",
    "7": "prefill fp8 n_q=1024 W=128 causal limit 7168+i",
    "8": "key-cache store: 65536 bf16 key rows into e4m3 pages (+ scales), random slots of 2048 pages",
    "9": "decode fp8 B=64 W=4097 L log-uniform 512..32768, top-2048 positions per request",
    "9k256": "decode fp8 B=64 W=4097 L log-uniform 512..32768, top-256 positions per request",
    "9k512": "decode fp8 B=64 W=4097 L log-uniform 512..32768, top-512 positions per request",
}
# default (steps, warmup): a timed region of roughly one second per GPU
DEFAULT_STEPS = {"1": 100000, "2": 100000, "2a": 100000, "2b": 100000, "3": 20000, "3ref": 20000, "3short": 40000,
                 "3short_capped": 100000, "4": 10000, "4s": 40000, "5": 1000, "6": 2000, "6v": 2000, "7": 5000,
                 "8": 10000, "9": 20000, "9k256": 20000, "9k512": 20000}
METRIC = "indexer key-positions scored/s & achieved HBM GB/s (frac of roofline), 1 GB300"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="4", choices=sorted(wl.NAMED))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration records")
    ap.add_argument("--kernel-ms", type=float, default=200.0,
                    help="device time of each back-to-back kernel region")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget-s", type=float, default=60.0,
                    help="host-time budget of the reference (oracle) arm")
    ap.add_argument("--profile", type=int, default=0, metavar="N",
                    help="only run each call of one step N times (for ncu) and exit")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)

        def pick(*names):
            for n in names:
                if n in d and isinstance(d[n], (int, float)):
                    return float(d[n])
            return None
        hbm = pick("hbm_gbs", "hbm_GBs", "hbm_copy_gbs")
        bf = pick("bf16_tflops", "bf16_tflops_burst")
        bfs = pick("bf16_tflops_sustained")
        if hbm and bf:
            return {"hbm_gbs": hbm, "bf16_tflops": bf,
                    "bf16_tflops_sustained": bfs or bf, "source": "measured"}
    except (OSError, ValueError):
        pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED, "source": "fallback"}


KERNEL_SOURCES = {   # each kernel's own source and the shared code it includes
    kind: (f"{kind}_sm103.cu", "dsa_common.cuh", "sm100_ptx.cuh", "tensor_maps.cu",
           "tensor_maps.cuh")
    for kind in ("decode", "prefill", "store")
}
KERNEL_SOURCES["decode"] += ("topk_slots.cuh",)
# decode, then the selection (two passes) or the merge (fused)
KERNEL_SOURCES["topk"] = KERNEL_SOURCES["decode"] + ("topk_sm103.cu", "topk_fused_sm103.cu")


def kernel_source_hash(kernel: str | None = None):
    """Hash of a kernel's source code (all kernels' when kernel is None):
    comments and whitespace are left out, so that an edited comment does not
    disown a profile of the same code."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_paged_gb300", "csrc")
    names = KERNEL_SOURCES[kernel] if kernel else os.listdir(csrc)
    for f in sorted(names):
        if f.endswith((".cu", ".cuh")) and os.path.exists(os.path.join(csrc, f)):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                code = fh.read()
            code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
            code = re.sub(r"//[^\n]*", " ", code)
            code = re.sub(r"\s+", " ", code)
            h.update(f.encode())
            h.update(code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(f"{kernel}@{workload}")
        if e and e.get("kernel_source_hash") == kernel_source_hash(kernel):
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.samples.append((time.time(), line.strip()))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        used = inside if inside else rows
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in used:
            for n, v in zip(names, r[3][5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        out = {"sm_mhz": statistics.median(r[1] for r in used),
               "sm_max_mhz": max(r[2] for r in used), "reasons": sorted(reasons),
               "samples": len(used)}
        if not inside:
            out["note"] = "timed region shorter than the sampling period; nearest samples"
        return out


# ---------------------------------------------------------------------------
# aggregation over ranks (weak scaling: every rank runs the same per-GPU work)

def max_over_ranks(elapsed_ms: float, device=None) -> float:
    """The slowest rank's time: the job is done when every rank is."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, units_per_step: int, elapsed_ms: float) -> float:
    """Units processed by all ranks per second of the slowest rank's time."""
    return world * steps * units_per_step / (elapsed_ms / 1e3)


# ---------------------------------------------------------------------------
# our arm

VARLEN_REQUESTS_PER_LAUNCH = 128    # the library's request map per varlen launch


class DeviceCall:
    """One library call with device-resident inputs and its own output."""

    def __init__(self, w, device, views=None):
        """`views`: this copy's device tensors (q, wt, kcache, bt, seqlens,
        out, status), carved from stacked allocations by make_copies; None =
        allocate and upload its own."""
        import torch
        self.w = w
        self._fn = None
        self.cu_q = None                       # request offsets of a varlen prefill call
        if views is not None:
            for name, t in views.items():
                setattr(self, name, t)
            self.kscale = (None if w.kscale_offset is None
                           else self.kcache.data_ptr() + w.kscale_offset)
            return
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        if w.kind == "store":
            self.k = torch.from_numpy(w.k_bits.view(np.int16)).to(device)
            self.slots = torch.from_numpy(w.slots).to(device)
            self.kcache = torch.from_numpy(w.kcache).to(device)
            return
        self.q = torch.from_numpy(w.q_bits.view(np.int16)).to(device)
        self.wt = torch.from_numpy(w.w).to(device)
        self.kcache = torch.from_numpy(w.kcache).to(device)
        if w.meta.get("varlen"):              # one table row per request, and the offsets
            self.cu_q, self.req_table = wl.request_tables(w)
            self.bt = torch.from_numpy(self.req_table).to(device)
        else:
            self.bt = torch.from_numpy(w.block_table).to(device)
        self.seqlens = torch.from_numpy(w.seqlens).to(device)
        if w.kind == "topk":
            k = w.meta["k_top"]
            self.idx = torch.empty((w.R, k), dtype=torch.int32, device=device)
            self.val = torch.empty((w.R, k), dtype=torch.float32, device=device)
            self.ws = torch.empty(w.R * w.W * w.P, dtype=torch.float32, device=device)
            self.out = self.idx
        else:
            self.out = torch.empty((w.R, w.W * w.P), dtype=torch.float32, device=device)
        self.kscale = (None if w.kscale_offset is None
                       else self.kcache.data_ptr() + w.kscale_offset)

    def host_table(self):
        """The block table this call copies in: per request or per row."""
        return self.req_table if self.cu_q is not None else self.w.block_table

    def launches(self):
        """Kernels one call launches."""
        if self.w.kind == "topk":
            return 2
        if self.cu_q is not None:
            # the varlen prefill: one launch per group of up to
            # VARLEN_REQUESTS_PER_LAUNCH requests that holds any row
            c, n = list(self.cu_q), len(self.cu_q) - 1
            g = VARLEN_REQUESTS_PER_LAUNCH
            return sum(1 for b0 in range(0, n, g) if c[min(b0 + g, n)] > c[b0])
        return 1

    def nbytes(self):
        if self.w.kind == "store":
            ts = (self.k, self.slots, self.kcache)
        elif self.w.kind == "topk":
            ts = (self.q, self.wt, self.kcache, self.bt, self.seqlens, self.idx, self.val, self.ws)
        else:
            ts = (self.q, self.wt, self.kcache, self.bt, self.seqlens, self.out)
        return sum(t.numel() * t.element_size() for t in ts)

    def store(self, k=None, slots=None):
        import torch
        import sparse_attention_paged_gb300 as lib
        w = self.w
        st = lib.dsa_kcache_store(self.k if k is None else k, self.slots if slots is None else slots,
                                  w.n, self.kcache, w.page_stride, w.num_pages, w.kv_dtype,
                                  w.D, w.P, self.status, torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise RuntimeError(f"library call failed: {lib.dsa_status_string(st)}")

    def __call__(self, q=None, wt=None, bt=None, seqlens=None, out=None):
        import torch
        import sparse_attention_paged_gb300 as lib
        w = self.w
        if w.kind == "store":
            return self.store()
        if w.kind == "topk":
            k = w.meta["k_top"]
            st = lib.dsa_indexer_topk_decode(
                self.q if q is None else q, self.wt if wt is None else wt, self.kcache,
                self.kscale, w.page_stride, w.num_pages, w.kv_dtype,
                self.bt if bt is None else bt, w.bt_stride,
                self.seqlens if seqlens is None else seqlens, w.R, w.H, w.D, w.P, w.W, k,
                self.idx, self.val, k, self.ws, self.ws.numel(), self.status,
                torch.cuda.current_stream().cuda_stream)
            if st != 0:
                raise RuntimeError(f"library call failed: {lib.dsa_status_string(st)}")
            if out is not None and out is not self.idx:     # e2e: both results to one buffer
                out[:, :k].copy_(self.idx.view(torch.float32))
                out[:, k:].copy_(self.val)
            return
        if self.cu_q is not None:
            out = self.out if out is None else out
            st = lib.dsa_indexer_logits_prefill_varlen(
                self.q if q is None else q, self.wt if wt is None else wt, self.kcache,
                self.kscale, w.page_stride, w.num_pages, w.kv_dtype,
                self.bt if bt is None else bt, w.W, self.cu_q,
                self.seqlens if seqlens is None else seqlens, w.H, w.D, w.P, w.W, out,
                out.stride(0), self.status, torch.cuda.current_stream().cuda_stream)
            if st != 0:
                raise RuntimeError(f"library call failed: {lib.dsa_status_string(st)}")
            return
        if self._fn is None:
            self._fn = (lib.dsa_indexer_logits_decode if w.kind == "decode"
                        else lib.dsa_indexer_logits_prefill)
            self._ptrs = (self.q.data_ptr(), self.wt.data_ptr(), self.kcache.data_ptr(),
                          self.bt.data_ptr(), self.seqlens.data_ptr(), self.out.data_ptr(),
                          self.status.data_ptr())
        pq, pw, pk, pb, ps, po, pst = self._ptrs
        out = self.out if out is None else out
        st = self._fn(pq if q is None else q.data_ptr(), pw if wt is None else wt.data_ptr(), pk,
                      self.kscale, w.page_stride, w.num_pages, w.kv_dtype,
                      pb if bt is None else bt.data_ptr(), w.bt_stride,
                      ps if seqlens is None else seqlens.data_ptr(), w.R, w.H, w.D, w.P, w.W,
                      po if out is self.out else out.data_ptr(), out.stride(0), pst,
                      torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise RuntimeError(f"library call failed: {lib.dsa_status_string(st)}")


# every configuration of the indexer's five, each timed on its own (config 2
# is two calls of different shape: both are listed)
SWEEP = ("1", "2a", "2b", "3", "3ref", "3short", "3short_capped", "4", "5")


def n_copies_for(works):
    """Copies of a step's inputs and outputs to rotate over, so that one pass
    over them moves more than twice the L2's bytes (every launch then reads
    HBM, not L2)."""
    per = sum(w.algorithmic_bytes() for w in works)
    return max(1, math.ceil(2 * L2_BYTES / max(per, 1)))


def make_copies(works, device, n):
    """n independent copies of every call of a step: own inputs, own output,
    own status word.  For plain decode and prefill calls each field of all
    copies is one stacked device allocation (so a small workload can rotate
    over thousands of copies); other calls allocate each copy on its own."""
    import torch
    out = [[None] * len(works) for _ in range(n)]
    for j, w in enumerate(works):
        if w.kind not in ("decode", "prefill") or w.meta.get("varlen"):
            for i in range(n):
                out[i][j] = DeviceCall(w, device)
            continue

        def stack(a):
            t = torch.from_numpy(np.ascontiguousarray(a)).to(device)
            return t.unsqueeze(0).expand(n, *t.shape).contiguous()
        q, wt, kc = stack(w.q_bits.view(np.int16)), stack(w.w), stack(w.kcache)
        bt, sl = stack(w.block_table), stack(w.seqlens)
        o = torch.empty((n, w.R, w.W * w.P), dtype=torch.float32, device=device)
        st = torch.zeros((n, 4), dtype=torch.int32, device=device)
        for i in range(n):
            out[i][j] = DeviceCall(w, device, views=dict(
                q=q[i], wt=wt[i], kcache=kc[i], bt=bt[i], seqlens=sl[i], out=o[i],
                status=st[i, :1]))
    return out


def kernel_region(copies, idx, min_ms):
    """Average duration of call `idx` of a step, launched back to back over
    the rotating copies: one CUDA graph that walks every copy (at least 64
    launches), replayed until at least `min_ms` of device time has passed,
    with CUDA events on the launching stream at the region's two ends only
    (an event pair around every launch would add microseconds to each).
    Returns (us per launch, launches, region ms, wall-clock start, end)."""
    import torch
    n = len(copies)
    Lg = n * max(1, math.ceil(64 / n))
    for i in range(n):                            # first touch of every copy, untimed
        copies[i][idx]()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(Lg):
            copies[i % n][idx]()
    g.replay()                                    # first replay, untimed
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    reps = max(1, math.ceil(min_ms / max(e0.elapsed_time(e1), 1e-3)))
    t_wall0 = time.time()
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    ms = e0.elapsed_time(e1)
    del g
    return ms * 1e3 / (reps * Lg), reps * Lg, ms, t_wall0, t_wall1


def roofline_record(w, us, peaks):
    """One call's roofline: algorithmic bytes over HBM bandwidth against
    FLOPs over the bf16 tensor peak, whichever is slower."""
    s = us / 1e6
    t_hbm = w.algorithmic_bytes() / (peaks["hbm_gbs"] * 1e9)
    t_tc = w.flops() / (peaks["bf16_tflops"] * 1e12)
    rec = {"algorithmic_bytes": w.algorithmic_bytes(), "flops": w.flops(),
           "t_roof_us": max(t_hbm, t_tc) * 1e6}
    if w.kind == "prefill" or t_tc > t_hbm:
        ach = w.flops() / s / 1e12
        rec.update(bound="tensor", achieved=ach, unit="TFLOP/s", peak=peaks["bf16_tflops"],
                   frac=ach / peaks["bf16_tflops"],
                   peak_sustained=peaks["bf16_tflops_sustained"],
                   frac_sustained=ach / peaks["bf16_tflops_sustained"])
    else:
        ach = w.algorithmic_bytes() / s / 1e9
        rec.update(bound="hbm", achieved=ach, unit="GB/s", peak=peaks["hbm_gbs"],
                   frac=ach / peaks["hbm_gbs"])
    return rec


def config_record(name, w, us, launches, region_ms, n_copies, resident, peaks, clocks):
    rec = {"workload": WORKLOAD_DESC[name], "call": w.name, "kernel": w.kind,
           "avg_launch_us": us, "launches": launches, "region_ms": region_ms,
           "positions_per_s": w.valid_positions / (us / 1e6)}
    rec.update(roofline_record(w, us, peaks))
    # ncu DRAM bytes per launch, where profiles/dram_traffic.json holds them
    # for the current kernel sources (else None)
    rec["traffic"] = recorded_traffic(w.kind, w.name)
    rec["l2"] = (f"rotates over {n_copies} copies ({resident / 2**20:.0f} MiB resident)")
    rec["clocks"] = clocks
    return rec


def run_config_sweep(device, peaks, sampler, min_ms, reuse):
    """Every configuration's dominant kernel on its own: a record each with
    its back-to-back launch time and roofline fraction.  `reuse` maps a
    workload name to a record already measured in this run."""
    import torch
    out = {}
    for name in SWEEP:
        if name in reuse:
            out[name] = reuse[name]
            continue
        works = wl.NAMED[name]()
        n = n_copies_for(works)
        copies = make_copies(works, device, n)
        resident = sum(c.nbytes() for cs in copies for c in cs)
        us, launches, ms, t0, t1 = kernel_region(copies, 0, min_ms)
        for cs in copies:
            for c in cs:
                if int(c.status.item()) != 0:
                    raise RuntimeError(f"{name}: kernel status {int(c.status.item())}")
        out[name] = config_record(name, works[0], us, launches, ms, n, resident, peaks,
                                  sampler.summary(t0, t1))
        del copies
        torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from sparse_attention_paged_gb300 import _native

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    _native.load()
    works = wl.NAMED[args.workload]()
    step_bytes = sum(w.algorithmic_bytes() for w in works)
    step_positions = sum(w.valid_positions for w in works)
    step_flops = sum(w.flops() for w in works)
    n_copies = n_copies_for(works)
    copies = make_copies(works, device, n_copies)
    resident = sum(c.nbytes() for cs in copies for c in cs)

    K = args.steps if args.steps is not None else DEFAULT_STEPS[args.workload]
    Wm = max(3, args.warmup if args.warmup is not None else max(3, K // 100))
    S = min(K, 500)                           # steps per captured graph

    def capture(n_steps, offset):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_steps):
                for c in copies[(offset + i) % n_copies]:
                    c()
        return g

    # the dominant kernel: the call with the largest algorithmic roofline time
    peaks = read_peaks()

    def roof_time(w):
        tb = w.algorithmic_bytes() / (peaks["hbm_gbs"] * 1e9)
        tf = w.flops() / (peaks["bf16_tflops"] * 1e12)
        return max(tb, tf)
    dom_idx = max(range(len(works)), key=lambda j: roof_time(works[j]))
    dom = works[dom_idx]

    # warm-up (untimed), graphs of the same shape as the timed ones
    for c in [c for cs in copies for c in cs]:
        c()
    torch.cuda.synchronize()
    wg = capture(min(Wm, S), 0)
    done = 0
    while done < Wm:
        wg.replay()
        done += min(Wm, S)
    torch.cuda.synchronize()

    # the timed graphs: K = reps * S + rem steps, no event nodes inside (an
    # event pair around a launch inside a graph costs microseconds)
    reps, rem = divmod(K, S)
    g_main = capture(S, 0)
    g_rem = capture(rem, (reps * S) % n_copies) if rem else None
    # one untimed replay of each so that first-replay costs stay outside
    g_main.replay()
    if g_rem is not None:
        g_rem.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record()
    for _ in range(reps):
        g_main.replay()
    if g_rem is not None:
        g_rem.replay()
    e1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    elapsed_ms = e0.elapsed_time(e1)
    del g_main, g_rem, wg

    # per-launch duration of the dominant kernel: a second timed region of
    # back-to-back launches of that call alone (rotating copies, at least
    # args.kernel_ms of device time), events at the region's ends, on the
    # same stream
    dom_us, dom_launches, dom_region_ms, k_wall0, k_wall1 = kernel_region(
        copies, dom_idx, args.kernel_ms)
    kernel_timing = (f"{dom_launches} back-to-back launches of the dominant call over "
                     f"{dom_region_ms:.0f} ms (CUDA graph walking the copies, events at the "
                     "region's ends)")

    elapsed_ms = max_over_ranks(elapsed_ms, device)

    # status check: the timed calls raised no data error
    for cs in copies:
        for c in cs:
            if int(c.status.item()) != 0:
                raise RuntimeError(f"kernel status {int(c.status.item())}")

    value = job_throughput(world, K, step_positions, elapsed_ms)
    rr = roofline_record(dom, dom_us, peaks)
    roof = {"bound": rr["bound"], "achieved": rr["achieved"], "peak": rr["peak"],
            "unit": rr["unit"], "frac": rr["frac"]}
    if rr["bound"] == "tensor":
        roof["peak_sustained"] = rr["peak_sustained"]
        roof["frac_sustained"] = rr["frac_sustained"]
    kname = dom.kind
    roof["traffic"] = recorded_traffic(kname, dom.name)
    roof["kernel"] = f"{kname} ({dom.name})"
    roof["algorithmic_bytes_per_launch"] = dom.algorithmic_bytes()
    roof["flops_per_launch"] = dom.flops()
    roof["avg_launch_us"] = dom_us
    roof["peak_source"] = ("MEASURED_PEAKS.json (of measured)" if peaks["source"] == "measured"
                           else "profiling recipe's fallback (of fallback)")
    roof["kernel_timing"] = kernel_timing

    main_clocks = sampler.summary(t_wall0, t_wall1)
    kernel_clocks = sampler.summary(k_wall0, k_wall1)
    line = {
        "metric": METRIC, "value": value, "unit": "key-positions/s",
        "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": (("bf16 keys -> e4m3 codes + f32 scale" if dom.kv_dtype == wl.KV_E4M3
                   else "bf16 keys copied") if dom.kind == "store" else
                  "e4m3 keys x bf16 q -> f32" if dom.kv_dtype == wl.KV_E4M3 else "bf16 -> f32"),
        "data": "synthetic (seeded generator; no dataset)",
        "config": {"workload": WORKLOAD_DESC[args.workload],
                   "calls_per_step": len(works),
                   "positions_per_step": step_positions,
                   "algorithmic_bytes_per_step": step_bytes,
                   "flops_per_step": step_flops,
                   "l2": f"inputs and outputs rotate over {n_copies} copies "
                         f"({resident / 2**20:.0f} MiB resident, > 2x L2)",
                   "timing": f"CUDA graphs of {S} steps, events on the launching stream",
                   "parallelism": f"replicas x{world} (requests are independent)"},
        "gb_per_s": K * step_bytes / (elapsed_ms / 1e3) / 1e9,
        "roofline": roof,
        # the timed steps may be shorter than one clock sample: where they
        # are, the clocks are those of the dominant kernel's region (the same
        # kernel, right after), which is at least args.kernel_ms long
        "clocks": (main_clocks if "note" not in main_clocks else
                   dict(kernel_clocks, window="dominant-kernel region (the timed steps were "
                                                "shorter than one 100 ms sample)")),
        # a top-k call is two kernels (logits, then the selection); a varlen
        # prefill call one per request
        "gpu_launches": K * sum(c.launches() for c in copies[0]),
        "gpu_launches_kernel_region": dom_launches * copies[0][dom_idx].launches(),
    }
    main_record = None
    if len(works) == 1 and args.workload in SWEEP:
        main_record = config_record(args.workload, dom, dom_us, dom_launches, dom_region_ms,
                                    n_copies, resident, peaks, kernel_clocks)
    del copies
    torch.cuda.empty_cache()

    if not args.no_e2e:
        line["e2e"] = (run_e2e_store(works, device, min(K, 2000)) if dom.kind == "store"
                       else run_e2e(works, device, K))
    if not args.no_configs:
        line["configs"] = run_config_sweep(
            device, peaks, sampler, args.kernel_ms,
            {args.workload: main_record} if main_record else {})
    sampler.stop()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(works)
    if rank == 0:
        print(json.dumps(line), flush=True)


def _time_e2e_steps(step, n_steps):
    """Time n_steps end-to-end steps two ways: eagerly (every call issued
    from Python) and as replays of a CUDA graph of up to 100 steps (the
    library calls are capturable); every step, either way, copies its own
    inputs in and its results out.  Returns (graph ms, eager ms, steps)."""
    import torch
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n_steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1)
    G = min(100, n_steps)
    reps = max(1, n_steps // G)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(G):
            step()
    g.replay()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), eager_ms, reps * G, G


def run_e2e(works, device, n_steps):
    """The same metric through the public API with host buffers.  Every step
    copies its inputs (q, w, block tables and lengths of every call, packed
    in one pinned staging buffer) to the device in one copy, runs the calls
    and copies all results back to pinned memory in one copy; the key cache
    stays resident on the device, as in serving.  Steps are pipelined over
    two device buffer sets: step i+1's upload (copy stream) and step i-1's
    download (a second copy stream) run while step i computes; events order
    each buffer's reuse.  The same steps run one after another on one stream
    are reported beside it (`serial_*`)."""
    import torch
    calls = [DeviceCall(w, device) for w in works]

    def pack(tensors):
        offs, total = [], 0
        for t in tensors:
            total = (total + 15) // 16 * 16
            offs.append(total)
            total += t.numel() * t.element_size()
        return offs, total

    host_parts = []
    for c in calls:
        host_parts += [torch.from_numpy(c.w.q_bits.view(np.int16)), torch.from_numpy(c.w.w),
                       torch.from_numpy(c.host_table()), torch.from_numpy(c.w.seqlens)]
    in_offs, in_total = pack(host_parts)
    h_in = torch.empty(in_total, dtype=torch.uint8).pin_memory()
    for t, o in zip(host_parts, in_offs):
        n = t.numel() * t.element_size()
        h_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
    outs_meta = [torch.empty((c.w.R, 2 * c.w.meta["k_top"]) if c.w.kind == "topk" else c.out.shape,
                             dtype=torch.float32) for c in calls]
    out_offs, out_total = pack(outs_meta)

    slots = []
    for _ in range(2):
        d_in = torch.empty(in_total, dtype=torch.uint8, device=device)
        d_out = torch.empty(out_total, dtype=torch.uint8, device=device)
        views = [d_in[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for t, o in zip(host_parts, in_offs)]
        outs = [d_out[o:o + m.numel() * 4].view(torch.float32).view(m.shape)
                for o, m in zip(out_offs, outs_meta)]
        h_out = torch.empty(out_total, dtype=torch.uint8).pin_memory()
        slots.append((d_in, d_out, views, outs, h_out))

    def run_calls(views, outs):
        for j, c in enumerate(calls):
            q, wt, bt, sl = views[4 * j: 4 * j + 4]
            c(q=q, wt=wt, bt=bt, seqlens=sl, out=outs[j])

    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {(k, s): torch.cuda.Event() for k in ("in", "comp", "out") for s in (0, 1)}

    def pipelined(n):
        """n pipelined steps; returns the device ms from the first upload to
        the last download."""
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        up.wait_stream(comp)
        down.wait_stream(comp)
        for i in range(n):
            s = i & 1
            d_in, d_out, views, outs, h_out = slots[s]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(ev["comp", s])          # step i-2 no longer reads d_in
                d_in.copy_(h_in, non_blocking=True)
                ev["in", s].record(up)
            comp.wait_event(ev["in", s])
            if i >= 2:
                comp.wait_event(ev["out", s])             # step i-2's results are out
            run_calls(views, outs)
            ev["comp", s].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(ev["comp", s])
                h_out.copy_(d_out, non_blocking=True)
                ev["out", s].record(down)
        comp.wait_stream(up)
        comp.wait_stream(down)
        e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def serial(n):
        d_in, d_out, views, outs, h_out = slots[0]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        for _ in range(n):
            d_in.copy_(h_in, non_blocking=True)
            run_calls(views, outs)
            h_out.copy_(d_out, non_blocking=True)
        e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    pipelined(3)                                  # warm-up, untimed
    serial(3)
    n = max(3, n_steps)
    ms = pipelined(n)
    serial_ms = serial(n)
    pos = sum(w.valid_positions for w in works)
    return {"value": n * pos / (ms / 1e3), "unit": "key-positions/s",
            "steps": n, "ms_per_step": ms / n,
            "h2d_bytes_per_step": in_total, "d2h_bytes_per_step": out_total,
            "timing": "steps issued from Python, pipelined over two device buffer sets: "
                      "each step's H2D copy of its inputs from pinned memory (copy stream), "
                      "the calls (compute stream), its D2H copy of the results to pinned "
                      "memory (second copy stream); events at the region's ends",
            "serial_value": n * pos / (serial_ms / 1e3),
            "serial_ms_per_step": serial_ms / n}


def run_e2e_store(works, device, n_steps):
    """The store through the public API with host buffers: every step copies
    its key rows and slots from pinned host memory (one copy per call) and
    reads the status word back."""
    import torch
    calls = [DeviceCall(w, device) for w in works]
    h_k = [torch.from_numpy(c.w.k_bits.view(np.int16)).pin_memory() for c in calls]
    h_s = [torch.from_numpy(c.w.slots).pin_memory() for c in calls]
    d_k = [torch.empty_like(t, device=device) for t in h_k]
    d_s = [torch.empty_like(t, device=device) for t in h_s]
    h_st = torch.zeros(len(calls), dtype=torch.int32).pin_memory()

    def step():
        for j, c in enumerate(calls):
            d_k[j].copy_(h_k[j], non_blocking=True)
            d_s[j].copy_(h_s[j], non_blocking=True)
            c.store(k=d_k[j], slots=d_s[j])
            h_st[j:j + 1].copy_(c.status, non_blocking=True)
    ms, eager_ms, steps, G = _time_e2e_steps(step, n_steps)
    rows = sum(w.valid_positions for w in works)
    return {"value": steps * rows / (ms / 1e3), "unit": "key-positions/s",
            "steps": steps, "ms_per_step": ms / steps,
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in h_k + h_s),
            "d2h_bytes_per_step": 4 * len(calls),
            "timing": f"CUDA graphs of {G} steps (each: H2D copies of the step's rows and "
                      "slots from pinned memory, the store, D2H copy of the status)",
            "eager_value": n_steps * rows / (eager_ms / 1e3),
            "eager_ms_per_step": eager_ms / n_steps}


# ---------------------------------------------------------------------------
# the fp64 oracle on the host cores

def _page_sample(works, n_pages, seed=0):
    """Up to n_pages (row, page) units of the workload, each as its own
    one-page oracle row: returns oracle argument tuples and the positions."""
    rng = np.random.default_rng(seed)
    units = []
    for wi, w in enumerate(works):
        L = np.clip(w.seqlens.astype(np.int64), 0, w.W * w.P)
        for r in range(w.R):
            for p in range(int(math.ceil(L[r] / w.P))):
                units.append((wi, r, p))
    if len(units) > n_pages:
        idx = rng.choice(len(units), n_pages, replace=False)
        units = [units[i] for i in sorted(idx)]
    return units


def _oracle_units(works, units, nthreads):
    import oracle
    pos = 0
    by_w = {}
    for wi, r, p in units:
        by_w.setdefault(wi, []).append((r, p))
    for wi, lst in by_w.items():
        w = works[wi]
        rows = np.array([r for r, _ in lst])
        pages = np.array([p for _, p in lst])
        bt_rows = w.block_table[0] if w.bt_stride == 0 else None
        bt = np.array([(bt_rows if bt_rows is not None else w.block_table[r])[p]
                       for r, p in lst], dtype=np.int32).reshape(-1, 1)
        seq = np.clip(w.seqlens[rows].astype(np.int64) - pages * w.P, 0, w.P).astype(np.int32)
        oracle.logits(w.q_bits[rows], w.w[rows], w.kcache, w.kscale_offset, w.page_stride,
                      w.num_pages, w.kv_dtype, bt, 1, seq, len(rows), w.H, w.D, w.P, 1,
                      nthreads=nthreads)
        pos += int(seq.sum())
    return pos


def _store_sample(works, budget_s):
    """The oracle's store on a bounded sample of rows (one thread)."""
    import oracle
    w = works[0]
    cal = min(w.n, 256)
    pool = w.kcache.copy()
    t0 = time.perf_counter()
    oracle.kcache_store(w.k_bits[:cal], w.slots[:cal], pool, w.page_stride, w.num_pages,
                        w.kv_dtype)
    t_row = (time.perf_counter() - t0) / cal
    n = int(min(w.n, max(cal, budget_s / max(t_row, 1e-9))))
    t0 = time.perf_counter()
    oracle.kcache_store(w.k_bits[:n], w.slots[:n], pool, w.page_stride, w.num_pages, w.kv_dtype)
    dt = time.perf_counter() - t0
    rows = int(((w.slots[:n] >= 0) & (w.slots[:n] < w.num_pages * w.P)).sum())
    return rows, dt, f"{n} of {w.n} key rows of the workload, {dt:.1f} s, C oracle, one thread"


def _logits_only_note(works):
    """The oracle computes logits; a top-k workload's selection is not part
    of the timed CPU work."""
    return "; logits only (the top-k selection is not timed)" if works[0].kind == "topk" else ""


def cpu_baseline(works, budget_s=15.0):
    """The oracle as it stands, on the host cores, on a bounded sample."""
    import oracle
    if works[0].kind == "store":
        rows, dt, sample = _store_sample(works, budget_s)
        return {"value": rows / dt, "unit": "key-positions/s", "cores": 1, "kind": "oracle",
                "sample": sample}
    cores = oracle.cpu_count()
    total_units = len(_page_sample(works, 10**12))
    # calibrate on a small sample, then size the measured sample to the budget
    cal = _page_sample(works, min(total_units, 4 * cores), seed=1)
    t0 = time.perf_counter()
    _oracle_units(works, cal, cores)
    t_unit = (time.perf_counter() - t0) / max(len(cal), 1)
    n = int(min(total_units, max(cores, budget_s / max(t_unit, 1e-9))))
    units = _page_sample(works, n, seed=2)
    t0 = time.perf_counter()
    pos = _oracle_units(works, units, cores)
    dt = time.perf_counter() - t0
    return {"value": pos / dt, "unit": "key-positions/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(units)} of {total_units} (row, page) units of the workload, "
                      f"{pos} positions, {dt:.1f} s, fp64 C oracle with {cores} threads"
                      + _logits_only_note(works)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    works = wl.NAMED[args.workload]()
    K = args.steps if args.steps is not None else DEFAULT_STEPS[args.workload]
    Wm = max(3, args.warmup if args.warmup is not None else 3)
    if works[0].kind == "store":
        w = works[0]
        per_step_budget = args.ref_budget_s / (K + Wm)
        rows, dt1, _ = _store_sample(works, per_step_budget)
        n = max(1, min(w.n, int(rows * per_step_budget / max(dt1, 1e-9))))
        pool = w.kcache.copy()
        for _ in range(Wm):
            oracle.kcache_store(w.k_bits[:n], w.slots[:n], pool, w.page_stride, w.num_pages,
                                w.kv_dtype)
        t0 = time.perf_counter()
        for _ in range(K):
            oracle.kcache_store(w.k_bits[:n], w.slots[:n], pool, w.page_stride, w.num_pages,
                                w.kv_dtype)
        dt = time.perf_counter() - t0
        stored = int(((w.slots[:n] >= 0) & (w.slots[:n] < w.num_pages * w.P)).sum())
        value = K * stored / dt
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "key-positions/s",
                "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": dt * 1e3 / K,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32 (the store's decisions)", "data": "synthetic (seeded generator; no dataset)",
                "config": {"workload": WORKLOAD_DESC[args.workload]},
                "cpu_baseline": {"value": value, "unit": "key-positions/s", "cores": 1,
                                 "kind": "oracle",
                                 "sample": f"each step: {n} of {w.n} key rows, C oracle, one thread"},
                "e2e": {"value": value, "unit": "key-positions/s",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    cores = oracle.cpu_count()
    total_units = len(_page_sample(works, 10**12))
    cal = _page_sample(works, min(total_units, 2 * cores), seed=1)
    t0 = time.perf_counter()
    _oracle_units(works, cal, cores)
    t_unit = (time.perf_counter() - t0) / max(len(cal), 1)
    per_step = int(min(total_units, max(1, args.ref_budget_s / (K + Wm) / max(t_unit, 1e-9))))
    units = _page_sample(works, per_step, seed=2)
    for _ in range(Wm):
        _oracle_units(works, units, cores)
    t0 = time.perf_counter()
    pos = 0
    for _ in range(K):
        pos += _oracle_units(works, units, cores)
    dt = time.perf_counter() - t0
    value = pos / dt
    sample = (f"each step: {len(units)} of {total_units} (row, page) units of the workload "
              f"({pos // K} positions), fp64 C oracle, {cores} threads" + _logits_only_note(works))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "key-positions/s",
            "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": dt * 1e3 / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded generator; no dataset)",
            "config": {"workload": WORKLOAD_DESC[args.workload]},
            "cpu_baseline": {"value": value, "unit": "key-positions/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "key-positions/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile(args):
    """Each call of one step, N times in a row, nothing else: the command to
    put under ncu (launch k of call j is launch k * calls + j)."""
    import torch
    from sparse_attention_paged_gb300 import _native
    _native.load()
    works = wl.NAMED[args.workload]()
    calls = [DeviceCall(w, torch.device("cuda", 0)) for w in works]
    torch.cuda.synchronize()
    for _ in range(args.profile):
        for c in calls:
            c()
    torch.cuda.synchronize()
    for c in calls:
        assert int(c.status.item()) == 0


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.profile:
        run_profile(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
