#!/usr/bin/env python
"""Benchmark of paged asymmetric-KV attention (QK 192 / V 128) on one or more GPUs.

Headline workload: batched paged decode (32 requests x 1 token, 16 q / 2 KV heads,
context U[1024, 32768] not page aligned, page 128, bf16 K/V in a shuffled 1.2M-slot
pool).  A step is one attn_run_paged call (split-KV kernel + log-sum-exp merge)
over that batch; inputs are resident in HBM.  The KV stream (~0.7 GB) is far larger
than L2 (129 MB), so no L2 flush is needed between steps.

  value      algorithmic bytes per step x ranks / time per step (GB/s)
  roofline   the split-KV kernel alone: algorithmic bytes / its own CUDA-event time
  e2e        through the C ABI from pinned host buffers: q and the batch metadata
             copied in, attn_run_paged, the output copied back, every step
  extra      the other named workloads (tiny decode, verify at page 128 and 1,
             SWA with sinks, fp8 chunked prefill) with their own roofline fraction
  cpu_baseline  the FP64 oracle on a bounded sample of the headline workload

Under torchrun every rank runs its own replica of the workload (independent
requests: no collective on the data path) and the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode/verify KV-read GB/s & % HBM roofline; prefill TFLOP/s & % tensor peak"
HEADLINE = "c2_batched_decode"
DQK, DV = 192, 128


# ---------------------------------------------------------------- accounting

def algorithmic_bytes(w) -> int:
    """Every visible key of every (request, KV head) once (K and V rows), Q in,
    bf16 out, touched page-table entries and the sinks; split partials and
    masked slots excluded."""
    es = 2 if w.kv_dtype == "bf16" else 1
    keys = 0
    pages = 0
    for b in range(w.batch):
        lo, hi = w.visible_range(b)
        if hi > lo:
            keys += hi - lo
            pages += (hi - 1) // w.page_size - lo // w.page_size + 1
    total = keys * w.hkv * (w.dqk + DV) * es
    total += w.total_q * w.hq * (w.dqk + DV) * 2
    total += pages * 4
    if w.sinks is not None:
        total += w.hq * 4
    return int(total)


def algorithmic_flops(w) -> int:
    """2 * (Dqk + 128) FLOPs per visible (query row, key) pair (Dqk = 192)."""
    pairs = 0
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        n = int(w.qo_indptr[b + 1] - w.qo_indptr[b])
        i = L - n + np.arange(n, dtype=np.int64)
        lo = np.maximum(0, i - w.window + 1) if w.window > 0 else np.zeros_like(i)
        pairs += int((i + 1 - lo).sum())
    return 2 * (w.dqk + DV) * pairs * w.hq


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def kernel_of(workload: str) -> str:
    """The attention kernel a named workload's plan launches: the prefill kernel
    for blocks of more than 128 query rows, the split-KV kernel otherwise."""
    return "attn_prefill" if workload.startswith("c5") else "attn_tc"


def split_kernel_traffic(workload: str):
    """DRAM bytes per launch of the workload's attention kernel from a committed ncu
    summary, when that summary was taken on the kernel source as it is now (else
    None)."""
    kern = kernel_of(workload)
    path = os.path.join(ROOT, "profiles", f"{kern}_{workload}.md")
    src = os.path.join(ROOT, "asymmetric_kv_paged_gb300", "csrc", f"{kern}.cu")
    if not os.path.exists(path):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    fields = {}
    for line in open(path):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256_16") != digest:
        return None
    try:
        return int(float(fields["dram_bytes_per_launch_full_size"]))
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        """Median SM clock and the throttle reasons seen inside [t0, t1].  When no
        sample falls inside (a timed region shorter than the sampling period) the
        in-region fields are null and `outside` summarises the samples taken while
        this process ran the same workload around it."""
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        rec = self._stats(inside)
        rec["samples_in_timed_region"] = len(inside)
        rec["timed_region_ms"] = (t1 - t0) * 1e3
        if not inside:
            rec["outside"] = self._stats([p for _, p in self.samples])
        return rec

    @staticmethod
    def _stats(use):
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": None, "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[0]) for p in use if num(p[0]) is not None]
        mx = [num(p[1]) for p in use if num(p[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for p in use for n, v in zip(names, p[4:8]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(use)}


# ---------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- our arm

def evict_l2(buf, k: int) -> None:
    """Evicts the workload from L2 between timed steps: the 256 MB buffer is
    written (twice L2's 129 MB), then read back, so that L2 holds clean lines
    of the buffer only and none of its dirty lines is written back to DRAM
    inside the next step's timed kernels."""
    import torch
    buf.fill_(k & 0xFF)
    buf.view(torch.int32).max()


def time_workload(dw, steps: int, warmup: int, world: int, flush_l2: bool = False,
                  sampler=None):
    """Returns dict with step ms, split/merge kernel ms (CUDA events on the launch
    stream) and the wall-clock bounds of the timed region."""
    import torch
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda") if flush_l2 else None
    for _ in range(warmup):
        dw.run_phase(0, stream)
        dw.run_phase(1, stream)
    from asymmetric_kv_paged_gb300 import binding
    # kernels per step: the attention kernel, the merge kernel when the plan
    # leaves blocks to it, the staging pass of a prefill plan, the device
    # planner of a replayable plan
    per_step = (1 + (binding.attn_plan_merge_ctas(dw.plan) > 0)
                + (len(binding.attn_plan_stage_units(dw.plan)) > 0)
                + bool(getattr(dw, "replayable", False)))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(steps):
        if flush is not None:
            evict_l2(flush, k)
        ev[k][0].record(stream)
        dw.run_phase(0, stream)
        ev[k][1].record(stream)
        dw.run_phase(1, stream)
        ev[k][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    split = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    merge = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    attn = float(np.mean([e[0].elapsed_time(e[2]) for e in ev]))
    # The step itself is timed in a second pass without events between the
    # two kernels: the merge is a programmatic dependent launch and overlaps
    # the attention kernel's tail, which an event in between would prevent.
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for k in range(steps):
        if flush is not None:
            evict_l2(flush, k)
        ev2[k][0].record(stream)
        dw.run_phase(0, stream)
        dw.run_phase(1, stream)
        ev2[k][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    step = float(np.mean([e[0].elapsed_time(e[1]) for e in ev2]))
    total = start.elapsed_time(end) / steps
    return dict(step_ms=(step if flush_l2 else total), split_ms=split, merge_ms=merge,
                attn_ms=step, t0=t0, t1=t1, launches=steps * per_step)


def grown_workload(w, extra: int):
    """A copy of decode workload `w` whose requests can grow by `extra` tokens: the
    page table gains fresh pages from the pool's unused ones, and seq_lens become
    the upper bounds of a replayable plan."""
    import copy
    P = w.page_size
    L = w.seq_lens.astype(np.int64)
    have = (L + P - 1) // P
    need = (L + extra + P - 1) // P
    used = set(int(x) for x in np.unique(w.page_table))
    free = [p for p in range(w.num_pages) if p not in used]
    assert len(free) > int((need - have).sum()), "pool too small to grow the batch"
    # columns past a request's pages point at an unused (NaN) page, as in the workload
    pt = np.full((w.batch, int(need.max())), free.pop(), np.int32)
    pt[:, :w.page_table.shape[1]] = w.page_table
    it = iter(free)
    for b in range(w.batch):
        for j in range(int(have[b]), int(need[b])):
            pt[b, j] = next(it)
    g = copy.copy(w)
    g.page_table = pt
    g.seq_lens = (L + extra).astype(np.int32)
    return g


def e2e_measure(w, steps: int, warmup: int, world: int):
    """One decode serving step per timed step, through the C ABI from pinned host
    memory: every request grows by one token per step.  Per step: q, the new
    token's K/V rows, the lengths, qo_indptr and the page table are copied in,
    attn_append_kv writes the new K/V into the paged cache, attn_run_paged runs on
    a replayable plan (lengths read on the device: planner kernel, attention,
    merge), and the output is copied back; the copies of one step overlap the
    computation of its neighbours (double-buffered, streams of their own).  The
    K/V cache is state and stays resident.  Also reported: the same copies around a static plan whose lengths
    never change (`static`), and the host cost of attn_plan for this batch."""
    import torch
    from asymmetric_kv_paged_gb300 import binding as B
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    total = warmup + steps
    g = grown_workload(w, total)
    dw = DeviceWorkload(g, device=torch.cuda.current_device(), with_lse=False, replayable=True)
    stream = torch.cuda.current_stream()
    L0 = w.seq_lens.astype(np.int64)
    rng = np.random.default_rng(7)
    h_q = torch.from_numpy(w.q).view(torch.bfloat16).pin_memory()
    h_kn = torch.from_numpy(rng.standard_normal((w.total_q, w.hkv, w.dqk), dtype=np.float32)).to(
        torch.bfloat16).pin_memory()
    h_vn = torch.from_numpy(rng.standard_normal((w.total_q, w.hkv, DV), dtype=np.float32)).to(
        torch.bfloat16).pin_memory()
    h_pt = torch.from_numpy(g.page_table).pin_memory()
    h_qo = torch.from_numpy(w.qo_indptr).pin_memory()
    h_sl = torch.from_numpy(np.stack([(L0 + s).astype(np.int32) for s in range(total)])).pin_memory()
    h_out = torch.empty(dw.out.shape, dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_kn, h_vn, h_pt, h_qo)) + h_sl[0].numel() * 4
    d2h = h_out.numel() * h_out.element_size()
    ks, vs = (w.k_scale, w.v_scale) if w.kv_dtype == "fp8" else (1.0, 1.0)

    # The step's inputs other than the lengths (q, the new K and V rows,
    # qo_indptr, the page table) sit packed in one pinned buffer and cross in
    # one copy, the lengths in a second.  Device inputs and outputs are
    # double-buffered and the copies run on streams of their own, so that step
    # s+1's inputs and step s's output move while step s computes.
    consts = (h_q, h_kn, h_vn, h_qo, h_pt)
    offs, nbytes = [], 0
    for t in consts:
        offs.append(nbytes)
        nbytes += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    for t, o in zip(consts, offs):
        h_in[o:o + t.numel() * t.element_size()].copy_(t.reshape(-1).view(torch.uint8))
    d_in = [torch.empty(nbytes, dtype=torch.uint8, device=dw.q.device) for _ in range(2)]
    d_views = [[buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for t, o in zip(consts, offs)] for buf in d_in]
    d_sl = [torch.empty_like(h_sl[0], device=dw.q.device) for _ in range(2)]
    d_out = [torch.empty_like(dw.out) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def step(s):
        b = s % 2
        q, kn, vn, qo, pt = d_views[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_done[b])          # step s-2 has finished with these inputs
            d_in[b].copy_(h_in, non_blocking=True)
            d_sl[b].copy_(h_sl[s], non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if used[b]:
            stream.wait_event(ev_out[b])             # step s-2's output has been read back
        B.attn_append_kv(dw.plan, kn, vn, dw.k_cache, dw.v_cache, pt, d_sl[b], qo, ks, vs, stream)
        B.attn_run_paged(dw.plan, q, dw.k_cache, dw.v_cache, pt, d_sl[b], qo, dw.sinks, g.window,
                         g.softmax_scale, ks, vs, d_out[b], None, dw.workspace, stream)
        ev_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            h_out.copy_(d_out[b], non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for s in range(warmup):
        step(s)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for s in range(warmup, total):
        step(s)
    stream.wait_event(ev_out[(total - 1) % 2])      # the last output is on the host
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    assert B.attn_get_device_error(dw.plan) == 0
    grown_bytes = [algorithmic_bytes(_with_lens(w, L0 + s)) for s in range(warmup, total)]
    ms = start.elapsed_time(end) / steps
    del dw
    torch.cuda.empty_cache()

    # the static-plan figure: same batch, lengths fixed, no append
    sw = DeviceWorkload(w, device=torch.cuda.current_device(), with_lse=False)
    h_pt0 = torch.from_numpy(w.page_table).pin_memory()
    h_sl0 = torch.from_numpy(w.seq_lens).pin_memory()

    def static_step():
        sw.q.copy_(h_q, non_blocking=True)
        sw.page_table.copy_(h_pt0, non_blocking=True)
        sw.seq_lens.copy_(h_sl0, non_blocking=True)
        sw.qo_indptr.copy_(h_qo, non_blocking=True)
        sw.run(stream)
        h_out.copy_(sw.out, non_blocking=True)

    for _ in range(warmup):
        static_step()
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        static_step()
    end.record(stream)
    torch.cuda.synchronize()
    static_ms = start.elapsed_time(end) / steps
    t = time.time()
    for _ in range(3):
        sw.make_plan().destroy()
    plan_ms = (time.time() - t) / 3 * 1e3
    del sw
    torch.cuda.empty_cache()
    return dict(ms=ms, h2d=h2d, d2h=d2h, bytes=float(np.mean(grown_bytes)), static_ms=static_ms,
                static_h2d=sum(t.numel() * t.element_size() for t in (h_q, h_pt0, h_sl0, h_qo)),
                plan_ms=plan_ms)


def _with_lens(w, lens):
    import copy
    g = copy.copy(w)
    g.seq_lens = np.asarray(lens, dtype=np.int32)
    return g


def cpu_baseline(w, budget_s: float = 12.0):
    """The FP64 oracle, as it stands, on whole requests of the workload until about
    budget_s of wall time has been spent."""
    from oracle import oracle
    pb = w.host_arrays()
    done_bytes = 0
    done_req = 0
    t_total = 0.0
    for b in range(w.batch):
        toks = np.arange(w.qo_indptr[b], w.qo_indptr[b + 1], dtype=np.int64)
        rows = (toks[:, None] * w.hq + np.arange(w.hq)[None, :]).reshape(-1)
        t = time.time()
        oracle.attn_paged(pb, rows=rows)
        t_total += time.time() - t
        lo, hi = w.visible_range(b)
        done_bytes += (hi - lo) * w.hkv * (w.dqk + DV) * (2 if w.kv_dtype == "bf16" else 1)
        done_bytes += len(toks) * w.hq * (w.dqk + DV) * 2
        done_req += 1
        if t_total >= budget_s:
            break
    return {"value": done_bytes / t_total / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{done_req} of {w.batch} requests of {w.name} (all their rows), "
                      f"{t_total:.1f} s FP64 on host cores"}


def measure_append(name: str, pk: dict, steps: int, warmup: int):
    """attn_append_kv on the new tokens of a named workload: their K/V rows read
    (bf16) and written into the pages (bf16 or E4M3) once, plus the page-table
    entries, lengths and offsets read; L2 flushed between steps."""
    import torch
    from asymmetric_kv_paged_gb300 import binding, workloads
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    w = workloads.named(name)
    dw = DeviceWorkload(w, device=torch.cuda.current_device(), with_lse=False)
    rng = np.random.default_rng(99)
    dev = torch.device("cuda", torch.cuda.current_device())
    kn = torch.from_numpy(rng.standard_normal((w.total_q, w.hkv, w.dqk), dtype=np.float32)).to(
        dev).to(torch.bfloat16)
    vn = torch.from_numpy(rng.standard_normal((w.total_q, w.hkv, DV), dtype=np.float32)).to(
        dev).to(torch.bfloat16)
    es = 2 if w.kv_dtype == "bf16" else 1
    nbytes = (w.total_q * w.hkv * (w.dqk + DV) * (2 + es) + w.total_q * 4 * 3
              + (w.batch + 1) * 4 + w.batch * 4)
    ks, vs = (w.k_scale, w.v_scale) if w.kv_dtype == "fp8" else (1.0, 1.0)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step():
        binding.attn_append_kv(dw.plan, kn, vn, dw.k_cache, dw.v_cache, dw.page_table,
                               dw.seq_lens, dw.qo_indptr, ks, vs, stream)

    for _ in range(warmup):
        step()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        evict_l2(flush, k)
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    assert binding.attn_get_device_error(dw.plan) == 0
    achieved = nbytes / (ms * 1e-3) / 1e9
    out = {"workload": f"kv_append_{name}", "value": achieved, "unit": "GB/s", "ms_per_step": ms,
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                        "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": None},
           "algorithmic_bytes": nbytes, "tokens": w.total_q, "kv_dtype": w.kv_dtype,
           "l2": "flushed between steps (256 MB written, then read)"}
    del dw
    torch.cuda.empty_cache()
    return out


def measure_extra(name: str, pk: dict, steps: int, warmup: int, world: int):
    import torch
    from asymmetric_kv_paged_gb300 import workloads
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    w = workloads.named(name)
    dw = DeviceWorkload(w, device=torch.cuda.current_device())
    nbytes = algorithmic_bytes(w)
    flops = algorithmic_flops(w)
    small = nbytes < 256e6          # fits in L2 across steps: flush between steps
    r = time_workload(dw, steps, warmup, world, flush_l2=small)
    if name.startswith("c5"):
        achieved = flops / (r["split_ms"] * 1e-3) / 1e12
        peak = pk["bf16_tflops"]
        out = {"workload": name, "value": flops / (r["attn_ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": r["attn_ms"], "roofline": {"bound": "tensor", "achieved": achieved,
                                                           "peak": peak, "unit": "TFLOP/s",
                                                           "frac": achieved / peak,
                                                           "traffic": split_kernel_traffic(name),
                                                           "kernel": kernel_of(name) + "_kernel"}}
    else:
        achieved = nbytes / (r["split_ms"] * 1e-3) / 1e9
        peak = pk["hbm_gbs"]
        out = {"workload": name, "value": nbytes / (r["attn_ms"] * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": r["attn_ms"], "roofline": {"bound": "hbm", "achieved": achieved,
                                                           "peak": peak, "unit": "GB/s",
                                                           "frac": achieved / peak,
                                                           "traffic": split_kernel_traffic(name),
                                                           "kernel": kernel_of(name) + "_kernel"}}
    out.update(split_ms=r["split_ms"], merge_ms=r["merge_ms"], algorithmic_bytes=nbytes,
               flops=flops,
               l2="flushed between steps (256 MB written, then read)" if small
               else "inputs larger than L2")
    del dw
    torch.cuda.empty_cache()
    return out


def measure_replayable(name: str, steps: int, warmup: int):
    """The workload through a replayable plan (lengths read on the device at every
    run, bounds = the workload's lengths), replayed from one CUDA graph: the device
    planner, the attention kernel and the merge per step."""
    import torch
    from asymmetric_kv_paged_gb300 import binding, workloads
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    w = workloads.named(name)
    dw = DeviceWorkload(w, device=torch.cuda.current_device(), replayable=True)
    nbytes = algorithmic_bytes(w)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    dw.run(stream=side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        dw.run(stream=side)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        g.replay()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        ev[k][0].record(stream)
        g.replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    assert binding.attn_get_device_error(dw.plan) == 0
    out = {"workload": name, "plan": "replayable, one CUDA graph", "value": nbytes / (ms * 1e-3) / 1e9,
           "unit": "GB/s", "ms_per_step": ms, "launches_per_step": 3,
           "l2": "inputs larger than L2" if nbytes >= 256e6 else "not flushed"}
    del dw, g
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from asymmetric_kv_paged_gb300 import binding, workloads
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    binding.load()
    pk = peaks()
    w = workloads.named(args.workload)
    dw = DeviceWorkload(w, device=torch.cuda.current_device())
    nbytes = algorithmic_bytes(w)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    # a workload smaller than L2 (a non-default --workload) is flushed between steps
    small = nbytes < 256e6
    r = time_workload(dw, args.steps, args.warmup, world, flush_l2=small)
    clocks = sampler.summary(r["t0"], r["t1"]) if sampler else None
    if sampler:
        sampler.stop()
    step_ms = max_over_ranks(r["step_ms"], world)
    split_ms = max_over_ranks(r["split_ms"], world)
    assert binding.attn_get_device_error(dw.plan) == 0
    del dw
    torch.cuda.empty_cache()
    e2e = None if args.no_e2e else e2e_measure(w, max(10, args.steps // 4), 3, world)
    e2e_ms = max_over_ranks(e2e["ms"], world) if e2e else None
    static_ms = max_over_ranks(e2e["static_ms"], world) if e2e else None
    achieved = nbytes / (split_ms * 1e-3) / 1e9
    tensor = kernel_of(args.workload) == "attn_prefill"
    if tensor:                 # the prefill chunk is compute-bound: FLOPs, tensor peak
        flops = algorithmic_flops(w)
        achieved = flops / (split_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": (flops * world / (step_ms * 1e-3) / 1e12 if tensor
                                    else nbytes * world / (step_ms * 1e-3) / 1e9),
        "unit": "TFLOP/s" if tensor else "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64; bf16 N(0,1) values, K scaled 0.5)",
        "config": workload_config(w, nbytes, world, flushed=small),
        "roofline": {"bound": "tensor" if tensor else "hbm", "achieved": achieved,
                     "peak": pk["bf16_tflops"] if tensor else pk["hbm_gbs"],
                     "unit": "TFLOP/s" if tensor else "GB/s",
                     "frac": achieved / (pk["bf16_tflops"] if tensor else pk["hbm_gbs"]),
                     "traffic": split_kernel_traffic(args.workload),
                     "kernel": kernel_of(args.workload) + "_kernel", "kernel_ms": split_ms,
                     "merge_ms": r["merge_ms"],
                     "peak_source": f"{pk['source']} ({'bf16_tflops' if tensor else 'hbm_gbs'})"},
        "e2e": None if e2e is None else {
                "value": e2e["bytes"] * world / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": e2e_ms,
                "step": "serving decode step: every length +1 per step; inputs in two "
                        "copies (packed, lengths), KV append + replayable-plan attention "
                        "(planner kernel, attention, merge), output read back; copies "
                        "double-buffered on their own streams",
                "static": {"value": nbytes * world / (static_ms * 1e-3) / 1e9, "unit": "GB/s",
                           "ms_per_step": static_ms, "h2d_bytes_per_step": e2e["static_h2d"],
                           "d2h_bytes_per_step": e2e["d2h"],
                           "step": "static plan, lengths fixed, no append"},
                "plan_ms_per_batch_shape": e2e["plan_ms"]},
        "gpu_launches": r["launches"],
        "clocks": clocks,
    }
    if rank == 0 and not args.no_extra:
        extra = []
        for name in workloads.CONFIG_NAMES + workloads.EXTRA_NAMES:
            if name == args.workload:
                continue
            extra.append(measure_extra(name, pk, max(20, args.steps // 4), args.warmup, 1))
        # the KV-append step before attention: the headline decode's 32 tokens and
        # the prefill chunk's 4096 (E4M3)
        for name in ("c2_batched_decode", "c5_chunked_prefill"):
            extra.append(measure_append(name, pk, max(20, args.steps // 4), args.warmup))
        # the headline workload again, planned on the device at every run
        extra.append(measure_replayable(args.workload, max(20, args.steps // 4), args.warmup))
        line["extra"] = extra
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm

def workload_config(w, nbytes: int, world: int, flushed: bool = False) -> dict:
    """The `config` object of the JSON line; both arms report the same one."""
    return {"workload": w.name, "batch": w.batch,
            "q_tokens_per_request": int(w.qo_indptr[1] - w.qo_indptr[0]) if w.batch else 0,
            "num_q_heads": w.hq, "num_kv_heads": w.hkv, "head_dim_qk": w.dqk, "head_dim_v": DV,
            "page_size": w.page_size, "pool_slots": w.num_pages * w.page_size,
            "kv_tokens": int(w.seq_lens.sum()), "kv_dtype": w.kv_dtype,
            "algorithmic_bytes_per_step": nbytes,
            "l2": ("flushed between steps (256 MB written, then read)" if flushed else
                   "inputs larger than L2 (KV stream per step >> 129 MB); no flush"),
            "parallelism": f"replicas x{world} (independent requests, no collective)"}


def run_reference(args):
    """The FP64 oracle as it stands, on the host cores: each step computes a bounded
    sample (whole requests) of the headline workload."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    from asymmetric_kv_paged_gb300 import workloads
    from oracle import oracle
    w = workloads.named(args.workload)
    pb = w.host_arrays()
    reqs = list(range(min(2, w.batch)))          # ~1 s of FP64 work per step
    rows = np.concatenate([
        (np.arange(w.qo_indptr[b], w.qo_indptr[b + 1])[:, None] * w.hq
         + np.arange(w.hq)[None, :]).reshape(-1) for b in reqs])
    es = 2 if w.kv_dtype == "bf16" else 1
    nbytes = sum((w.visible_range(b)[1] - w.visible_range(b)[0]) * w.hkv * (w.dqk + DV) * es
                 + int(w.qo_indptr[b + 1] - w.qo_indptr[b]) * w.hq * (w.dqk + DV) * 2 for b in reqs)
    for _ in range(args.warmup):
        oracle.attn_paged(pb, rows=rows)
    t = time.time()
    for _ in range(args.steps):
        oracle.attn_paged(pb, rows=rows)
    dt = (time.time() - t) / args.steps
    value = nbytes / dt / 1e9
    sample = f"requests {reqs} of {w.name} ({len(rows)} rows) per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64)",
            "config": workload_config(w, algorithmic_bytes(w), world),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end serving measurement")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
