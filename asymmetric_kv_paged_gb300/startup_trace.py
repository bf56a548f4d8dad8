"""Where a split-KV launch spends its time: per-CTA timestamps from the profiling
build of the library (``build.build(stamps=True)``; the kernel writes the GPU's
global timer at the points listed in include/attn_paged_debug.h,
attn_debug_stamps).

    python -m asymmetric_kv_paged_gb300.startup_trace c1_tiny_decode c4_swa_sinks

Per-SM stream rate: for CTAs with one segment, the time from the first S tile to
the last P.V divided by their key tiles (``tile_us``: minimum, median, maximum
over CTAs of its mean over the runs), whether each CTA ran on the same SM in
every run (``same_sm``: fraction of CTAs), and the correlation of each CTA's
rate between the first and second half of the runs (``rate_repeat``; near 1
when some SMs are persistently slower than others).

For each named workload the attention kernel alone (no merge) is launched
``--runs`` times after three warm-up steps, each time after L2 has been flushed
(a 256 MB buffer written and read back, as bench.py does between steps) and,
with ``--hot``, also without the flush.  Every event is reported in
microseconds after the earliest CTA's first instruction, as the median over the
runs of its minimum, median and maximum over the CTAs; ``event_us`` is the
launch's duration between CUDA events on its stream (launch latency included).
The profiling build's register allocation differs from the default build's, so
its times describe the structure of a launch, not the default build's speed.
Needs a GPU.
"""
from __future__ import annotations

import argparse
import json

import numpy as np

# (name, column of the stamp array), in the order a CTA usually reaches them
EVENTS = (("start", 0), ("head", 1), ("ready", 2), ("lookup", 13), ("first_load", 3),
          ("first_q", 4), ("first_qk", 5), ("first_s", 6), ("last_pv", 7), ("epi_begin", 8),
          ("epi_end", 9), ("end", 10))
SEGS, TILES, SM = 11, 12, 14


def _stats(stamps: np.ndarray, ctas: int) -> dict:
    rows = stamps[:min(ctas, stamps.shape[0])].astype(np.int64)
    live = rows[rows[:, 0] > 0]
    base = live[:, 0].min()
    out = {}
    for name, i in EVENTS:
        col = live[:, i]
        col = col[col > 0]
        if col.size:
            r = (col - base) / 1e3
            out[name] = (float(r.min()), float(np.median(r)), float(r.max()))
    epi = live[:, 9] - live[:, 8]
    epi = epi[(live[:, 8] > 0) & (live[:, 9] > 0)] / 1e3
    if epi.size:
        out["epi_len"] = (float(epi.min()), float(np.median(epi)), float(epi.max()))
    out["segs"] = (int(live[:, SEGS].min()), float(np.median(live[:, SEGS])), int(live[:, SEGS].max()))
    out["tiles"] = (int(live[:, TILES].min()), float(np.median(live[:, TILES])),
                    int(live[:, TILES].max()))
    out["ctas"] = int(live.shape[0])
    return out


def trace(name: str, runs: int, flush: bool) -> dict:
    import torch

    from . import binding as B
    from . import workloads
    from .runner import DeviceWorkload

    w = workloads.named(name)
    dw = DeviceWorkload(w, device=torch.cuda.current_device())
    ctas = int(B.attn_plan_info(dw.plan)["ctas"])
    st = torch.cuda.current_stream()
    buf = torch.empty(256 << 20, dtype=torch.uint8, device=dw.q.device)
    for _ in range(3):
        dw.run_phase(0, st)
        dw.run_phase(1, st)
    torch.cuda.synchronize()
    B.attn_debug_stamps(clear=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per_run, times, raw = [], [], []
    for _ in range(runs):
        if flush:
            buf.fill_(1)
            buf.view(torch.int32).max()
        else:
            # keep the GPU busy while the launch is queued, as the flush does,
            # so that the events time the kernel and not the host's submission
            torch.cuda._sleep(100_000)
        e0.record(st)
        dw.run_phase(0, st)
        e1.record(st)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
        stamps = B.attn_debug_stamps(clear=True)
        per_run.append(_stats(stamps, ctas))
        raw.append(stamps[:min(ctas, stamps.shape[0])].astype(np.int64))
        dw.run_phase(1, st)
    torch.cuda.synchronize()
    assert B.attn_get_device_error(dw.plan) == 0
    out = {"workload": name, "l2": "flushed" if flush else "warm", "runs": runs,
           "event_us": round(float(np.median(times)), 2), "ctas": per_run[0]["ctas"],
           "segs": per_run[0]["segs"], "tiles": per_run[0]["tiles"]}
    for key in [name for name, _ in EVENTS] + ["epi_len"]:
        vals = [r[key] for r in per_run if key in r]
        if vals:
            out[key] = [round(float(np.median([v[j] for v in vals])), 2) for j in range(3)]
    out.update(_sm_rates(np.stack(raw)))
    return out


def _sm_rates(raw: np.ndarray) -> dict:
    """Stream rate of the one-segment CTAs and how it repeats across runs
    (raw: runs x CTAs x events)."""
    one = (raw[0, :, SEGS] == 1) & (raw[0, :, TILES] > 0) & np.all(raw[:, :, 0] > 0, axis=0)
    if one.sum() < 2 or raw.shape[0] < 2:
        return {}
    x = raw[:, one]
    rate = (x[:, :, 7] - x[:, :, 6]) / 1e3 / x[:, :, TILES]     # runs x CTAs, us per tile
    mean = rate.mean(axis=0)
    h = rate.shape[0] // 2
    rep = np.corrcoef(rate[:h].mean(axis=0), rate[h:].mean(axis=0))[0, 1]
    same = float(np.mean([np.unique(x[:, c, SM]).size == 1 for c in range(x.shape[1])]))
    return {"tile_us": [round(float(mean.min()), 3), round(float(np.median(mean)), 3),
                        round(float(mean.max()), 3)],
            "one_segment_ctas": int(one.sum()), "same_sm": round(same, 2),
            "rate_repeat": round(float(rep), 2)}


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("workloads", nargs="+")
    ap.add_argument("--runs", type=int, default=10)
    ap.add_argument("--hot", action="store_true", help="also trace without the L2 flush")
    args = ap.parse_args()
    from . import binding as B
    B.use_stamps_build()
    B.load()
    for name in args.workloads:
        for flush in ((True, False) if args.hot else (True,)):
            print(json.dumps(trace(name, args.runs, flush)), flush=True)


if __name__ == "__main__":
    main()
