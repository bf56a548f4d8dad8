"""Replayable plans on the GPU: one CUDA graph, captured once, replayed while
the request lengths change on the device (decode and verify run under CUDA
graph replay in sglang PR #41886, "Accuracy Tests").  Every replay is checked
row by row against the FP64 oracle at that replay's lengths, and the work list
the device planner wrote must equal the host mirror's bit for bit."""
import copy
import zlib

import numpy as np
import pytest

from asymmetric_kv_paged_gb300 import binding as B
from asymmetric_kv_paged_gb300 import workloads as W
from oracle import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-3), "fp8": (6e-2, 6e-3)}

CASES = [
    # name, length bounds, n, hq, hkv, P, window, sinks, kv
    ("decode_p128", [3000, 1200, 700, 2500], [1, 1, 1, 1], 16, 2, 128, 0, False, "bf16"),
    ("verify_p16_fp8", [2000, 900], [8, 8], 16, 2, 16, 0, True, "fp8"),
    ("swa_sinks_p1", [1500, 800, 300], [1, 8, 1], 16, 2, 1, 128, True, "bf16"),
    ("prefill_gather_p3", [900], [200], 16, 2, 3, 0, False, "bf16"),
]
# 8,400 blocks: the planner's scans run over several 1024-entry chunks, and its
# 152 CTA shares each cover about 55 blocks
_MANY = np.random.default_rng(77).integers(1, 41, 4200).tolist()
CASES.append(("many_blocks", _MANY, [1] * len(_MANY), 4, 2, 16, 0, False, "bf16"))
# ~10,000 key tiles over 152 CTAs: shares of 32 tiles or more, so the device
# deal charges every block for the segment switch
_LONG = np.random.default_rng(78).integers(8000, 20000, 24).tolist()
CASES.append(("decode_charged_p128", _LONG, [1] * len(_LONG), 16, 2, 128, 0, True, "bf16"))
SHRINK = [777, 300, 65, 1, 0]     # replay at bound - d (at least n)


def _bounded_workload(name, bounds, n, hq, hkv, P, window, sinks, kv):
    # values in every slot below the bound, so that any shorter run sees no filler
    w = W.make_workload(zlib.crc32(name.encode()) % 1000, bounds, n, hq=hq, hkv=hkv,
                        page_size=P, window=0, sinks=sinks, kv_dtype=kv, name=name)
    w.window = window
    return w


def _at(w, lens):
    w2 = copy.copy(w)
    w2.seq_lens = np.asarray(lens, np.int32)
    return w2


def _check(w, dw, lens):
    ref, ref_lse = oracle.attn_paged(_at(w, lens).host_arrays())
    got = dw.out.float().cpu().numpy().astype(np.float64)
    mx, mean = TOL[w.kv_dtype]
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert err.max() <= mx and err.mean() <= mean, (lens, err.max(), err.mean())
    lerr = np.abs(dw.lse.cpu().numpy() - ref_lse)
    assert lerr.max() <= (2e-3 if w.kv_dtype == "bf16" else 1e-2) * max(1.0, np.abs(ref_lse).max())


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_graph_replay_with_changing_lengths(case):
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    name, bounds, n = case[0], case[1], case[2]
    w = _bounded_workload(*case)
    dw = DeviceWorkload(w, replayable=True)
    num_sms = torch.cuda.get_device_properties(0).multi_processor_count
    prob, keep = B.make_problem(
        batch=w.batch, num_q_heads=w.hq, num_kv_heads=w.hkv, page_size=w.page_size,
        num_pages=w.num_pages, page_table_stride=w.page_table.shape[1],
        kv_dtype=B.ATTN_KV_BF16 if w.kv_dtype == "bf16" else B.ATTN_KV_FP8_E4M3,
        window=w.window, has_sinks=w.sinks is not None, qo_indptr=w.qo_indptr,
        seq_lens=w.seq_lens)
    mirror = B.attn_plan_replayable_host(prob, num_sms, keep)
    dw.run()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dw.run(stream=s)
    torch.cuda.synchronize()
    bnd = np.asarray(bounds)
    for d in SHRINK:
        lens = np.maximum(bnd - d, np.asarray(n)).astype(np.int32)
        dw.seq_lens.copy_(torch.from_numpy(lens))
        dw.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        _check(w, dw, lens)
        assert B.attn_get_device_error(dw.plan) == 0
        B.attn_plan_fetch_device(dw.plan)
        assert B.attn_plan_replan_host(mirror, lens) == 0
        assert np.array_equal(B.attn_plan_blocks(dw.plan), B.attn_plan_blocks(mirror))
        assert np.array_equal(B.attn_plan_segments(dw.plan), B.attn_plan_segments(mirror))
        assert np.array_equal(B.attn_plan_cta_heads(dw.plan), B.attn_plan_cta_heads(mirror))
        if name == "decode_charged_p128":
            # the switch charge is in force: CTAs that reach into more blocks hold fewer tiles
            segs = B.attn_plan_segments(dw.plan)
            loads = np.bincount(segs[:, 0], weights=segs[:, 3] - segs[:, 2])
            assert loads.max() - loads.min() > 1


def test_lengths_outside_bounds_are_clamped_and_flagged():
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    w = _bounded_workload("clamp", [1000, 400], [8, 1], 16, 2, 16, 0, True, "bf16")
    dw = DeviceWorkload(w, replayable=True)
    lens = np.array([5000, 0], np.int32)           # above the bound, below n
    dw.seq_lens.copy_(torch.from_numpy(lens))
    dw.run()
    torch.cuda.synchronize()
    assert B.attn_get_device_error(dw.plan) == 4
    _check(w, dw, np.array([1000, 1], np.int32))
