"""Device-side convenience around the C ABI: upload a host workload, plan it and run it.

Used by the tests and the benchmark; a serving integration would call the binding
directly with its own cache tensors.  No compute happens here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B


def _dev(a: np.ndarray, device, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device, non_blocking=False)


class DeviceWorkload:
    """A workload resident in device memory with its plan, output and workspace."""

    def __init__(self, w, device: int = 0, with_lse: bool = True, replayable: bool = False):
        self.w = w
        self.device = device
        self.replayable = replayable    # w.seq_lens are then upper bounds
        dev = torch.device("cuda", device)
        self.q = _dev(w.q, dev, torch.bfloat16)
        kv_t = torch.bfloat16 if w.kv_dtype == "bf16" else torch.uint8
        self.k_cache = _dev(w.k_cache, dev, kv_t)
        self.v_cache = _dev(w.v_cache, dev, kv_t)
        self.page_table = _dev(w.page_table, dev)
        self.seq_lens = _dev(w.seq_lens, dev)
        self.qo_indptr = _dev(w.qo_indptr, dev)
        self.sinks = None if w.sinks is None else _dev(w.sinks.astype(np.float32), dev)
        self.out = torch.empty((w.total_q, w.hq, 128), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.total_q, w.hq), dtype=torch.float32, device=dev) if with_lse else None
        self.plan = self.make_plan()
        nbytes = max(self.plan.workspace_bytes, 1)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def problem(self):
        w = self.w
        return B.make_problem(
            batch=w.batch, num_q_heads=w.hq, num_kv_heads=w.hkv, page_size=w.page_size,
            num_pages=w.num_pages, page_table_stride=w.page_table.shape[1],
            kv_dtype=B.ATTN_KV_BF16 if w.kv_dtype == "bf16" else B.ATTN_KV_FP8_E4M3,
            window=w.window, has_sinks=w.sinks is not None, qo_indptr=w.qo_indptr,
            seq_lens=w.seq_lens, head_dim_qk=w.dqk)

    def make_plan(self):
        prob, keep = self.problem()
        if self.replayable:
            return B.attn_plan_replayable(prob, self.device, keep)
        return B.attn_plan(prob, self.device, keep)

    def run_phase(self, phase: int, stream=None) -> None:
        w = self.w
        B.attn_run_phase(self.plan, phase, self.q, self.k_cache, self.v_cache, self.page_table,
                         self.seq_lens, self.qo_indptr, self.sinks, w.window, w.softmax_scale,
                         w.k_scale, w.v_scale, self.out, self.lse, self.workspace, stream)

    def run(self, stream=None, out=None, lse=None, plan=None) -> None:
        w = self.w
        B.attn_run_paged(plan or self.plan, self.q, self.k_cache, self.v_cache, self.page_table,
                         self.seq_lens, self.qo_indptr, self.sinks, w.window, w.softmax_scale,
                         w.k_scale, w.v_scale, self.out if out is None else out,
                         self.lse if lse is None else lse, self.workspace, stream)
