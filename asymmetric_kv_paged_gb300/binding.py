"""Thin ctypes binding of libattn_paged.so (include/attn_paged.h).

Argument marshalling only: every step of the attention runs in the library's CUDA
kernels.  Functions keep the C names.  Tensors are torch tensors (device memory and
streams come from PyTorch); the binding passes their raw pointers.  If the library
cannot be loaded the import fails loudly: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_WORKSPACE = -3
ATTN_ERR_CUDA = -4
ATTN_KV_BF16 = 0
ATTN_KV_FP8_E4M3 = 1

EXPORTED = ("attn_plan", "attn_run_paged", "attn_run_phase", "attn_plan_destroy", "attn_get_device_error",
            "attn_status_string", "attn_plan_host", "attn_plan_info", "attn_plan_blocks",
            "attn_plan_segments", "attn_plan_cta_heads", "attn_plan_stage_units",
            "attn_plan_merge_ctas",
            "attn_debug_tc_gemm", "attn_debug_stamps",
            "attn_run_paged_no_workspace",
            "attn_append_kv", "attn_plan_replayable", "attn_plan_replayable_host",
            "attn_plan_replan_host", "attn_plan_fetch_device")


class attn_problem_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim_qk", ctypes.c_int32),
                ("head_dim_v", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("page_table_stride", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int), ("window", ctypes.c_int32),
                ("has_sinks", ctypes.c_int32),
                ("qo_indptr_host", ctypes.POINTER(ctypes.c_int32)),
                ("seq_lens_host", ctypes.POINTER(ctypes.c_int32))]


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {attn_status_string(status)} ({status})")


_LIB = None
_STAMPS = False      # load the profiling build (attn_debug_stamps records) instead


def library_path() -> str:
    return _build.lib_path(_STAMPS)


def use_stamps_build() -> None:
    """Make load() use the profiling build of the same sources, whose split-KV
    kernel records timestamps (include/attn_paged_debug.h, attn_debug_stamps).
    Call before the library is first loaded."""
    global _STAMPS
    if _LIB is not None and not _STAMPS:
        raise RuntimeError("the default library is already loaded")
    _STAMPS = True


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libattn_paged.so (building it first when missing or stale)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.build(stamps=_STAMPS) if build_if_missing else library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libattn_paged.so not found at {path}")
    L = ctypes.CDLL(path)
    vp, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
    L.attn_plan.argtypes = [ctypes.POINTER(attn_problem_t), ctypes.c_int, ctypes.POINTER(vp),
                            ctypes.POINTER(ctypes.c_size_t)]
    L.attn_run_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int32, ctypes.c_float,
                                 ctypes.c_float, ctypes.c_float, vp, vp, vp, ctypes.c_size_t, vp]
    L.attn_run_phase.argtypes = [vp, ctypes.c_int32] + L.attn_run_paged.argtypes[1:]
    L.attn_run_paged_no_workspace.argtypes = L.attn_run_paged.argtypes[:14] + [vp]
    L.attn_append_kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp]
    L.attn_plan_destroy.argtypes = [vp]
    L.attn_get_device_error.argtypes = [vp, vp, i32p]
    L.attn_status_string.argtypes = [ctypes.c_int]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_plan_host.argtypes = [ctypes.POINTER(attn_problem_t), ctypes.c_int32, ctypes.POINTER(vp)]
    L.attn_plan_info.argtypes = [vp, i32p]
    L.attn_plan_blocks.argtypes = [vp, i32p]
    L.attn_plan_segments.argtypes = [vp, i32p]
    L.attn_plan_replayable.argtypes = L.attn_plan.argtypes
    L.attn_plan_replayable_host.argtypes = L.attn_plan_host.argtypes
    L.attn_plan_replan_host.argtypes = [vp, i32p, i32p]
    L.attn_plan_fetch_device.argtypes = [vp]
    L.attn_debug_tc_gemm.argtypes = [ctypes.c_int32] * 4 + [vp, vp, vp, vp, vp]
    L.attn_debug_stamps.argtypes = [vp, ctypes.c_int32]
    for name in EXPORTED:
        if name != "attn_status_string":
            getattr(L, name).restype = ctypes.c_int
    _LIB = L
    return L


def attn_status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, what)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


class Plan:
    """Owns an attn_plan_t handle (destroyed with the object)."""

    def __init__(self, handle: int, workspace_bytes: int, device: int, keep):
        self.handle = handle
        self.workspace_bytes = workspace_bytes
        self.device = device
        self._keep = keep

    def destroy(self) -> None:
        if self.handle:
            load().attn_plan_destroy(ctypes.c_void_p(self.handle))
            self.handle = 0

    def __del__(self):
        try:
            self.destroy()
        except Exception:  # interpreter shutdown
            pass


def make_problem(batch, num_q_heads, num_kv_heads, page_size, num_pages, page_table_stride,
                 kv_dtype, window, has_sinks, qo_indptr, seq_lens, head_dim_qk=192,
                 head_dim_v=128):
    """Build an attn_problem_t from host int32 sequences (numpy arrays or lists)."""
    import numpy as np
    qo = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    p = attn_problem_t(batch, num_q_heads, num_kv_heads, head_dim_qk, head_dim_v, page_size,
                       num_pages, page_table_stride, int(kv_dtype), window, int(bool(has_sinks)),
                       qo.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                       sl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    return p, (qo, sl)


def attn_plan(problem: attn_problem_t, device: int, keep=None) -> Plan:
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(load().attn_plan(ctypes.byref(problem), int(device), ctypes.byref(h), ctypes.byref(ws)),
           "attn_plan")
    return Plan(h.value, ws.value, device, keep)


def attn_plan_host(problem: attn_problem_t, num_sms: int, keep=None) -> Plan:
    h = ctypes.c_void_p()
    _check(load().attn_plan_host(ctypes.byref(problem), int(num_sms), ctypes.byref(h)),
           "attn_plan_host")
    return Plan(h.value, 0, -1, keep)


def attn_plan_replayable(bounds: attn_problem_t, device: int, keep=None) -> Plan:
    """A plan whose lengths are read on the device at every run (seq_lens in
    `bounds` are upper bounds; the query layout is fixed)."""
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(load().attn_plan_replayable(ctypes.byref(bounds), int(device), ctypes.byref(h),
                                       ctypes.byref(ws)), "attn_plan_replayable")
    return Plan(h.value, ws.value, device, keep)


def attn_plan_replayable_host(bounds: attn_problem_t, num_sms: int, keep=None) -> Plan:
    h = ctypes.c_void_p()
    _check(load().attn_plan_replayable_host(ctypes.byref(bounds), int(num_sms), ctypes.byref(h)),
           "attn_plan_replayable_host")
    return Plan(h.value, 0, -1, keep)


def attn_plan_replan_host(plan: Plan, seq_lens) -> int:
    """Rebuild a replayable plan's host work list for `seq_lens`; returns the
    device error bits the lengths would raise."""
    import numpy as np
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    err = ctypes.c_int32()
    _check(load().attn_plan_replan_host(ctypes.c_void_p(plan.handle),
                                        sl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                        ctypes.byref(err)), "attn_plan_replan_host")
    return err.value


def attn_plan_fetch_device(plan: Plan) -> None:
    """Copy the work list the device planner last wrote into the host copy."""
    _check(load().attn_plan_fetch_device(ctypes.c_void_p(plan.handle)), "attn_plan_fetch_device")


def attn_plan_destroy(plan: Plan) -> None:
    plan.destroy()


def _run_args(plan, q, k_cache, v_cache, page_table, seq_lens, qo_indptr, sinks, window,
              softmax_scale, k_scale, v_scale, out, lse_out, workspace, stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seq_lens),
            _ptr(qo_indptr), _ptr(sinks), int(window), float(softmax_scale), float(k_scale),
            float(v_scale), _ptr(out), _ptr(lse_out), _ptr(workspace), ws_bytes,
            ctypes.c_void_p(int(stream)))


def attn_run_paged(plan: Plan, q, k_cache, v_cache, page_table, seq_lens, qo_indptr, sinks,
                   window: int, softmax_scale: float, k_scale: float, v_scale: float, out,
                   lse_out=None, workspace=None, stream=None) -> None:
    """Launch on `stream` (a torch.cuda.Stream, a raw handle, or None for torch's
    current stream).  Pointer-only; nothing is synchronised."""
    args = _run_args(plan, q, k_cache, v_cache, page_table, seq_lens, qo_indptr, sinks, window,
                     softmax_scale, k_scale, v_scale, out, lse_out, workspace, stream)
    _check(load().attn_run_paged(ctypes.c_void_p(plan.handle), *args), "attn_run_paged")


def attn_run_phase(plan: Plan, phase: int, q, k_cache, v_cache, page_table, seq_lens,
                   qo_indptr, sinks, window: int, softmax_scale: float, k_scale: float,
                   v_scale: float, out, lse_out=None, workspace=None, stream=None) -> None:
    """One of the two launches of attn_run_paged (0: split-KV kernel, 1: merge)."""
    args = _run_args(plan, q, k_cache, v_cache, page_table, seq_lens, qo_indptr, sinks, window,
                     softmax_scale, k_scale, v_scale, out, lse_out, workspace, stream)
    _check(load().attn_run_phase(ctypes.c_void_p(plan.handle), int(phase), *args),
           "attn_run_phase")


NO_WORKSPACE_MAX_BYTES = 16 * 1024 * 1024


def attn_run_paged_no_workspace(plan: Plan, q, k_cache, v_cache, page_table, seq_lens, qo_indptr,
                                sinks, window: int, softmax_scale: float, k_scale: float,
                                v_scale: float, out, lse_out=None, stream=None) -> None:
    """attn_run_paged on the library's own scratch (no workspace argument), for
    callers that cannot allocate device memory."""
    args = _run_args(plan, q, k_cache, v_cache, page_table, seq_lens, qo_indptr, sinks, window,
                     softmax_scale, k_scale, v_scale, out, lse_out, None, stream)
    args = args[:13] + args[15:]        # drop the workspace pointer and size
    _check(load().attn_run_paged_no_workspace(ctypes.c_void_p(plan.handle), *args),
           "attn_run_paged_no_workspace")


def attn_append_kv(plan: Plan, k_new, v_new, k_cache, v_cache, page_table, seq_lens, qo_indptr,
                   k_scale: float = 1.0, v_scale: float = 1.0, stream=None) -> None:
    """Write the plan's new tokens' K/V rows into the paged caches (FP8 caches
    get E4M3 codes of value / scale)."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    _check(load().attn_append_kv(ctypes.c_void_p(plan.handle), _ptr(k_new), _ptr(v_new),
                                 _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seq_lens),
                                 _ptr(qo_indptr), float(k_scale), float(v_scale),
                                 ctypes.c_void_p(int(stream))), "attn_append_kv")


def attn_get_device_error(plan: Plan) -> int:
    err = ctypes.c_int32()
    _check(load().attn_get_device_error(ctypes.c_void_p(plan.handle), None, ctypes.byref(err)),
           "attn_get_device_error")
    return err.value


def attn_plan_info(plan: Plan) -> dict:
    info = (ctypes.c_int32 * 8)()
    _check(load().attn_plan_info(ctypes.c_void_p(plan.handle), info), "attn_plan_info")
    return dict(blocks=info[0], segments=info[1], ctas=info[2], rows_per_block=info[3],
                key_tile=info[4], multi_split_blocks=info[5],
                workspace_bytes=(info[7] << 31) | info[6])


def attn_plan_blocks(plan: Plan):
    import numpy as np
    n = attn_plan_info(plan)["blocks"]
    arr = np.zeros((max(n, 1), 8), np.int32)
    _check(load().attn_plan_blocks(ctypes.c_void_p(plan.handle),
                                   arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
           "attn_plan_blocks")
    return arr[:n]


def attn_plan_segments(plan: Plan):
    import numpy as np
    n = attn_plan_info(plan)["segments"]
    arr = np.zeros((max(n, 1), 5), np.int32)
    _check(load().attn_plan_segments(ctypes.c_void_p(plan.handle),
                                     arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
           "attn_plan_segments")
    return arr[:n]


def attn_plan_cta_heads(plan: Plan):
    """Each CTA's head record as 20 int32 (see attn_plan_cta_heads)."""
    import numpy as np
    n = attn_plan_info(plan)["ctas"]
    arr = np.zeros((max(n, 1), 20), np.int32)
    _check(load().attn_plan_cta_heads(ctypes.c_void_p(plan.handle),
                                      arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
           "attn_plan_cta_heads")
    return arr[:n]


def attn_plan_merge_ctas(plan: Plan) -> int:
    """CTAs of the merge kernel a run of `plan` launches (0: none)."""
    n = ctypes.c_int32(0)
    _check(load().attn_plan_merge_ctas(ctypes.c_void_p(plan.handle), ctypes.byref(n)),
           "attn_plan_merge_ctas")
    return n.value


def attn_plan_stage_units(plan: Plan):
    """A prefill plan's staging units as 8 int32 each (see attn_plan_stage_units)."""
    import numpy as np
    n = ctypes.c_int32(0)
    _check(load().attn_plan_stage_units(ctypes.c_void_p(plan.handle), ctypes.byref(n), None),
           "attn_plan_stage_units")
    arr = np.zeros((max(n.value, 1), 8), np.int32)
    _check(load().attn_plan_stage_units(ctypes.c_void_p(plan.handle), ctypes.byref(n),
                                        arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
           "attn_plan_stage_units")
    return arr[:n.value]


def attn_debug_tc_gemm(mode: int, variant: int, ab_type: int, n: int, a, b, d, status,
                       stream=None) -> None:
    """Tensor-core building-block self test (include/attn_paged_debug.h)."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    _check(load().attn_debug_tc_gemm(int(mode), int(variant), int(ab_type), int(n), _ptr(a),
                                     _ptr(b), _ptr(d), _ptr(status), ctypes.c_void_p(int(stream))),
           "attn_debug_tc_gemm")


ATTN_DEBUG_STAMP_CTAS = 160
ATTN_DEBUG_STAMP_EVENTS = 16


def attn_debug_stamps(clear: bool = True):
    """Timestamps of the split-KV kernel's last launches, a
    [ATTN_DEBUG_STAMP_CTAS, ATTN_DEBUG_STAMP_EVENTS] uint64 array (profiling build
    only; the default build raises ATTN_ERR_UNSUPPORTED)."""
    import numpy as np
    arr = np.zeros((ATTN_DEBUG_STAMP_CTAS, ATTN_DEBUG_STAMP_EVENTS), dtype=np.uint64)
    _check(load().attn_debug_stamps(ctypes.c_void_p(arr.ctypes.data), int(bool(clear))),
           "attn_debug_stamps")
    return arr
