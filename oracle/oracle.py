"""FP64 CPU oracle for paged attention with asymmetric K/V head dims (numpy front end).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg of
the benchmark are the only callers.  The product path never imports this module,
and this module imports nothing from the product package.

The arithmetic lives in ``attn_oracle.c`` (plain FP64 C, OpenMP over rows); this
file only builds it with gcc and marshals numpy arrays.  The definition it
computes is written out at the top of the C file.  Parity pins for every function
here live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_CACHE: dict = {}


def lib_path(mutant: int = 0) -> str:
    tag = "" if mutant == 0 else f"_mutant{mutant}"
    return os.path.join(_BUILD_DIR, f"liboracle_{platform.machine()}{tag}.so")


def build(force: bool = False, mutant: int = 0) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, IEEE semantics kept: no -ffast-math,
    no FMA contraction).  mutant > 0 builds a deliberately wrong variant for the
    pin-strength tests."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(
        ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
         "-ffp-contract=off", f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"],
        check=True)
    os.replace(tmp, out)
    return out


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _problem_args(pb: dict):
    """Marshal a problem dict (numpy arrays; see Workload.host_arrays)."""
    q = np.ascontiguousarray(pb["q"], dtype=np.uint16)
    kc = np.ascontiguousarray(pb["k_cache"])
    vc = np.ascontiguousarray(pb["v_cache"])
    assert kc.dtype == vc.dtype and kc.dtype in (np.uint16, np.uint8)
    kv_dtype = 0 if kc.dtype == np.uint16 else 1
    qo = np.ascontiguousarray(pb["qo_indptr"], dtype=np.int32)
    sl = np.ascontiguousarray(pb["seq_lens"], dtype=np.int32)
    pt = np.ascontiguousarray(pb["page_table"], dtype=np.int32)
    sinks = pb.get("sinks")
    sinks_arr = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float64)
    hq, dqk = q.shape[1], q.shape[2]
    num_pages, page_size, hkv, _ = kc.shape
    dv = vc.shape[3]
    keep = (q, kc, vc, qo, sl, pt, sinks_arr)
    args = [len(sl), hq, hkv, dqk, dv, page_size, pt.shape[1], kv_dtype, int(pb.get("window", 0)),
            num_pages, float(pb["softmax_scale"]), float(pb.get("k_scale", 1.0)),
            float(pb.get("v_scale", 1.0)), _ptr(qo, ctypes.c_int32), _ptr(sl, ctypes.c_int32),
            _ptr(pt, ctypes.c_int32), q.ctypes.data, kc.ctypes.data, vc.ctypes.data,
            None if sinks_arr is None else _ptr(sinks_arr, ctypes.c_double)]
    return args, keep, hq, dv, int(qo[-1])


class Oracle:
    """One loaded build of the oracle (the real one, or a planted mutant)."""

    def __init__(self, mutant: int = 0):
        L = ctypes.CDLL(build(mutant=mutant))
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        f64p = ctypes.POINTER(ctypes.c_double)
        vp = ctypes.c_void_p
        problem = [ctypes.c_int] * 9 + [ctypes.c_int64] + [ctypes.c_double] * 3 + \
            [i32p, i32p, i32p, vp, vp, vp, f64p]
        L.oracle_attn_paged.argtypes = problem + [i64p, ctypes.c_int64, f64p, f64p, ctypes.c_int]
        L.oracle_attn_paged.restype = ctypes.c_int
        L.oracle_attn_partial.argtypes = problem + [ctypes.c_int64, ctypes.c_int64, i64p,
                                                    ctypes.c_int64, f64p, f64p, ctypes.c_int]
        L.oracle_attn_partial.restype = ctypes.c_int
        L.oracle_merge.argtypes = [ctypes.c_int, ctypes.c_int, f64p, f64p, ctypes.c_double,
                                   f64p, f64p]
        L.oracle_merge.restype = None
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_double.restype = ctypes.c_double
        L.oracle_num_threads.restype = ctypes.c_int
        self.lib = L
        self.mutant = mutant

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def bf16_to_double(self, bits: int) -> float:
        return float(self.lib.oracle_bf16_to_double(int(bits)))

    def e4m3_to_double(self, code: int) -> float:
        return float(self.lib.oracle_e4m3_to_double(int(code)))

    def attn_paged(self, pb: dict, rows=None, nthreads: int = 0):
        """Full attention rows (sink included).  rows: flat indices tok*Hq+h, or None.

        Returns (out [n_rows, Dv] float64, lse [n_rows] float64); with rows=None the
        result is shaped [total_q, Hq, Dv] and [total_q, Hq].
        """
        args, keep, hq, dv, total_q = _problem_args(pb)
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = total_q * hq if rows is None else rows_arr.size
        out = np.zeros((n, dv), np.float64)
        lse = np.zeros(n, np.float64)
        rc = self.lib.oracle_attn_paged(
            *args, None if rows_arr is None else _ptr(rows_arr, ctypes.c_int64), n,
            _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), int(nthreads))
        del keep
        if rc:
            raise ValueError(f"oracle_attn_paged failed with status {rc}")
        if rows is None:
            return out.reshape(total_q, hq, dv), lse.reshape(total_q, hq)
        return out, lse

    def attn_partial(self, pb: dict, key_lo: int, key_hi: int, rows=None, nthreads: int = 0):
        """Split partial over logical keys [key_lo, key_hi): normalised out and lse, no sink."""
        args, keep, hq, dv, total_q = _problem_args(pb)
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = total_q * hq if rows is None else rows_arr.size
        out = np.zeros((n, dv), np.float64)
        lse = np.zeros(n, np.float64)
        rc = self.lib.oracle_attn_partial(
            *args, int(key_lo), int(key_hi),
            None if rows_arr is None else _ptr(rows_arr, ctypes.c_int64), n,
            _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), int(nthreads))
        del keep
        if rc:
            raise ValueError(f"oracle_attn_partial failed with status {rc}")
        return out, lse

    def merge(self, o_parts, lse_parts, sigma: float = float("-inf")):
        """LSE combine of split partials of one row: o_parts [S, Dv], lse_parts [S]."""
        o = np.ascontiguousarray(o_parts, dtype=np.float64)
        l = np.ascontiguousarray(lse_parts, dtype=np.float64)
        S, dv = o.shape
        out = np.zeros(dv, np.float64)
        lse = np.zeros(1, np.float64)
        self.lib.oracle_merge(S, dv, _ptr(o, ctypes.c_double), _ptr(l, ctypes.c_double),
                              float(sigma), _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
        return out, float(lse[0])


def load(mutant: int = 0) -> Oracle:
    with _LOCK:
        if mutant not in _CACHE:
            _CACHE[mutant] = Oracle(mutant)
        return _CACHE[mutant]


def num_threads() -> int:
    return load().num_threads()


def attn_paged(pb: dict, rows=None, nthreads: int = 0):
    return load().attn_paged(pb, rows, nthreads)


def attn_partial(pb: dict, key_lo: int, key_hi: int, rows=None, nthreads: int = 0):
    return load().attn_partial(pb, key_lo, key_hi, rows, nthreads)


def merge(o_parts, lse_parts, sigma: float = float("-inf")):
    return load().merge(o_parts, lse_parts, sigma)
