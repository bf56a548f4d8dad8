"""Build the CUDA library libattn_paged.so in-tree (nvcc, sm_103a only).

Objects and the shared library go to ``asymmetric_kv_paged_gb300/_build/<machine>/``;
translation units compile in parallel.  ``build(stamps=True)`` makes the profiling
build (the split-KV kernel records start-up and epilogue timestamps, read with
attn_debug_stamps) in ``_build/<machine>-stamps/``; nothing else loads it.  The CUDA runtime is linked statically and
the driver API is reached through the runtime's entry-point query, so the library
loads (and its symbols can be listed) on a machine without a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "attn_tc.cu", "attn_prefill.cu", "merge.cu", "replan.cu", "no_workspace.cu", "kv_append.cu",
           "kv_stage.cu",
           "tc_selftest.cu", "planner.cpp"]
HEADERS = ["plan.hpp", "replan.hpp", "kernels.hpp", "tc_common.cuh", "e4m3.cuh", "stamps.cuh"]


def build_dir(stamps: bool = False) -> str:
    return os.path.join(PKG, "_build", platform.machine() + ("-stamps" if stamps else ""))


def lib_path(stamps: bool = False) -> str:
    return os.path.join(build_dir(stamps), "libattn_paged.so")


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files += [os.path.join(INCLUDE, h) for h in os.listdir(INCLUDE) if h.endswith(".h")]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, obj: str, stamps: bool = False) -> None:
    path = os.path.join(CSRC, src)
    if src.endswith(".cpp"):
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", f"-I{INCLUDE}", f"-I{CSRC}",
               "-c", path, "-o", obj]
    else:
        cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}", "-c", path, "-o", obj]
        if os.environ.get("AKP_PTXAS_VERBOSE"):
            cmd.insert(1, "-Xptxas=-v")
        if stamps:
            cmd.insert(1, "-DAKP_STAMPS")
    subprocess.run(cmd, check=True)


def build(force: bool = False, verbose: bool = False, stamps: bool = False) -> str:
    out = lib_path(stamps)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= _inputs_mtime():
        return out
    bdir = build_dir(stamps)
    os.makedirs(bdir, exist_ok=True)
    objs = [os.path.join(bdir, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 1)) as ex:
        futs = [ex.submit(_compile, s, o, stamps) for s, o in zip(SOURCES, objs)]
        for f in futs:
            f.result()
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run([_nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, out)
    if verbose:
        print(f"built {out}", file=sys.stderr)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, stamps="--stamps" in sys.argv)
