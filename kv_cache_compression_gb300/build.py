"""Build libsnapkv.so in-tree for sm_103a with nvcc (one -gencode, translation units in parallel).

build(checked=True) makes libsnapkv_checked.so instead: the same kernels compiled with
-DSNAPKV_CHECKED, where every global index a kernel computes is checked before the access and a
violation is reported as SNAPKV_ERR_INTERNAL (the tests run part of the parity suite on it)."""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

_HERE = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_HERE, "csrc")
_BUILD = os.path.join(_HERE, "_build")
SOURCES = ["abi.cu", "vote_simt.cu", "vote_tc.cu", "vote_cluster.cu", "pool_topk.cu", "gather.cu", "decode.cu", "hit_rate.cu"]
HEADERS = ["snapkv_common.cuh", "snapkv_internal.h", "sm100_ptx.cuh", "tc_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def lib_path(checked: bool = False) -> str:
    return os.path.join(_HERE, "libsnapkv_checked.so" if checked else "libsnapkv.so")


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{proc.stdout}\n{proc.stderr}")
    return proc.stdout + proc.stderr


def _stale(out, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    """Compile every kernel file and link libsnapkv.so (or the bounds-checked libsnapkv_checked.so)
    next to this package."""
    build_dir = _BUILD + ("_checked" if checked else "")
    extra = ["-DSNAPKV_CHECKED"] if checked else []
    os.makedirs(build_dir, exist_ok=True)
    header_deps = [os.path.join(_CSRC, h) for h in HEADERS] + [
        os.path.join(os.path.dirname(_HERE), "include", "snapkv.h")]
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(_CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + header_deps):
            cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", s, "-o", o]
            if verbose_ptxas:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)
    logs = []
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            logs = list(ex.map(_run, jobs))
    out = lib_path(checked)
    if force or jobs or _stale(out, objs):
        tmp = out + ".tmp"
        _run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, out)
    if verbose_ptxas:
        print("\n".join(logs))
    return out


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose_ptxas="-v" in sys.argv))
