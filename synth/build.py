"""Build the host (gcc) and device (nvcc, sm_103a) copies of the input generator in-tree."""
from __future__ import annotations

import os
import shutil
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def host_lib_path() -> str:
    return os.path.join(_HERE, "libsynth_host.so")


def dev_lib_path() -> str:
    return os.path.join(_HERE, "libsynth_dev.so")


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    proc = subprocess.run(cmd, cwd=_HERE, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{proc.stdout}\n{proc.stderr}")


def _stale(out: str, srcs) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(os.path.join(_HERE, s)) > t for s in srcs)


def build_host(force: bool = False) -> str:
    out = host_lib_path()
    srcs = ["synth_host.c", "synth_gen.h"]
    if force or _stale(out, srcs):
        tmp = out + ".tmp"
        _run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
              "-pthread", "-o", tmp, "synth_host.c"])
        os.replace(tmp, out)
    return out


def build_dev(force: bool = False) -> str:
    out = dev_lib_path()
    srcs = ["synth_dev.cu", "synth_gen.h"]
    if force or _stale(out, srcs):
        tmp = out + ".tmp"
        _run([_nvcc(), "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-Xcompiler", "-fPIC", "-shared", "-o", tmp, "synth_dev.cu"])
        os.replace(tmp, out)
    return out


def build_all(force: bool = False):
    return build_host(force), build_dev(force)


if __name__ == "__main__":
    print(build_all(force=True))
