"""The bounds-checked build of the library, a stand-in for a memory checker on this GPU pool.

kv_cache_compression_gb300.build.build(checked=True) compiles the same kernels with -DSNAPKV_CHECKED:
every global index a kernel computes from data or from its own bookkeeping (gathered source rows and
cache rows, vote and row-sum entries, decode cache rows and bulk-copy ranges) is checked before the
access, and a violation is reported as SNAPKV_ERR_INTERNAL in the device status word. Here a child
process loads that build (SNAPKV_CHECKED=1; one build per process) and runs a cross-section of the
GPU parity tests on it: every call must report a clean status and match the oracle.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

SUBSET = [
    "tests/test_gpu_compress.py::test_tiny_fp32_every_head",
    "tests/test_gpu_compress.py::test_llama_layer_every_head",
    "tests/test_gpu_compress.py::test_edge_cases",
    "tests/test_gpu_compress.py::test_large_batch_top_k_shapes",
    "tests/test_gpu_compress.py::test_zero_queries_keep_the_first_k_at_large_batch",
    "tests/test_gpu_decode.py",
    "tests/test_gpu_varlen.py",
    "tests/test_gpu_gqa.py",
    "tests/test_gpu_hit_rate.py",
]


def test_parity_subset_on_the_bounds_checked_build(gpu_device):
    from kv_cache_compression_gb300 import build as kbuild
    path = kbuild.build(checked=True)
    assert path.endswith("libsnapkv_checked.so") and os.path.exists(path)
    env = dict(os.environ, SNAPKV_CHECKED="1")
    probe = subprocess.run([sys.executable, "-c", "from kv_cache_compression_gb300 import snapkv; "
                            "print(snapkv.lib()._name)"], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip().endswith("libsnapkv_checked.so"), probe.stderr
    run = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *SUBSET],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert run.returncode == 0, run.stdout[-4000:] + run.stderr[-2000:]
    assert " passed" in run.stdout
