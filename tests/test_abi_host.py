"""Host-only checks of the C ABI: the library loads, exports every symbol include/snapkv.h
declares, and rejects bad arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import subprocess

import pytest

from kv_cache_compression_gb300 import build as kbuild
from kv_cache_compression_gb300 import snapkv as sk


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return sk.lib()


def test_exports_every_declared_function(lib):
    names = sk.declared_functions()
    assert len(names) == 17
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", sk.library_path()], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported
    assert lib.snapkv_abi_version() == 100


def test_params_struct_layout():
    assert ctypes.sizeof(sk.CompressParams) == 56
    assert sk.CompressParams.l_prompt.offset == 16 and sk.CompressParams.ratio_p.offset == 32
    assert sk.CompressParams.dtype.offset == 48


def _params(**kw):
    base = dict(batch=1, heads=4, head_dim=64, l_obs=32, l_prompt=1024, pool_kernel=7, ratio_p=0.05, budget=0,
                scope="prompt_causal", dtype=sk.F32)
    base.update(kw)
    return sk.make_params(**base)


def test_kept_slots_on_host(lib):
    assert sk.kept(_params()) == 49                       # floor(0.05 * 992)
    assert sk.kept(_params(budget=1024, l_prompt=16384)) == 1024
    assert sk.kept(_params(budget=10 ** 9)) == 992        # budget beyond the prefix keeps everything
    assert sk.kept(_params(ratio_p=1.0)) == 992
    assert sk.kept(_params(ratio_p=0.0)) == 0
    assert sk.kept(_params(l_prompt=32)) == -1             # L_obs must be < L_prompt
    assert sk.kept(_params(pool_kernel=4)) == -1          # even kernel unsupported
    assert sk.kept(_params(head_dim=96)) == -1
    assert sk.kept(_params(ratio_p=1.5)) == -1
    for kw in ({}, {"budget": 7}, {"ratio_p": 1.0}, {"l_prompt": 32}):
        assert sk.compress_k(_params(**kw)) == sk.kept(_params(**kw))   # the alias gives the same k
    assert sk.kept(_params(ratio_p=float("nan"))) == -1


def test_workspace_size_is_positive_and_monotone(lib):
    a = sk.compress_workspace_size(_params())
    b = sk.compress_workspace_size(_params(l_prompt=4096))
    assert 0 < a < b and a % 256 == 0
    assert sk.compress_workspace_size(_params(pool_kernel=2)) == 0
    assert sk.decode_workspace_size(2, 4, 128, 1000) > 0
    assert sk.decode_workspace_size(2, 4, 100, 1000) == 0


def _call_compress(lib, params, **ptrs):
    P = ctypes.c_void_p
    good = {"q": 0x1000, "k": 0x100000, "v": 0x200000, "ko": 0x300000, "vo": 0x400000, "len": 0x500000,
            "ws": 0x600000}
    good.update(ptrs)
    return lib.snapkv_compress(ctypes.byref(params), P(good["q"]), P(good["k"]), P(good["v"]), P(good["ko"]),
                               P(good["vo"]), ptrs.get("cap", 81), P(good["len"]), None, None, P(good["ws"]),
                               ptrs.get("ws_bytes", 1 << 30), None, None)


def test_compress_rejects_bad_arguments_before_launch(lib):
    p = _params()
    assert lib.snapkv_compress(None, None, None, None, None, None, 81, None, None, None, None, 0, None, None) \
        == sk.ERR_INVALID_ARG
    assert _call_compress(lib, p, q=0) == sk.ERR_INVALID_ARG                  # NULL query
    assert _call_compress(lib, p, k=0x100008) == sk.ERR_INVALID_ARG           # misaligned key pointer
    assert _call_compress(lib, p, cap=80) == sk.ERR_CAPACITY                  # cap < k + L_obs
    assert _call_compress(lib, p, ws=0) == sk.ERR_WORKSPACE
    assert _call_compress(lib, p, ws_bytes=16) == sk.ERR_WORKSPACE
    assert _call_compress(lib, p, ko=0x100000) == sk.ERR_INVALID_ARG          # output aliases input
    assert _call_compress(lib, _params(pool_kernel=6)) == sk.ERR_UNSUPPORTED
    assert _call_compress(lib, _params(head_dim=80)) == sk.ERR_UNSUPPORTED
    assert _call_compress(lib, _params(l_obs=0)) == sk.ERR_INVALID_ARG
    assert _call_compress(lib, _params(scope="prefix_only", dtype=7)) == sk.ERR_INVALID_ARG
    bad = _params()
    bad.algo = 4
    assert _call_compress(lib, bad) == sk.ERR_INVALID_ARG


def test_decode_and_append_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    assert lib.snapkv_append(None, P(16), P(32), P(48), 10, P(64), 1, 1, 64, 0, None, None) == sk.ERR_INVALID_ARG
    assert lib.snapkv_append(P(16), P(32), P(48), P(64), 10, P(80), 1, 1, 72, 0, None, None) == sk.ERR_UNSUPPORTED
    assert lib.snapkv_append(P(16), P(32), P(48), P(64), 0, P(80), 1, 1, 64, 0, None, None) == sk.ERR_INVALID_ARG
    assert lib.snapkv_decode_attend(P(16), P(32), P(48), 10, P(64), P(80), 1, 1, 64, 0, None, 0, None, None) \
        == sk.ERR_WORKSPACE
    assert lib.snapkv_decode_attend(P(16), P(32), P(48), 10, P(64), P(88), 1, 1, 64, 0, P(256), 1 << 20, None,
                                    None) == sk.ERR_INVALID_ARG               # misaligned output
    f = lib.snapkv_append_decode_attend
    ok = dict(q=P(16), kn=P(32), vn=P(48), kc=P(64), vc=P(80), lin=P(96), lout=P(112), out=P(128))

    def fused(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["kn"], a["vn"], a["kc"], a["vc"], 10, a["lin"], a["lout"], a["out"], 2, 1, 64, 0,
                 a.get("ws", P(256)), 1 << 20, None, None)
    assert fused(kn=None) == sk.ERR_INVALID_ARG
    assert fused(lout=None) == sk.ERR_INVALID_ARG
    assert fused(lout=P(100)) == sk.ERR_INVALID_ARG          # overlaps len_in (two sequences, 8 bytes)
    assert fused(lout=P(96)) == sk.ERR_INVALID_ARG           # the same array
    assert fused(vn=P(40)) == sk.ERR_INVALID_ARG             # misaligned new row
    assert fused(ws=None) == sk.ERR_WORKSPACE


def test_gqa_rejects_bad_groupings(lib):
    P = ctypes.c_void_p
    p = _params(heads=4)
    ws = sk.compress_workspace_size(p, 8)
    assert ws > sk.compress_workspace_size(p)               # more window rows per KV head
    assert sk.compress_workspace_size(p, 6) == 0             # not a multiple of the KV heads
    assert sk.compress_workspace_size(p, 20) == 0            # 5 x 32 window rows > 128
    args = (P(16), P(32), P(48), P(64), P(80), 200, P(96), None, None, P(256), ws, None, None)
    assert lib.snapkv_compress_gqa(ctypes.byref(p), 6, *args) == sk.ERR_INVALID_ARG
    assert lib.snapkv_compress_gqa(ctypes.byref(p), 2, *args) == sk.ERR_INVALID_ARG   # fewer query heads
    assert lib.snapkv_compress_gqa(ctypes.byref(p), 20, *args) == sk.ERR_UNSUPPORTED


def test_varlen_workspace_and_validation(lib):
    import numpy as np
    P = ctypes.c_void_p
    p = _params(heads=2, l_prompt=1024)
    ok = np.array([1024, 200, 600], dtype=np.int64)
    p.batch = 3
    size = lib.snapkv_compress_varlen_workspace_size(ctypes.byref(p), ok.ctypes.data_as(P))
    full = sk.compress_workspace_size(_params(heads=2, l_prompt=1024, batch=3))
    assert size == full            # one launch over the batch lays it out with the longest sequence's sizes
    for bad in ([1025, 200, 600], [32, 200, 600], [0, 200, 600]):   # longer than the padding, <= L_obs
        b = np.array(bad, dtype=np.int64)
        assert lib.snapkv_compress_varlen_workspace_size(ctypes.byref(p), b.ctypes.data_as(P)) == 0
        assert lib.snapkv_compress_varlen(ctypes.byref(p), b.ctypes.data_as(P), P(16), P(32), P(48), P(64), P(80),
                                          100, P(96), None, None, P(256), 1 << 30, None, None) == sk.ERR_INVALID_ARG
    # cap must hold the longest sequence's k + L_obs
    assert lib.snapkv_compress_varlen(ctypes.byref(p), ok.ctypes.data_as(P), P(16), P(32), P(48), P(64), P(80),
                                      sk.kept(p) + 31, P(96), None, None, P(256), 1 << 30, None, None) \
        == sk.ERR_CAPACITY


def test_hit_rate_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    ok = dict(q=P(16), k=P(32), cap=100, len_=P(48), l_prefix=90, idx=P(64), k_sel=10, B=1, H=2, d=128, dt=1,
              theta=0.05, hits=P(80), total=P(96))

    def call(**kw):
        a = {**ok, **kw}
        return lib.snapkv_hit_rate(a["q"], a["k"], a["cap"], a["len_"], a["l_prefix"], a["idx"], a["k_sel"], a["B"],
                                   a["H"], a["d"], a["dt"], a["theta"], a["hits"], a["total"], None, None)
    assert call(q=None) == sk.ERR_INVALID_ARG
    assert call(l_prefix=0) == sk.ERR_INVALID_ARG
    assert call(l_prefix=101) == sk.ERR_INVALID_ARG           # beyond the cache
    assert call(theta=-0.1) == sk.ERR_INVALID_ARG
    assert call(theta=float("nan")) == sk.ERR_INVALID_ARG
    assert call(idx=None) == sk.ERR_INVALID_ARG                # k > 0 needs indices
    assert call(d=96) == sk.ERR_UNSUPPORTED
    assert call(q=P(24)) == sk.ERR_INVALID_ARG                 # misaligned


def test_status_strings(lib):
    assert sk.status_string(0) == "SNAPKV_OK"
    assert sk.status_string(4) == "SNAPKV_ERR_CAPACITY"
    assert sk.status_string(4 | 16).startswith("SNAPKV_ERR_TIMEOUT")
    assert sk.status_string(-3) == "SNAPKV_ERR_UNKNOWN"


def test_bench_decode_bytes_match_the_closed_form():
    """The decode workload's algorithmic bytes: 2080 + t rows (t = 1..128) read per head-step, over
    64 x 32 heads and 32 layers, is 274,496 rows x 2048 heads x 32 layers x 512 B = 9.21 TB, plus the
    query, output and appended row (4 rows of d bf16 per head-step)."""
    import bench
    got = bench.decode_pass_bytes([2080] * 64, 32, 128, 128, 32)
    rows = sum(2080 + t for t in range(1, 129))
    assert rows == 274_496
    assert got == (2 * rows + 4 * 128) * 64 * 32 * 32 * 128 * 2
    assert abs(got / 9.21e12 - 1) < 2e-3
