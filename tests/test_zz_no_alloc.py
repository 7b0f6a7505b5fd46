"""snapkv_decode_attend_noalloc: decode attention for callers that cannot allocate device memory.

Some callers of this library cannot hand it a workspace: a plugin or custom-operator interface
that passes only inputs and outputs, or a latency-critical loop where cudaMalloc is not allowed.
This entry point keeps the scratch that long caches need (the split kernel's partials and tickets)
in an array built into the library instead. These checks call it through the C ABI:

  * on caches longer than 16384 rows, which take the split kernel and so write and read the
    built-in array, on two calls in a row whose cache length, split count and lengths differ,
    against the CPU oracle and against snapkv_decode_attend (the workspace entry point);
  * on a short cache (no scratch used) and on a decode-workload-shaped call that is accepted;
  * that a long-cache problem too large for the array is refused before anything runs.

This file is named to be collected last, so a run that stops at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import snapkv_oracle as orc
from tests.parity import check_decode, to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(gpu_device):
    import __graft_entry__
    __graft_entry__.build()
    return gpu_device


def _noalloc(lib, q, kc, vc, length, out, status, stream):
    B, H, cap, d = kc.shape
    P = ctypes.c_void_p
    return lib.snapkv_decode_attend_noalloc(P(q.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()), cap,
                                            P(length.data_ptr()), P(out.data_ptr()), B, H, d,
                                            1 if kc.dtype == torch.bfloat16 else 0, P(status.data_ptr()),
                                            P(stream.cuda_stream))


def _against_oracle(q, kc, vc, lens, out, where):
    o, qh, kh, vh = to_numpy_f32(out), to_numpy_f32(q), to_numpy_f32(kc), to_numpy_f32(vc)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            n = min(int(lens[b]), kc.shape[2])
            ref = orc.decode_attend(qh[b, h], kh[b, h, :n], vh[b, h, :n]) if n > 0 else np.zeros(q.shape[-1])
            check_decode(o[b, h], ref, kc.dtype == torch.bfloat16, where=f"{where} b{b} h{h} n{n}")


def test_noalloc_long_caches_use_the_built_in_scratch_on_two_calls(dev):
    """Two calls in a row on caches beyond 16384 rows (the split kernel): the second has a different
    capacity, so a different number of splits and another partial layout in the array, and different
    lengths; each is checked against the oracle and bit for bit against the workspace entry point."""
    from kv_cache_compression_gb300 import snapkv
    lib = snapkv.lib()
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator().manual_seed(321)
    calls = [(2, 2, 17000, torch.tensor([17000, 1], dtype=torch.int32), 1.0),
             (2, 3, 20500, torch.tensor([9000, 20499], dtype=torch.int32), 2.5)]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for n, (B, H, cap, lens, qscale) in enumerate(calls):
        d = 128
        assert cap > 16384   # the split kernel, with its scratch in the built-in array
        kc = torch.randn(B, H, cap, d, generator=g).to(torch.bfloat16).to(dev)
        vc = torch.randn(B, H, cap, d, generator=g).to(torch.bfloat16).to(dev)
        q = (torch.randn(B, H, d, generator=g) * qscale).to(torch.bfloat16).to(dev)
        length = lens.to(dev)
        out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
        free_before = torch.cuda.mem_get_info(dev)[0]
        st = _noalloc(lib, q, kc, vc, length, out, status, stream)
        torch.cuda.synchronize(dev)
        assert st == snapkv.OK, snapkv.status_string(st)
        assert int(status.item()) == 0
        if n > 0:   # after the first long-cache call on the device nothing more is set up
            assert torch.cuda.mem_get_info(dev)[0] == free_before
        _against_oracle(q, kc, vc, lens.tolist(), out, f"call {n}")
        ref = snapkv.decode_attend(q, kc, vc, length)
        torch.cuda.synchronize(dev)
        assert torch.equal(out, ref)   # same kernel, same split order: identical bits


def test_noalloc_short_caches_and_decode_shaped_calls(dev):
    """Caches of up to 16384 rows need no scratch: a ragged short-cache call matches the oracle, and a
    call shaped like the decode workload (64 x 32 heads, 2208 rows), whose split partials would not
    fit the array, is accepted and matches the workspace entry point."""
    from kv_cache_compression_gb300 import snapkv
    lib = snapkv.lib()
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator().manual_seed(123)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B, H, cap, d = 4, 8, 1100, 128
    kc = torch.randn(B, H, cap, d, generator=g).to(torch.bfloat16).to(dev)
    vc = torch.randn(B, H, cap, d, generator=g).to(torch.bfloat16).to(dev)
    q = torch.randn(B, H, d, generator=g).to(torch.bfloat16).to(dev)
    lens = [1, 300, 1099, 1100]
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    st = _noalloc(lib, q, kc, vc, torch.tensor(lens, dtype=torch.int32, device=dev), out, status, stream)
    torch.cuda.synchronize(dev)
    assert st == snapkv.OK and int(status.item()) == 0
    _against_oracle(q, kc, vc, lens, out, "short cache")

    B, H, cap = 64, 32, 2208
    assert snapkv.decode_workspace_size(B, H, d, cap) > 16 << 20
    kc = torch.randn(B, H, cap, d, device=dev).to(torch.bfloat16)
    vc = torch.randn(B, H, cap, d, device=dev).to(torch.bfloat16)
    q = torch.randn(B, H, d, device=dev).to(torch.bfloat16)
    length = torch.randint(2081, 2209, (B,), dtype=torch.int32, device=dev)
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    st = _noalloc(lib, q, kc, vc, length, out, status, stream)
    ref = snapkv.decode_attend(q, kc, vc, length)
    torch.cuda.synchronize(dev)
    assert st == snapkv.OK and int(status.item()) == 0
    assert torch.equal(out, ref)


def test_noalloc_refuses_long_problems_beyond_its_scratch(dev):
    from kv_cache_compression_gb300 import snapkv
    lib = snapkv.lib()
    stream = torch.cuda.current_stream(dev)
    # 8 x 32 heads over a 17000-row cache need 256 heads x 133 splits x 130 floats = 17.7 MB of partials.
    B, H, cap, d = 8, 32, 17000, 128
    kc = torch.empty(B, H, cap, d, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    q = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    length = torch.full((B,), 10, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    assert snapkv.decode_workspace_size(B, H, d, cap) > 16 << 20
    st = _noalloc(lib, q, kc, vc, length, out, status, stream)
    assert st == snapkv.ERR_WORKSPACE
