"""snapkv_decode_attend_noalloc: decode attention for callers that cannot allocate device memory.

Some callers of this library cannot hand it a workspace — a plugin or custom-operator interface
that passes only inputs and outputs, or a latency-critical loop where cudaMalloc is not allowed.
This entry point keeps its scratch in an array built into the library instead. These checks call
it through the C ABI and compare it with snapkv_decode_attend (the workspace entry point) on two
calls in a row, within the decode tolerance the other tests use, and check that a problem too
large for the built-in array is refused before anything runs. This file is named to be collected
last, so a run that stops at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

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


def test_noalloc_matches_workspace_entry_point_on_two_calls(dev):
    from kv_cache_compression_gb300 import snapkv
    lib = snapkv.lib()
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator().manual_seed(123)
    B, H, cap, d = 4, 8, 1100, 128
    kc = torch.randn(B, H, cap, d, generator=g).to(torch.bfloat16).to(dev)
    vc = torch.randn(B, H, cap, d, generator=g).to(torch.bfloat16).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    calls = [(torch.tensor([1, 300, 1099, 1100], dtype=torch.int32), 1.0),
             (torch.tensor([1024, 7, 256, 513], dtype=torch.int32), 3.0)]
    for n, (lens, qscale) in enumerate(calls):
        q = (torch.randn(B, H, d, generator=g) * qscale).to(torch.bfloat16).to(dev)
        length = lens.to(dev)
        ref = snapkv.decode_attend(q, kc, vc, length)
        free_before = torch.cuda.mem_get_info(dev)[0]
        st = _noalloc(lib, q, kc, vc, length, out, status, stream)
        torch.cuda.synchronize(dev)
        assert st == snapkv.OK, snapkv.status_string(st)
        assert int(status.item()) == 0
        if n > 0:   # after the first call on the device nothing more is set up
            assert torch.cuda.mem_get_info(dev)[0] == free_before
        check_decode(to_numpy_f32(out), to_numpy_f32(ref).astype("float64"), True, where=f"call {n}")
        assert torch.equal(out, ref)   # same kernel, same split order: identical bits


def test_noalloc_refuses_problems_beyond_its_scratch(dev):
    from kv_cache_compression_gb300 import snapkv
    lib = snapkv.lib()
    stream = torch.cuda.current_stream(dev)
    # 64 x 32 heads over a 4096-row cache need 2048 * 16 splits * 130 floats = 17 MB of partials.
    B, H, cap, d = 64, 32, 4096, 128
    kc = torch.empty(B, H, cap, d, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    q = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    length = torch.full((B,), 10, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    assert snapkv.decode_workspace_size(B, H, d, cap) > 16 << 20
    st = _noalloc(lib, q, kc, vc, length, out, status, stream)
    assert st == snapkv.ERR_WORKSPACE
