"""Values in page-locked host memory, and the top-k path for prefixes beyond a cluster's reach.

The compression reads only the kept rows and the window rows of V ([SnapKV] アルゴリズム: the
gather of the selected prefix and the appended window), so V may stay in page-locked host memory
mapped into the device's address space. Every path must then give the same bytes as with V in
device memory, and match the oracle; pageable host memory is refused before anything runs.
Prefixes of more than 8 x 24K keys, or pooling kernels wider than 1025, take the single-CTA top-k
and the separate gather kernel: they are checked here against the oracle, with V on either side.
"""
import pytest
import torch

import synth
from oracle import snapkv_oracle as orc
from tests.parity import check_compress_head, to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(gpu_device):
    import __graft_entry__
    __graft_entry__.build()
    return gpu_device


def _compress(q, k, v, wl, **kw):
    from kv_cache_compression_gb300 import snapkv
    status = torch.zeros(1, dtype=torch.int32, device=k.device)
    res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p, budget=wl.budget,
                          want_vote=True, dev_status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return res


def _assert_gathered(res, k, v, lengths, l_obs):
    """Every head's cache rows are its kept rows of K and V, then the window, byte for byte."""
    for b, L in enumerate(lengths):
        ks = res["ks"][b] if "ks" in res else res["k"]
        assert int(res["len"][b]) == ks + l_obs
        for h in range(k.shape[1]):
            rows = torch.cat([res["idx"][b, h, :ks].long(), torch.arange(L - l_obs, L, device=k.device)])
            assert torch.equal(res["k_out"][b, h, :ks + l_obs], k[b, h, rows]), (b, h)
            assert torch.equal(res["v_out"][b, h, :ks + l_obs], v[b, h, rows]), (b, h)


def _check_heads(res, wl, L, heads, seq=0):
    for h in heads:
        hi = synth.host_head(wl, 0, seq, h, l_prompt=L)
        ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p,
                                budget=wl.budget)
        check_compress_head(gpu_idx=res["idx"][0, h].cpu().numpy(), gpu_kc=to_numpy_f32(res["k_out"][0, h]),
                            gpu_vc=to_numpy_f32(res["v_out"][0, h]), gpu_vote=res["vote"][0, h].cpu().numpy(),
                            ref=ref, k_in=hi.k, v_in=hi.v, l_prefix=L - wl.l_obs, l_obs=wl.l_obs,
                            where=f"L {L} K_pool {wl.pool_kernel} head {h}")


@pytest.mark.parametrize("algo", ["auto", "tensor_core_cluster", "simt"])
def test_llama_layer_values_on_host(dev, algo):
    """The Llama-2-7B-shaped layer (cluster top-k with the fused gather) with V on the host."""
    wl = synth.WORKLOADS[1]
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, wl.l_prompt, dev)
    on_host = _compress(q, k, v.cpu().pin_memory(), wl, algo=algo)
    _assert_gathered(on_host, k, v, [wl.l_prompt], wl.l_obs)
    _check_heads(on_host, wl, wl.l_prompt, heads=[0, 31])
    if algo == "tensor_core_cluster":   # deterministic: the same bits as with V on the device
        on_dev = _compress(q, k, v, wl, algo=algo)
        for key in ("k_out", "v_out", "len", "idx", "vote"):
            assert torch.equal(on_dev[key], on_host[key]), key


@pytest.mark.parametrize("v_on_host", [False, True])
def test_prefix_beyond_cluster_reach(dev, v_on_host):
    """L_prefix = 200000 > 8 x 24K: single-CTA top-k (P in global memory), then the gather kernel."""
    wl = synth.WORKLOADS[1].with_(heads=2, l_prompt=200_032)
    L = wl.l_prompt
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, L, dev)
    res = _compress(q, k, v.cpu().pin_memory() if v_on_host else v, wl)
    assert res["len"].cpu().tolist() == [wl.budget + wl.l_obs]
    _check_heads(res, wl, L, heads=range(wl.heads))


@pytest.mark.parametrize("v_on_host", [False, True])
def test_pool_kernel_beyond_cluster_reach(dev, v_on_host):
    """K_pool = 1027 > 1025 takes the single-CTA top-k too; wide plateaus of tied pooled values."""
    wl = synth.WORKLOADS[1].with_(heads=3, l_prompt=5000, pool_kernel=1027, budget=0, ratio_p=0.3)
    L = wl.l_prompt
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, L, dev)
    res = _compress(q, k, v.cpu().pin_memory() if v_on_host else v, wl)
    assert res["k"] == int(0.3 * (L - wl.l_obs))
    _check_heads(res, wl, L, heads=range(wl.heads))


def test_ragged_batch_values_on_host(dev):
    """One launch over a ragged batch with V on the host: the same bytes as with V on the device."""
    from kv_cache_compression_gb300 import snapkv
    lengths = [3000, 9000, 4097]
    wl = synth.WORKLOADS[1].with_(heads=4, plants=0)
    q, k, v = synth.device_inputs_padded(wl, 0, 0, lengths, dev)
    res = snapkv.compress_varlen(q, k, v.cpu().pin_memory(), lengths, pool_kernel=7, ratio_p=0.1)
    torch.cuda.synchronize()
    _assert_gathered(res, k, v, lengths, wl.l_obs)
    for b, L in enumerate(lengths):
        hi = synth.host_head(wl, 0, b, 1, l_prompt=L)
        ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=7, ratio_p=0.1)
        got = res["idx"][b, 1, :res["ks"][b]].cpu().numpy()
        diff = set(got.tolist()) ^ set(ref.idx.tolist())
        assert all(abs(ref.p[j] - ref.tau) <= 1e-5 * ref.tau for j in diff), (b, sorted(diff)[:8])


def test_grouped_query_values_on_host(dev):
    """Grouped-query compression (4 query heads per KV head) with V on the host."""
    from kv_cache_compression_gb300 import snapkv
    g = torch.Generator().manual_seed(5)
    q = torch.randn(1, 16, 32, 128, generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn(1, 4, 6000, 128, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(1, 4, 6000, 128, generator=g).to(torch.bfloat16)
    res = snapkv.compress(q, k, v.pin_memory(), pool_kernel=7, budget=512)
    torch.cuda.synchronize()
    _assert_gathered(res, k, v.to(dev), [6000], 32)
    for h in (0, 3):
        ref = orc.compress_kv_head_gqa(q[0, 4 * h:4 * h + 4].float().cpu().numpy(), k[0, h].float().cpu().numpy(),
                                       v[0, h].float().numpy(), pool_kernel=7, budget=512)
        got = res["idx"][0, h].cpu().numpy()
        diff = set(got.tolist()) ^ set(ref.idx.tolist())
        assert all(abs(ref.p[j] - ref.tau) <= 1e-5 * ref.tau for j in diff), (h, sorted(diff)[:8])


def test_pageable_values_are_refused(dev):
    """Pageable host memory is not mapped into the device: refused on the host, nothing written."""
    from kv_cache_compression_gb300 import snapkv
    g = torch.Generator().manual_seed(6)
    q = torch.randn(1, 2, 16, 64, generator=g).to(dev)
    k = torch.randn(1, 2, 1000, 64, generator=g).to(dev)
    v = torch.randn(1, 2, 1000, 64, generator=g)       # pageable
    assert not v.is_pinned()
    k_out = torch.full((1, 2, 116, 64), 7.0, device=dev)
    v_out = torch.full((1, 2, 116, 64), 7.0, device=dev)
    with pytest.raises(snapkv.SnapKVError) as e:
        snapkv.compress(q, k, v, pool_kernel=7, budget=100, k_out=k_out, v_out=v_out)
    assert e.value.status == snapkv.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool(torch.all(k_out == 7.0)) and bool(torch.all(v_out == 7.0))
