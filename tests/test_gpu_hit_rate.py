"""GPU parity of snapkv_hit_rate (the explainer's Hit Rate diagnostic) against the CPU oracle."""
import numpy as np
import pytest
import torch

import synth
from oracle import snapkv_oracle as orc
from tests.parity import to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(gpu_device):
    import __graft_entry__
    __graft_entry__.build()
    return gpu_device


def _setup(dev, wl, L):
    """Compress the prompt, then build the uncompressed cache (prompt + one decode token)."""
    from kv_cache_compression_gb300 import snapkv
    q, k, v, _ = synth.device_inputs(wl, 0, 0, wl.batch, L, dev)
    res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p, budget=wl.budget)
    qn, kn, _ = synth.device_decode_tokens(wl, 0, 0, 0, wl.batch, dev)
    cache = torch.cat([k, kn[:, :, None, :]], dim=2).contiguous()
    length = torch.full((wl.batch,), L + 1, dtype=torch.int32, device=dev)
    return res, qn, cache, length


@pytest.mark.parametrize("theta", [0.05, 0.01, 0.0])
def test_hit_rate_matches_oracle(dev, theta):
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1].with_(heads=6, l_prompt=4096)
    L = wl.l_prompt
    l_prefix = L - wl.l_obs
    res, qn, cache, length = _setup(dev, wl, L)
    hits, total = snapkv.hit_rate(qn, cache, length, res["idx"], l_prefix, theta=theta)
    torch.cuda.synchronize()
    hits, total = hits.cpu().numpy(), total.cpu().numpy()
    for h in range(wl.heads):
        ref = orc.hit_count(to_numpy_f32(qn[0, h]), to_numpy_f32(cache[0, h]), l_prefix,
                            res["idx"][0, h].cpu().numpy(), theta=theta)
        if theta == 0.0:
            assert (int(total[0, h]), int(hits[0, h])) == (l_prefix, res["k"])
            continue
        # positions whose weight lies within 1e-4 relative of theta may fall on either side in fp32
        band = int(np.sum(np.abs(ref.weights - theta) <= 1e-4 * theta))
        assert abs(int(total[0, h]) - ref.total) <= band, (h, total[0, h], ref.total)
        assert abs(int(hits[0, h]) - ref.hits) <= band, (h, hits[0, h], ref.hits)


def test_hit_rate_whole_prefix_kept_and_ragged_lengths(dev):
    """Every prefix position kept: hits == total. A sequence whose cache holds fewer rows than the
    prefix counts only the rows it holds."""
    from kv_cache_compression_gb300 import snapkv
    g = torch.Generator().manual_seed(7)
    B, H, d, cap, l_prefix = 2, 3, 64, 300, 250
    cache = (torch.randn(B, H, cap, d, generator=g) * 2).to(torch.bfloat16).to(dev)
    q = torch.randn(B, H, d, generator=g).to(torch.bfloat16).to(dev)
    idx = torch.arange(l_prefix, dtype=torch.int32).repeat(B, H, 1).contiguous().to(dev)
    length = torch.tensor([300, 120], dtype=torch.int32).to(dev)
    hits, total = snapkv.hit_rate(q, cache, length, idx, l_prefix, theta=0.01)
    torch.cuda.synchronize()
    assert torch.equal(hits, total)
    for b, n in [(0, 300), (1, 120)]:
        for h in range(H):
            ref = orc.hit_count(to_numpy_f32(q[b, h]), to_numpy_f32(cache[b, h, :n]), min(l_prefix, n),
                                np.arange(min(l_prefix, n)), theta=0.01)
            band = int(np.sum(np.abs(ref.weights - 0.01) <= 1e-4 * 0.01))
            assert abs(int(total[b, h]) - ref.total) <= band


def test_hit_rate_threshold_splits_the_prefix(dev):
    """A decode query aimed at six prefix keys, three that the oracle keeps and three it drops: it is
    the least-squares solution of q . k_j = 11 sqrt(d) over those keys, so each takes a weight well
    above theta = 0.05 and nothing else comes near it. Both sides then count 0 < hits < total on every
    head (three of six), the GPU's counts equal to the oracle's. The kept set passed to both is the
    oracle's own selection."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1].with_(heads=6, l_prompt=4096)
    L, d = wl.l_prompt, wl.head_dim
    lp = L - wl.l_obs
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, L, dev)
    rng = np.random.default_rng(11)
    qdec = np.zeros((1, wl.heads, d), dtype=np.float32)
    idx_ref, k_host = [], []
    for h in range(wl.heads):
        hi = synth.host_head(wl, 0, 0, h, l_prompt=L)
        ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, budget=wl.budget)
        dropped = np.setdiff1d(np.arange(lp), ref.idx)
        targets = np.concatenate([rng.choice(ref.idx, 3, replace=False), rng.choice(dropped, 3, replace=False)])
        kt = hi.k[targets].astype(np.float64)
        qdec[0, h] = kt.T @ np.linalg.solve(kt @ kt.T, np.full(6, 11.0 * np.sqrt(d)))
        idx_ref.append(ref.idx.astype(np.int32))
        k_host.append(hi.k)
    qd = torch.from_numpy(qdec).to(torch.bfloat16).to(dev)
    idx = torch.from_numpy(np.stack(idx_ref)[None]).contiguous().to(dev)
    length = torch.full((1,), L, dtype=torch.int32, device=dev)
    hits, total = snapkv.hit_rate(qd, k, length, idx, lp, theta=0.05)
    torch.cuda.synchronize()
    hits, total = hits.cpu().numpy(), total.cpu().numpy()
    qv = to_numpy_f32(qd)
    for h in range(wl.heads):
        ref = orc.hit_count(qv[0, h], k_host[h], lp, idx_ref[h], theta=0.05)
        assert 0 < ref.hits < ref.total, (h, ref.hits, ref.total)
        band = int(np.sum(np.abs(ref.weights - 0.05) <= 1e-4 * 0.05))
        assert band == 0, f"head {h}: a weight sits at the threshold"
        assert (int(hits[0, h]), int(total[0, h])) == (ref.hits, ref.total), (h, hits[0, h], total[0, h])
