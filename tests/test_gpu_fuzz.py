"""Seeded random shapes through the C ABI against the CPU oracle: compress (every vote path, both
softmax scopes, ratio and budget rules), ragged batches, and decode on ragged caches. The shapes are
drawn once from a fixed seed, so every run checks the same cases."""
import numpy as np
import pytest
import torch

import synth
from oracle import snapkv_oracle as orc
from tests.parity import check_compress_head, check_decode, to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(gpu_device):
    import __graft_entry__
    __graft_entry__.build()
    return gpu_device


def _compress_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        bf16 = bool(rng.integers(0, 4) > 0)             # mostly bf16 (the tensor-core paths)
        d = int(rng.choice([64, 128]))
        l_obs = int(rng.choice([1, 3, 8, 16, 17, 32, 48, 64, 100]))
        L = int(rng.integers(l_obs + 2, 6000))
        pool = int(rng.choice([1, 3, 5, 7, 9, 13, 31]))
        if rng.integers(0, 2):
            p, budget = float(rng.choice([0.01, 0.05, 0.2, 0.5, 1.0])), 0
        else:
            p, budget = 0.0, int(rng.integers(1, L))
        scope = "prompt_causal" if rng.integers(0, 3) else "prefix_only"
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        cases.append((i, bf16, d, l_obs, L, pool, p, budget, scope, B, H))
    return cases


@pytest.mark.parametrize("case", _compress_cases(32, 20261202), ids=lambda c: f"fuzz{c[0]}")
def test_fuzz_compress(dev, case):
    from kv_cache_compression_gb300 import snapkv
    i, bf16, d, l_obs, L, pool, p, budget, scope, B, H = case
    wl = synth.Workload(f"fuzz {i}", 100 + i, bf16=bf16, batch=B, heads=H, head_dim=d, layers=1, l_prompt=L,
                        l_obs=l_obs, pool_kernel=pool, ratio_p=p, budget=budget)
    q, k, v, _ = synth.device_inputs(wl, 0, 0, B, L, dev)
    algos = ["auto", "simt"] + (["tensor_core_cluster"] if bf16 and l_obs <= 64 else [])
    l_prefix = L - l_obs
    for algo in algos:
        try:
            res = snapkv.compress(q, k, v, pool_kernel=pool, ratio_p=p, budget=budget, scope=scope, algo=algo,
                                  want_vote=True)
        except snapkv.SnapKVError as e:
            # the cluster kernel takes only heads whose keys fit its CTAs' TMEM; refused, not wrong
            assert algo == "tensor_core_cluster" and e.status == snapkv.ERR_UNSUPPORTED
            continue
        torch.cuda.synchronize()
        for b in range(B):
            for h in range(H):
                hi = synth.host_head(wl, 0, b, h, l_prompt=L)
                ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=pool, ratio_p=p, budget=budget, scope=scope)
                check_compress_head(gpu_idx=res["idx"][b, h].cpu().numpy()[:res["k"]],
                                    gpu_kc=to_numpy_f32(res["k_out"][b, h]), gpu_vc=to_numpy_f32(res["v_out"][b, h]),
                                    gpu_vote=res["vote"][b, h].cpu().numpy(), ref=ref, k_in=hi.k, v_in=hi.v,
                                    l_prefix=l_prefix, l_obs=l_obs, where=f"fuzz {i} {algo} b{b} h{h}")


def _long_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        l_obs = int(rng.choice([5, 16, 24, 32, 40, 64, 65, 100]))
        L = int(rng.integers(20000, 90000))
        pool = int(rng.choice([1, 5, 7, 13, 31]))
        if rng.integers(0, 2):
            p, budget = float(rng.choice([0.01, 0.05, 0.2])), 0
        else:
            p, budget = 0.0, int(rng.integers(1, 8192))
        cases.append((i, l_obs, L, pool, p, budget))
    return cases


@pytest.mark.parametrize("case", _long_cases(8, 777001), ids=lambda c: f"long{c[0]}")
def test_fuzz_long_prompts(dev, case):
    """Long random prompts on the default path, so that heads of more items than the grid has CTAs
    take the vote kernel's late-vote or key re-read modes, and prefixes beyond one CTA take clusters in
    the top-k kernel."""
    from kv_cache_compression_gb300 import snapkv
    i, l_obs, L, pool, p, budget = case
    wl = synth.Workload(f"long fuzz {i}", 900 + i, bf16=True, batch=1, heads=2, head_dim=128, layers=1,
                        l_prompt=L, l_obs=l_obs, pool_kernel=pool, ratio_p=p, budget=budget)
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, L, dev)
    res = snapkv.compress(q, k, v, pool_kernel=pool, ratio_p=p, budget=budget, want_vote=True)
    torch.cuda.synchronize()
    for h in range(2):
        hi = synth.host_head(wl, 0, 0, h, l_prompt=L)
        ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=pool, ratio_p=p, budget=budget)
        check_compress_head(gpu_idx=res["idx"][0, h].cpu().numpy()[:res["k"]], gpu_kc=to_numpy_f32(res["k_out"][0, h]),
                            gpu_vc=to_numpy_f32(res["v_out"][0, h]), gpu_vote=res["vote"][0, h].cpu().numpy(),
                            ref=ref, k_in=hi.k, v_in=hi.v, l_prefix=L - l_obs, l_obs=l_obs, where=f"long fuzz {i} h{h}")


@pytest.mark.parametrize("seed", [1, 2, 3, 8, 9])
def test_fuzz_varlen(dev, seed):
    from kv_cache_compression_gb300 import snapkv
    rng = np.random.default_rng(1000 + seed)
    l_obs = int(rng.choice([8, 16, 32]))
    B = int(rng.integers(2, 7))
    lengths = [int(x) for x in rng.integers(l_obs + 40, 5000, size=B)]
    p = float(rng.choice([0.05, 0.1, 0.3]))
    wl = synth.WORKLOADS[1].with_(heads=2, l_obs=l_obs, plants=0)
    q, k, v = synth.device_inputs_padded(wl, 0, 0, lengths, dev)
    res = snapkv.compress_varlen(q, k, v, lengths, pool_kernel=7, ratio_p=p, want_vote=True)
    torch.cuda.synchronize()
    assert res["len"].cpu().tolist() == [kb + l_obs for kb in res["ks"]]
    idx, vote = res["idx"].cpu().numpy(), res["vote"].cpu().numpy()
    for b, L in enumerate(lengths):
        kb, lp = res["ks"][b], L - l_obs
        for h in range(wl.heads):
            hi = synth.host_head(wl, 0, b, h, l_prompt=L)
            ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=7, ratio_p=p)
            check_compress_head(gpu_idx=idx[b, h, :kb], gpu_kc=to_numpy_f32(res["k_out"][b, h]),
                                gpu_vc=to_numpy_f32(res["v_out"][b, h]), gpu_vote=vote[b, h, :lp], ref=ref,
                                k_in=hi.k, v_in=hi.v, l_prefix=lp, l_obs=l_obs, where=f"varlen seed {seed} b{b} h{h}")


@pytest.mark.parametrize("seed", [4, 5, 6, 7, 10, 11])
def test_fuzz_decode(dev, seed):
    from kv_cache_compression_gb300 import snapkv
    rng = np.random.default_rng(2000 + seed)
    d = int(rng.choice([64, 128]))
    dtype = torch.bfloat16 if rng.integers(0, 3) else torch.float32
    B, H = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    cap = int(rng.integers(1, 40000))
    lens = [int(x) for x in rng.integers(0, cap + 1, size=B)]
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn(B, H, cap, d, generator=g).to(dtype)
    vc = torch.randn(B, H, cap, d, generator=g).to(dtype)
    q = (torch.randn(B, H, d, generator=g) * 1.5).to(dtype)
    out = snapkv.decode_attend(q.to(dev), kc.to(dev), vc.to(dev), torch.tensor(lens, dtype=torch.int32).to(dev))
    torch.cuda.synchronize()
    o = to_numpy_f32(out)
    for b in range(B):
        for h in range(H):
            n = lens[b]
            if n == 0:
                assert np.all(o[b, h] == 0.0)
                continue
            ref = orc.decode_attend(q[b, h].float().numpy(), kc[b, h, :n].float().numpy(), vc[b, h, :n].float().numpy())
            check_decode(o[b, h], ref, dtype == torch.bfloat16, where=f"seed {seed} b{b} h{h} n{n} cap {cap}")
    # one decode step as the fused call and as append + decode: the same bytes
    kn = torch.randn(B, H, d, generator=g).to(dtype).to(dev)
    vn = torch.randn(B, H, d, generator=g).to(dtype).to(dev)
    qd, length = q.to(dev), torch.tensor(lens, dtype=torch.int32).to(dev)
    k1, v1, len1 = kc.to(dev), vc.to(dev), length.clone()
    snapkv.append(kn, vn, k1, v1, len1)
    out1 = snapkv.decode_attend(qd, k1, v1, len1)
    k2, v2 = kc.to(dev), vc.to(dev)
    out2, len2 = snapkv.append_decode_attend(qd, kn, vn, k2, v2, length)
    torch.cuda.synchronize()
    assert torch.equal(len2, len1) and torch.equal(k2, k1) and torch.equal(v2, v1) and torch.equal(out2, out1)
