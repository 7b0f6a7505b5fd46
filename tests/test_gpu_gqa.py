"""GPU parity of snapkv_compress_gqa (grouped-query attention: G query heads share a KV head) against
the CPU oracle, through the C ABI, on every vote path."""
import numpy as np
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


CASES = [  # (G, L_obs, KV heads, L_prompt, pool, budget)
    (2, 32, 4, 4096, 7, 300),
    (4, 32, 2, 3000, 7, 256),    # 128 window rows per KV head
    (4, 16, 3, 5000, 5, 400),
    (8, 8, 2, 2100, 3, 100),
]


@pytest.mark.parametrize("algo", ["auto", "tensor_core_cluster", "simt"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"G{c[0]}-obs{c[1]}-Hkv{c[2]}-L{c[3]}")
def test_gqa_matches_oracle(dev, case, algo):
    from kv_cache_compression_gb300 import snapkv
    G, l_obs, hkv, L, pool, budget = case
    hq = G * hkv
    wl = synth.WORKLOADS[1].with_(heads=hq, l_prompt=L, l_obs=l_obs, plants=16)
    q, k_all, v_all, _ = synth.device_inputs(wl, 0, 0, 1, L, dev)
    k = k_all[:, :hkv].contiguous()       # KV head h uses the keys and values of generated head h
    v = v_all[:, :hkv].contiguous()
    res = snapkv.compress(q, k, v, pool_kernel=pool, budget=budget, algo=algo, want_vote=True)
    torch.cuda.synchronize()
    assert res["len"].cpu().tolist() == [res["k"] + l_obs]
    for h in range(hkv):
        kv = synth.host_head(wl, 0, 0, h, l_prompt=L)
        qg = np.stack([synth.host_head(wl, 0, 0, h * G + g, l_prompt=L).q_obs for g in range(G)])
        ref = orc.compress_kv_head_gqa(qg, kv.k, kv.v, pool_kernel=pool, budget=budget)
        check_compress_head(gpu_idx=res["idx"][0, h].cpu().numpy(), gpu_kc=to_numpy_f32(res["k_out"][0, h]),
                            gpu_vc=to_numpy_f32(res["v_out"][0, h]), gpu_vote=res["vote"][0, h].cpu().numpy(),
                            ref=ref, k_in=kv.k, v_in=kv.v, l_prefix=L - l_obs, l_obs=l_obs,
                            where=f"G{G} kv head {h}")
