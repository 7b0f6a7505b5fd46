"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every wait inside the streaming score/vote kernel (the key-tile ring, the TMEM slots, a vote item's
wait for the rest of its head) gives up after a limit of SM cycles, reports SNAPKV_ERR_TIMEOUT in the
device status word, drains the copies and tensor-core operations it started, frees its TMEM and
returns, so that the context stays usable. The limit is about two seconds; the host reads a shorter
one from SNAPKV_WAIT_LIMIT_CYCLES, which only tests set. Here it is set so short that the first waits
for key tiles run out: the call must report the timeout, and the next call on the same stream,
workspace and outputs (limit back to the default) must match the oracle exactly.
"""
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


def test_vote_wait_that_runs_out_reports_timeout_and_the_context_stays_usable(dev, monkeypatch):
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1].with_(heads=4, l_prompt=4096, budget=256, plants=16)
    L = wl.l_prompt
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, L, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    monkeypatch.setenv("SNAPKV_WAIT_LIMIT_CYCLES", "64")
    res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, budget=wl.budget, algo="tensor_core",
                          want_vote=True, dev_status=status, stream=stream)
    torch.cuda.synchronize(dev)
    assert int(status.item()) & snapkv.ERR_TIMEOUT, snapkv.status_string(int(status.item()))

    monkeypatch.delenv("SNAPKV_WAIT_LIMIT_CYCLES")
    status.zero_()
    again = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, budget=wl.budget, algo="tensor_core",
                            k_out=res["k_out"], v_out=res["v_out"], len_out=res["len"], idx_out=res["idx"],
                            vote_out=res["vote"], workspace=res["workspace"], dev_status=status, stream=stream)
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0, snapkv.status_string(int(status.item()))
    assert again["len"].cpu().tolist() == [wl.budget + wl.l_obs]
    for h in range(wl.heads):
        hi = synth.host_head(wl, 0, 0, h)
        ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, budget=wl.budget)
        check_compress_head(gpu_idx=again["idx"][0, h].cpu().numpy(), gpu_kc=to_numpy_f32(again["k_out"][0, h]),
                            gpu_vc=to_numpy_f32(again["v_out"][0, h]), gpu_vote=again["vote"][0, h].cpu().numpy(),
                            ref=ref, k_in=hi.k, v_in=hi.v, l_prefix=L - wl.l_obs, l_obs=wl.l_obs, where=f"head {h}")
    assert np.isfinite(again["vote"].cpu().numpy()).all()
