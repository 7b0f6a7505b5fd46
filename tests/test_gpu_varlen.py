"""GPU parity of snapkv_compress_varlen (one call over sequences of different prompt lengths, so
that under the ratio rule k = floor(p * L_prefix) differs per sequence) against the CPU oracle run
on each sequence alone, and of decoding on the resulting truly ragged cache."""
import numpy as np
import pytest
import torch

import synth
from oracle import snapkv_oracle as orc
from tests.parity import assert_canary, canary_like, check_compress_head, check_decode, to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(gpu_device):
    import __graft_entry__
    __graft_entry__.build()
    return gpu_device


def _check(res, wl, lengths, heads, *, ratio_p, budget, scope="prompt_causal"):
    B = len(lengths)
    l_obs = wl.l_obs
    assert res["len"].cpu().tolist() == [kb + l_obs for kb in res["ks"]]
    idx, vote = res["idx"].cpu().numpy(), res["vote"].cpu().numpy()
    excused = 0
    for b, L in enumerate(lengths):
        kb, lp = res["ks"][b], L - l_obs
        assert kb == orc.kept_slots(lp, ratio_p=ratio_p, budget=budget)
        # rows past this sequence's own k and L_prefix are left as they were
        assert (idx[b, :, kb:] == -1).all(), f"seq {b}: idx written past k_b"
        assert (vote[b, :, lp:] == 0).all(), f"seq {b}: vote written past L_prefix_b"
        for h in heads:
            hi = synth.host_head(wl, 0, b, h, l_prompt=L)
            ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, ratio_p=ratio_p,
                                    budget=budget, scope=scope)
            rep = check_compress_head(gpu_idx=idx[b, h, :kb], gpu_kc=to_numpy_f32(res["k_out"][b, h]),
                                      gpu_vc=to_numpy_f32(res["v_out"][b, h]), gpu_vote=vote[b, h, :lp], ref=ref,
                                      k_in=hi.k, v_in=hi.v, l_prefix=lp, l_obs=l_obs, where=f"seq {b} (L {L}) head {h}")
            excused += rep.excused
    return excused


@pytest.mark.parametrize("algo", ["auto", "tensor_core_cluster", "simt"])
def test_varlen_ratio_rule_bf16(dev, algo):
    """Llama-shaped heads, four prompts of different lengths (ragged tails, one short), p = 0.1."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1].with_(heads=6, plants=16)
    lengths = [4096, 2500, 5001, 417]
    q, k, v = synth.device_inputs_padded(wl, 0, 0, lengths, dev)
    k_max = orc.kept_slots(max(lengths) - wl.l_obs, ratio_p=0.1)
    cap = k_max + wl.l_obs + 2   # every sequence's rows past its own k_b + L_obs are a canary guard band
    k_out = canary_like((len(lengths), wl.heads, cap, wl.head_dim), torch.bfloat16, dev)
    v_out = canary_like((len(lengths), wl.heads, cap, wl.head_dim), torch.bfloat16, dev)
    res = snapkv.compress_varlen(q, k, v, lengths, pool_kernel=wl.pool_kernel, ratio_p=0.1, algo=algo,
                                 want_vote=True, k_out=k_out, v_out=v_out)
    torch.cuda.synchronize()
    assert len(set(res["ks"])) == len(lengths)               # truly ragged k
    for b, kb in enumerate(res["ks"]):
        assert_canary(k_out[b, :, kb + wl.l_obs:], f"seq {b}: k_out rows past k_b + L_obs")
        assert_canary(v_out[b, :, kb + wl.l_obs:], f"seq {b}: v_out rows past k_b + L_obs")
    _check(res, wl, lengths, range(wl.heads), ratio_p=0.1, budget=0)


def test_varlen_longest_prompt_past_one_chunk_per_cta(dev):
    """A ragged batch keeps every sequence's logits in TMEM; when its longest prompt has more key
    chunks than the grid has CTAs (one per SM), the vote of an item comes one item late and only two
    epilogue warpgroups take items. The short sequences share the queue with it."""
    from kv_cache_compression_gb300 import snapkv
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    wl = synth.WORKLOADS[1].with_(heads=2, plants=16)
    lengths = [sms * 512 + 2000, 3000, 77]
    assert (lengths[0] + 511) // 512 > sms   # 512 keys per item for a 32-row window
    q, k, v = synth.device_inputs_padded(wl, 0, 0, lengths, dev)
    res = snapkv.compress_varlen(q, k, v, lengths, pool_kernel=wl.pool_kernel, budget=1024, want_vote=True)
    torch.cuda.synchronize()
    _check(res, wl, lengths, range(wl.heads), ratio_p=0.0, budget=1024)


def test_varlen_tiny_fp32_prefix_only_and_padding_longer_than_any_prompt(dev):
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[0]
    lengths = [1024, 700, 333]
    q, k, v = synth.device_inputs_padded(wl, 0, 0, lengths, dev, l_pad=1100)
    res = snapkv.compress_varlen(q, k, v, lengths, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p,
                                 scope="prefix_only", want_vote=True)
    torch.cuda.synchronize()
    excused = _check(res, wl, lengths, range(wl.heads), ratio_p=wl.ratio_p, budget=0, scope="prefix_only")
    assert excused == 0


def test_varlen_budget_rule_with_prompts_shorter_than_budget(dev):
    """Under a budget, a prompt whose L_prefix is below it keeps its whole prefix (k = L_prefix)."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1].with_(heads=4, plants=16)
    lengths = [3000, 600, 1056, 2049]
    q, k, v = synth.device_inputs_padded(wl, 0, 0, lengths, dev)
    res = snapkv.compress_varlen(q, k, v, lengths, pool_kernel=wl.pool_kernel, budget=1024, want_vote=True)
    torch.cuda.synchronize()
    assert res["ks"] == [1024, 568, 1024, 1024]
    _check(res, wl, lengths, range(wl.heads), ratio_p=0.0, budget=1024)


def test_varlen_ratio_workload_then_ragged_decode(dev):
    """The ragged-prompt decode workload's first 8 sequences under p = 0.125 (so each sequence keeps a
    different number of rows), then 16 steps of append + attention on the ragged cache, each
    sequence's output checked against the oracle continuing from the GPU's kept set."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[4]
    B, steps, p = 8, 16, 0.125
    lengths = wl.prompt_lengths()[:B]
    q, k, v = synth.device_inputs_padded(wl, 0, 0, lengths, dev)
    k_max = orc.kept_slots(max(lengths) - wl.l_obs, ratio_p=p)
    cap = k_max + wl.l_obs + steps
    res = snapkv.compress_varlen(q, k, v, lengths, pool_kernel=wl.pool_kernel, ratio_p=p, cap=cap, want_vote=True)
    del q, k, v
    torch.cuda.synchronize()
    assert len(set(res["ks"])) == B
    heads = [0, 21]
    _check(res, wl, lengths, heads, ratio_p=p, budget=0)
    outs = []
    for t in range(steps):
        qn, kn, vn = synth.device_decode_tokens(wl, 0, t, 0, B, dev)
        snapkv.append(kn, vn, res["k_out"], res["v_out"], res["len"])
        outs.append(snapkv.decode_attend(qn, res["k_out"], res["v_out"], res["len"])[:, heads].cpu())
    torch.cuda.synchronize()
    assert res["len"].cpu().tolist() == [kb + wl.l_obs + steps for kb in res["ks"]]
    idx = res["idx"].cpu().numpy()
    for b, L in enumerate(lengths):
        for j, h in enumerate(heads):
            hi = synth.host_head(wl, 0, b, h, l_prompt=L)
            got = idx[b, h, :res["ks"][b]]
            kc = orc.gather_with_window(hi.k, got, L - wl.l_obs)
            vc = orc.gather_with_window(hi.v, got, L - wl.l_obs)
            for t in range(steps):
                qn, kn, vn = synth.host_decode_token(wl, 0, b, h, t)
                kc, vc = orc.append(kc, vc, kn, vn)
                check_decode(to_numpy_f32(outs[t][b, j]), orc.decode_attend(qn, kc, vc), True,
                             where=f"seq {b} head {h} step {t}")


def test_varlen_matches_separate_calls_bitwise(dev):
    """One varlen call gives the same bytes as one snapkv_compress call per sequence."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1].with_(heads=4, plants=16)
    lengths = [2200, 1300, 3100]
    q, k, v = synth.device_inputs_padded(wl, 0, 0, lengths, dev)
    res = snapkv.compress_varlen(q, k, v, lengths, pool_kernel=wl.pool_kernel, ratio_p=0.2, want_vote=True)
    for b, L in enumerate(lengths):
        one = snapkv.compress(q[b:b + 1].contiguous(), k[b:b + 1, :, :L].contiguous(), v[b:b + 1, :, :L].contiguous(),
                              pool_kernel=wl.pool_kernel, ratio_p=0.2, want_vote=True)
        kb = one["k"]
        assert kb == res["ks"][b]
        assert torch.equal(one["idx"][0], res["idx"][b, :, :kb])
        assert torch.equal(one["vote"][0], res["vote"][b, :, :L - wl.l_obs])
        assert torch.equal(one["k_out"][0, :, :kb + wl.l_obs], res["k_out"][b, :, :kb + wl.l_obs])
        assert torch.equal(one["v_out"][0, :, :kb + wl.l_obs], res["v_out"][b, :, :kb + wl.l_obs])


def test_varlen_with_a_sequence_that_keeps_nothing(dev):
    """p * L_prefix < 1 for one short prompt: that sequence keeps only its window (k = 0), the others
    keep their own k (the batch then takes one compression per sequence)."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1].with_(heads=3, plants=16)
    lengths = [3000, 50, 1500]
    q, k, v = synth.device_inputs_padded(wl, 0, 0, lengths, dev)
    res = snapkv.compress_varlen(q, k, v, lengths, pool_kernel=wl.pool_kernel, ratio_p=0.05, want_vote=True)
    torch.cuda.synchronize()
    assert res["ks"][1] == 0
    _check(res, wl, lengths, range(wl.heads), ratio_p=0.05, budget=0)
