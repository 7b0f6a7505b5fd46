"""GPU parity of snapkv_compress against the CPU oracle, through the C ABI.

Inputs are generated on the device by the seeded generator and regenerated bit-identically on
the host for the oracle. Every workload of the benchmark suite is covered: the tiny fp32 case and
the Llama-2-7B-shaped layer on every head, the long-context case, the 32-layer batch-8 prefill and
the ragged-prompt decode workload on seeded samples, plus edge cases (k = 0, k = L_prefix, L_obs = 1,
odd tails, both softmax scopes, several batches, exact ties).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import snapkv_oracle as orc
from tests import oracle_pool
from tests.conftest import golden
from tests.parity import assert_canary, bf16_bits, canary_like, check_compress_head, to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(gpu_device):
    import __graft_entry__
    __graft_entry__.build()
    return gpu_device


def _run_workload(dev, wl, layer=0, seq0=0, nseq=None, l_prompt=None, heads=None, scope="prompt_causal",
                  algo="auto"):
    from kv_cache_compression_gb300 import snapkv
    nseq = nseq if nseq is not None else wl.batch
    L = l_prompt if l_prompt is not None else wl.prompt_lengths()[seq0]
    q, k, v, _ = synth.device_inputs(wl, layer, seq0, nseq, L, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    l_prefix = L - wl.l_obs
    ksel = orc.kept_slots(l_prefix, ratio_p=wl.ratio_p, budget=wl.budget)
    R = ksel + wl.l_obs
    cap = R + 3   # rows past k + L_obs are a canary guard band the call must leave untouched
    k_out = canary_like((nseq, wl.heads, cap, wl.head_dim), k.dtype, dev)
    v_out = canary_like((nseq, wl.heads, cap, wl.head_dim), k.dtype, dev)
    res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p, budget=wl.budget, scope=scope,
                          algo=algo, want_vote=True, dev_status=status, cap=cap, k_out=k_out, v_out=v_out)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert res["k"] == ksel
    assert res["len"].cpu().tolist() == [ksel + wl.l_obs] * nseq
    assert_canary(k_out[:, :, R:], "k_out rows past k + L_obs")
    assert_canary(v_out[:, :, R:], "v_out rows past k + L_obs")
    excused = 0
    for b in range(nseq):
        for h in (heads if heads is not None else range(wl.heads)):
            hi = synth.host_head(wl, layer, seq0 + b, h, l_prompt=L)
            ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p,
                                    budget=wl.budget, scope=scope)
            rep = check_compress_head(gpu_idx=res["idx"][b, h].cpu().numpy(),
                                      gpu_kc=to_numpy_f32(res["k_out"][b, h]), gpu_vc=to_numpy_f32(res["v_out"][b, h]),
                                      gpu_vote=res["vote"][b, h].cpu().numpy(), ref=ref, k_in=hi.k, v_in=hi.v,
                                      l_prefix=l_prefix, l_obs=wl.l_obs, where=f"layer {layer} seq {seq0 + b} head {h}")
            excused += rep.excused
    return res, excused


def test_tiny_fp32_every_head(dev):
    _, excused = _run_workload(dev, synth.WORKLOADS[0])
    assert excused == 0


def test_tiny_fp32_prefix_only_scope(dev):
    _run_workload(dev, synth.WORKLOADS[0], scope="prefix_only")


@pytest.mark.parametrize("algo", ["tensor_core", "tensor_core_cluster", "simt"])
def test_llama_layer_every_head(dev, algo):
    _, excused = _run_workload(dev, synth.WORKLOADS[1], algo=algo)
    print(f"boundary-excused indices ({algo}): {excused}")


def _compress_jobs(wl, res, layer, seq0, units, L, scope="prompt_causal"):
    """Oracle-pool jobs for the (sequence offset b, head h) units of one compression result."""
    idx, vote = res["idx"].cpu().numpy(), res["vote"].cpu().numpy()
    R = res["k"] + wl.l_obs
    kc, vc = bf16_bits(res["k_out"][:, :, :R]), bf16_bits(res["v_out"][:, :, :R])
    return [dict(wl=wl, layer=layer, seq=seq0 + b, head=h, l_prompt=L, scope=scope, idx=idx[b, h], kc_bits=kc[b, h],
                 vc_bits=vc[b, h], vote=vote[b, h], where=f"layer {layer} seq {seq0 + b} head {h}") for b, h in units]


def _pool_verdict(results):
    errors = [f"{w}: {e}" for w, _, e in results if e is not None]
    assert not errors, "\n".join(errors[:5]) + (f"\n... {len(errors)} heads failed" if len(errors) > 5 else "")
    return sum(r for _, r, _ in results)


def test_long_context_every_head(dev):
    """The long-context workload (131072 keys, L_obs 64, K_pool 13, budget 4096) on every head, in the
    launch configuration of the default (streaming tensor-core) path."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[3]
    L = wl.l_prompt
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, L, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, budget=wl.budget, want_vote=True, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    jobs = _compress_jobs(wl, res, 0, 0, [(0, h) for h in range(wl.heads)], L)
    del q, k, v
    excused = _pool_verdict(oracle_pool.run(oracle_pool.check_compress_job, jobs))
    print(f"long context: {len(jobs)} heads, {excused} boundary-excused indices")


@pytest.mark.parametrize("l_obs,grids,tail", [(100, 2, 333), (100, 4, 777), (64, 1, 999), (32, 4, 777)])
def test_long_heads_in_every_queue_mode(dev, l_obs, grids, tail):
    """Heads with more key chunks than the grid has CTAs (one per SM) cannot take the vote right
    after their own statistics. A window padded to 128 rows (two epilogue warpgroups) keeps the
    logits in TMEM and votes one item late while a head has at most four chunks per CTA (grids = 2),
    and past that alternates statistics and vote items that read the keys again from L2 (grids = 4).
    Windows of up to 64 rows (three warpgroups) take the re-read mode as soon as a head has more
    chunks than CTAs (grids = 1 and 4). Every prompt ends in a ragged tail."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    n_pad = 128 if l_obs > 64 else (64 if l_obs > 32 else 32)
    keys_per_item = (128 // n_pad) * 128
    L = grids * sms * keys_per_item + tail
    n_chunk = (L + keys_per_item - 1) // keys_per_item
    assert grids * sms < n_chunk <= grids * sms + 8
    wl = synth.WORKLOADS[1].with_(heads=2, l_obs=l_obs, l_prompt=L)
    _run_workload(dev, wl, l_prompt=L, algo="tensor_core")


_PRESETS = [(pre["name"], pre["l_obs"], pre["pool_kernel"], budget)
            for pre in golden("snapkv_presets.json")["presets"] for budget in sorted(set(pre["max_kept"]))]


@pytest.mark.parametrize("name,l_obs,pool,budget", _PRESETS, ids=lambda x: str(x))
def test_explainer_presets_on_the_tensor_core_path(dev, name, l_obs, pool, budget):
    """The hyper-parameter presets of the explainer's implementation section (observation window,
    pooling kernel, kept budget) on the default tensor-core path, every head of B2 H4 with a
    9000-key prompt (a ragged last tile): windows of 16, 32 and 64 rows, kernels of 5, 7 and 13."""
    wl = synth.WORKLOADS[1].with_(batch=2, heads=4, l_obs=l_obs, pool_kernel=pool, budget=budget, l_prompt=9000,
                                  plants=16)
    _run_workload(dev, wl, l_prompt=9000, algo="tensor_core")


def test_long_context_sampled_heads_simt(dev):
    _run_workload(dev, synth.WORKLOADS[3], heads=[0, 13, 31], algo="simt")


def test_llama_layer_prefix_only_tensor_core(dev):
    _run_workload(dev, synth.WORKLOADS[1].with_(heads=8), scope="prefix_only", algo="tensor_core")


def prefill_parity_units(seed=0xC2):
    """The 32-layer prefill's parity coverage: every (sequence, head) of layers 0 and 31, plus 64 seeded
    (layer, sequence, head) units drawn from all 32 layers; layer -> sorted (sequence, head) list."""
    rng = np.random.default_rng(seed)
    units = {0: {(b, h) for b in range(8) for h in range(32)}, 31: {(b, h) for b in range(8) for h in range(32)}}
    for u in rng.choice(32 * 8 * 32, size=64, replace=False):
        layer, b, h = int(u // 256), int((u // 32) % 8), int(u % 32)
        units.setdefault(layer, set()).add((b, h))
    return {layer: sorted(bh) for layer, bh in sorted(units.items())}


def test_prefill_32_layers_parity_coverage(dev):
    """The 32-layer batch-8 prefill in the benchmark's launch configuration (one call per layer over
    B8 x 32 heads, p = 0.05, K with per-channel scales): every head of layers 0 and 31 and 64 seeded
    units from the other layers against the oracle, and the cache rows past k + L_obs untouched."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[2]
    L, B, H = wl.l_prompt, wl.batch, wl.heads
    ksel = orc.kept_slots(L - wl.l_obs, ratio_p=wl.ratio_p)
    R = ksel + wl.l_obs
    cap = R + 1
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    jobs = []
    units = prefill_parity_units()
    assert sum(len(u) for u in units.values()) >= 512 + 60
    for layer, bhs in units.items():
        q, k, v, _ = synth.device_inputs(wl, layer, 0, B, L, dev)
        k_out = canary_like((B, H, cap, wl.head_dim), k.dtype, dev)
        v_out = canary_like((B, H, cap, wl.head_dim), k.dtype, dev)
        res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p, cap=cap, k_out=k_out,
                              v_out=v_out, want_vote=True, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and res["k"] == ksel
        assert res["len"].cpu().tolist() == [R] * B
        assert_canary(k_out[:, :, R:], f"layer {layer}: k_out row R")
        assert_canary(v_out[:, :, R:], f"layer {layer}: v_out row R")
        jobs += _compress_jobs(wl, res, layer, 0, bhs, L)
        del q, k, v, res
    excused = _pool_verdict(oracle_pool.run(oracle_pool.check_compress_job, jobs))
    print(f"32-layer prefill: {len(jobs)} heads over {len(units)} layers, {excused} boundary-excused indices")


@pytest.mark.parametrize("batch,l_prompt,budget", [(16, 4096, 0), (4, 8192, 0), (2, 12000, 0), (10, 12000, 6000),
                                                   (4, 16384, 12000), (12, 3000, 2968)])
def test_large_batch_top_k_shapes(dev, batch, l_prompt, budget):
    """Batches that put the pooled top-k on one CTA per head (its own kernel, the boundary bin's values
    in a candidate list), on clusters of two and four CTAs, and kept lists longer than the shared-memory
    list a CTA holds (6000 kept rows on one CTA, about 6000 per CTA of a 2-CTA cluster), so that the
    gather reads the kept positions back from the index output; and a batch keeping its whole prefix;
    every head against the oracle."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[2].with_(batch=batch, l_prompt=l_prompt, layers=1, budget=budget)
    q, k, v, _ = synth.device_inputs(wl, 5, 0, batch, l_prompt, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p, budget=budget, want_vote=True,
                          dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    jobs = _compress_jobs(wl, res, 5, 0, [(b, h) for b in range(batch) for h in range(wl.heads)], l_prompt)
    del q, k, v
    _pool_verdict(oracle_pool.run(oracle_pool.check_compress_job, jobs))


def test_zero_queries_keep_the_first_k_at_large_batch(dev):
    """q = 0 on a batch of 320 heads (one CTA per head): every pooled score is equal, the first digit's
    bin holds the whole prefix (too many values for the candidate list), and ties go to the lower
    index, so I = 0..k-1 exactly; likewise when k is larger than the CTA's shared-memory kept list."""
    from kv_cache_compression_gb300 import snapkv
    B, H, L, lo, d = 10, 32, 8000, 32, 128
    k = torch.randn(B, H, L, d, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).to(dev)
    q = torch.zeros(B, H, lo, d, dtype=torch.bfloat16, device=dev)
    for budget in (300, 5000):
        res = snapkv.compress(q, k, k, pool_kernel=7, budget=budget)
        torch.cuda.synchronize()
        want = torch.arange(budget, dtype=torch.int32, device=dev).expand(B, H, budget)
        assert torch.equal(res["idx"], want)
        assert torch.equal(res["k_out"][:, :, :budget], k[:, :, :budget])
        assert torch.equal(res["k_out"][:, :, budget:], k[:, :, L - lo:])


def test_ragged_prompts_sampled(dev):
    wl = synth.WORKLOADS[4]
    lens = wl.prompt_lengths()
    for seq in (int(np.argmin(lens)), int(np.argmax(lens)), 17):
        _run_workload(dev, wl, layer=seq % 32, seq0=seq, nseq=1, heads=[0, 31])


EDGE_CASES = [
    # (bf16, d, l_obs, pool, l_prompt, ratio_p, budget, scope, batch, heads)
    (False, 64, 1, 1, 37, 0.5, 0, "prompt_causal", 1, 1),
    (True, 128, 16, 5, 1000, 0.0, 100, "prefix_only", 1, 2),
    (True, 64, 64, 13, 3001, 0.05, 0, "prompt_causal", 1, 3),
    (True, 128, 128, 3, 2049, 1.0, 0, "prompt_causal", 1, 2),
    (False, 128, 32, 7, 1025, 0.0, 0, "prompt_causal", 2, 2),
    (True, 128, 8, 9, 65, 0.0, 10000, "prompt_causal", 1, 1),
    (True, 128, 32, 7, 777, 0.2, 0, "prompt_causal", 3, 5),
    (False, 64, 48, 15, 4099, 0.03, 0, "prefix_only", 2, 2),
]


@pytest.mark.parametrize("algo", ["auto", "tensor_core_cluster", "simt"])
@pytest.mark.parametrize("case", EDGE_CASES, ids=lambda c: f"bf16={c[0]}-d{c[1]}-obs{c[2]}-K{c[3]}-L{c[4]}")
def test_edge_cases(dev, case, algo):
    bf16, d, l_obs, pool, L, p, budget, scope, B, H = case
    if algo == "tensor_core_cluster" and (not bf16 or l_obs > 64):
        pytest.skip("the cluster tensor-core kernel takes bf16 with L_obs <= 64")
    wl = synth.Workload("edge", 40 + L % 17, bf16=bf16, batch=B, heads=H, head_dim=d, layers=1, l_prompt=L,
                        l_obs=l_obs, pool_kernel=pool, ratio_p=p, budget=budget)
    _run_workload(dev, wl, scope=scope, algo=algo)


def test_tensor_core_path_is_refused_when_ineligible(dev):
    from kv_cache_compression_gb300 import snapkv
    q = torch.zeros(1, 1, 32, 64, device=dev)
    k = torch.zeros(1, 1, 256, 64, device=dev)
    with pytest.raises(snapkv.SnapKVError) as e:
        snapkv.compress(q, k, k.clone(), pool_kernel=7, budget=10, algo="tensor_core")   # fp32 input
    assert e.value.status == snapkv.ERR_UNSUPPORTED


@pytest.mark.parametrize("algo", ["tensor_core", "tensor_core_cluster", "simt"])
def test_zero_queries_keep_the_first_k(dev, algo):
    """q = 0 makes every pooled score equal; ties go to the lower index, so I = 0..k-1 exactly."""
    from kv_cache_compression_gb300 import snapkv
    B, H, L, lo, d = 1, 3, 3000, 32, 128
    k = torch.randn(B, H, L, d, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16).to(dev)
    q = torch.zeros(B, H, lo, d, dtype=torch.bfloat16, device=dev)
    res = snapkv.compress(q, k, k.clone(), pool_kernel=7, budget=300, algo=algo)
    torch.cuda.synchronize()
    for h in range(H):
        assert res["idx"][0, h].cpu().tolist() == list(range(300))


@pytest.mark.parametrize("algo", ["auto", "tensor_core_cluster"])
def test_workspace_is_reusable(dev, algo):
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1].with_(heads=4, l_prompt=4096)
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, wl.l_prompt, dev)
    first = snapkv.compress(q, k, v, pool_kernel=7, budget=wl.budget, algo=algo, want_vote=True)
    again = snapkv.compress(q, k, v, pool_kernel=7, budget=wl.budget, algo=algo, want_vote=True,
                            workspace=first["workspace"])
    torch.cuda.synchronize()
    if algo == "tensor_core_cluster":   # row sums folded in a fixed order: bit for bit
        assert torch.equal(first["vote"], again["vote"])
    else:   # the streaming kernel adds them with fp64 atomics in a varying order
        assert torch.allclose(first["vote"], again["vote"], rtol=1e-6, atol=0)
    assert torch.equal(first["idx"], again["idx"])
    assert torch.equal(first["k_out"], again["k_out"])


@pytest.mark.parametrize("algo", ["auto", "tensor_core_cluster", "simt"])
def test_garbage_workspace_shared_across_shapes(dev, algo):
    """The workspace is scratch: random contents, and reuse by a call of another shape, change nothing."""
    from kv_cache_compression_gb300 import snapkv
    shapes = [(synth.WORKLOADS[1].with_(heads=2, l_prompt=3000), 7), (synth.WORKLOADS[1].with_(heads=5, l_prompt=9000), 5),
              (synth.WORKLOADS[1].with_(heads=3, l_prompt=1500, l_obs=16), 9)]
    need = max(snapkv.compress_workspace_size(snapkv.make_params(batch=1, heads=wl.heads, head_dim=wl.head_dim,
                                                                  l_obs=wl.l_obs, l_prompt=wl.l_prompt,
                                                                  pool_kernel=pk, budget=wl.budget,
                                                                  dtype=snapkv.BF16))
               for wl, pk in shapes)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, generator=torch.Generator().manual_seed(3)).to(dev)
    for round_ in range(2):
        for wl, pk in shapes:
            q, k, v, _ = synth.device_inputs(wl, round_, 0, 1, wl.l_prompt, dev)
            fresh = snapkv.compress(q, k, v, pool_kernel=pk, budget=wl.budget, algo=algo, want_vote=True)
            shared = snapkv.compress(q, k, v, pool_kernel=pk, budget=wl.budget, algo=algo, want_vote=True, workspace=ws)
            torch.cuda.synchronize()
            if algo in ("simt", "tensor_core_cluster"):   # fixed summation order: bit for bit
                assert torch.equal(fresh["vote"], shared["vote"])
                assert torch.equal(fresh["idx"], shared["idx"])
                assert torch.equal(fresh["k_out"], shared["k_out"]) and torch.equal(fresh["v_out"], shared["v_out"])
            else:   # the streaming kernel adds with fp64 atomics in a varying order: last bits may differ
                assert torch.allclose(fresh["vote"], shared["vote"], rtol=1e-6, atol=0)
            for h in range(wl.heads):
                hi = synth.host_head(wl, round_, 0, h, l_prompt=wl.l_prompt)
                ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=pk, budget=wl.budget)
                check_compress_head(gpu_idx=shared["idx"][0, h].cpu().numpy(),
                                    gpu_kc=to_numpy_f32(shared["k_out"][0, h]),
                                    gpu_vc=to_numpy_f32(shared["v_out"][0, h]),
                                    gpu_vote=shared["vote"][0, h].cpu().numpy(), ref=ref, k_in=hi.k, v_in=hi.v,
                                    l_prefix=wl.l_prompt - wl.l_obs, l_obs=wl.l_obs, where=f"shape {wl.l_prompt} head {h}")


def test_device_generator_matches_host(dev):
    wl = synth.WORKLOADS[2]
    q, k, v, _ = synth.device_inputs(wl, 5, 3, 1, 2048, dev)
    hi = synth.host_head(wl, 5, 3, 7, l_prompt=2048)
    assert np.array_equal(to_numpy_f32(k[0, 7]), hi.k)
    assert np.array_equal(to_numpy_f32(v[0, 7]), hi.v)
    assert np.array_equal(to_numpy_f32(q[0, 7]), hi.q_obs)


@pytest.mark.parametrize("algo", ["auto", "simt"])
def test_zero_queries_short_prefix(dev, algo):
    """Every pooled score equal on a prefix short enough for the top-k to gather all of them as
    candidates: ties still go to the lower index."""
    from kv_cache_compression_gb300 import snapkv
    B, H, L, lo, d = 1, 2, 2000, 32, 128
    k = torch.randn(B, H, L, d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).to(dev)
    q = torch.zeros(B, H, lo, d, dtype=torch.bfloat16, device=dev)
    res = snapkv.compress(q, k, k.clone(), pool_kernel=7, budget=500, algo=algo)
    torch.cuda.synchronize()
    for h in range(H):
        assert res["idx"][0, h].cpu().tolist() == list(range(500))


@pytest.mark.parametrize("algo", ["auto", "tensor_core_cluster", "simt"])
def test_tied_block_cut_across_slices(dev, algo):
    """A block of zero keys gets one exactly tied vote; the budget cuts inside the block so that the
    kept copies (lowest index first) run past the boundary between two CTAs' slices of the top-k."""
    from kv_cache_compression_gb300 import snapkv
    L, lo, d = 4032, 32, 128
    g = torch.Generator().manual_seed(7)
    q = torch.randn(1, 1, lo, d, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 1, L, d, generator=g)
    k[:, :, 1000:2500] = 0.0
    k = k.to(torch.bfloat16)
    v = torch.randn(1, 1, L, d, generator=g).to(torch.bfloat16)
    qf, kf, vf = (to_numpy_f32(t[0, 0]) for t in (q, k, v))
    l_prefix = L - lo
    c = orc.vote(qf, kf)
    p = orc.max_pool(c, 7)
    tie = p[1500]                                        # inside the block, away from its edges
    assert np.sum(p == tie) > 1300
    budget = int(np.sum(p > tie)) + 1200
    ref = orc.compress_head(qf, kf, vf, pool_kernel=7, budget=budget)
    res = snapkv.compress(q.to(dev), k.to(dev), v.to(dev), pool_kernel=7, budget=budget, algo=algo, want_vote=True)
    torch.cuda.synchronize()
    check_compress_head(gpu_idx=res["idx"][0, 0].cpu().numpy(), gpu_kc=to_numpy_f32(res["k_out"][0, 0]),
                        gpu_vc=to_numpy_f32(res["v_out"][0, 0]), gpu_vote=res["vote"][0, 0].cpu().numpy(), ref=ref,
                        k_in=kf, v_in=vf, l_prefix=l_prefix, l_obs=lo, where="tied block")
    kept_ties = np.intersect1d(res["idx"][0, 0].cpu().numpy(), np.nonzero(p == tie)[0])
    assert kept_ties.size == budget - int(np.sum(p > tie)) and kept_ties[-1] > 2000   # past the first slice


def _timing_event():
    try:
        return torch.cuda.Event(enable_timing=True, external=True)   # an event-record node under capture
    except TypeError:
        return torch.cuda.Event(enable_timing=True)


def test_profiled_compress_records_stage_events(dev):
    """snapkv_compress_profiled gives snapkv_compress's results and records the caller's events
    around each stage, eagerly and as event-record nodes of a captured CUDA graph (replayed)."""
    import ctypes
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1].with_(heads=4)
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, wl.l_prompt, dev)
    ref = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, budget=wl.budget, algo="tensor_core_cluster",
                          want_vote=True)
    params = snapkv.make_params(batch=1, heads=wl.heads, head_dim=wl.head_dim, l_obs=wl.l_obs,
                                l_prompt=wl.l_prompt, pool_kernel=wl.pool_kernel, budget=wl.budget,
                                algo="tensor_core_cluster")
    cap = ref["cap"]
    k_out, v_out = torch.zeros_like(ref["k_out"]), torch.zeros_like(ref["v_out"])
    ln, idx, vote = torch.zeros_like(ref["len"]), torch.zeros_like(ref["idx"]), torch.zeros_like(ref["vote"])
    ws = snapkv.new_workspace(snapkv.compress_workspace_size(params), dev)
    stream = torch.cuda.Stream(dev)
    evs = [_timing_event() for _ in range(8)]
    with torch.cuda.stream(stream):
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    P = ctypes.c_void_p
    arr = (ctypes.c_void_p * 8)(*[e.cuda_event for e in evs])

    def call():
        st = snapkv.lib().snapkv_compress_profiled(
            ctypes.byref(params), P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(k_out.data_ptr()),
            P(v_out.data_ptr()), cap, P(ln.data_ptr()), P(idx.data_ptr()), P(vote.data_ptr()), P(ws.data_ptr()),
            ws.numel(), None, P(stream.cuda_stream), arr, 8)
        assert st == snapkv.OK, snapkv.status_string(st)

    def check():
        for key, got in (("k_out", k_out), ("v_out", v_out), ("len", ln), ("idx", idx), ("vote", vote)):
            assert torch.equal(got, ref[key]), key
        stage = [evs[2 * s].elapsed_time(evs[2 * s + 1]) for s in range(4)]
        assert stage[0] > 0 and stage[2] > 0, stage      # score (+ vote), top-k (+ gather)
        assert all(t >= 0 for t in stage), stage

    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    check()
    for t in (k_out, v_out, ln, idx, vote):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    graph.replay()
    torch.cuda.synchronize()
    check()
