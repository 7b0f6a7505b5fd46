"""GPU parity of snapkv_append + snapkv_decode_attend against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import synth
from oracle import snapkv_oracle as orc
from tests.parity import check_decode, to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(gpu_device):
    import __graft_entry__
    __graft_entry__.build()
    return gpu_device


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 128),
                                     (torch.float32, 64)])
def test_decode_ragged_lengths(dev, dtype, d):
    from kv_cache_compression_gb300 import snapkv
    g = torch.Generator().manual_seed(d)
    B, H, cap = 5, 3, 700
    lens = [1, 255, 256, 699, 700]
    kc = torch.randn(B, H, cap, d, generator=g).to(dtype)
    vc = torch.randn(B, H, cap, d, generator=g).to(dtype)
    q = (torch.randn(B, H, d, generator=g) * 2).to(dtype)
    length = torch.tensor(lens, dtype=torch.int32)
    out = snapkv.decode_attend(q.to(dev), kc.to(dev), vc.to(dev), length.to(dev))
    torch.cuda.synchronize()
    o = to_numpy_f32(out)
    for b in range(B):
        for h in range(H):
            n = lens[b]
            ref = orc.decode_attend(q[b, h].float().numpy(), kc[b, h, :n].float().numpy(), vc[b, h, :n].float().numpy())
            check_decode(o[b, h], ref, dtype == torch.bfloat16, where=f"b{b} h{h} n{n}")


def test_decode_zero_length_gives_zero_and_overlong_is_reported(dev):
    from kv_cache_compression_gb300 import snapkv
    B, H, cap, d = 2, 2, 64, 128
    kc = torch.randn(B, H, cap, d, device=dev).to(torch.bfloat16)
    vc = torch.randn(B, H, cap, d, device=dev).to(torch.bfloat16)
    q = torch.randn(B, H, d, device=dev).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = snapkv.decode_attend(q, kc, vc, torch.tensor([0, cap + 5], dtype=torch.int32, device=dev),
                               dev_status=status)
    torch.cuda.synchronize()
    assert torch.all(out[0] == 0)
    assert int(status.item()) & snapkv.ERR_CAPACITY
    full = snapkv.decode_attend(q, kc, vc, torch.tensor([cap, cap], dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert torch.equal(out[1], full[1])     # clamped to the capacity


@pytest.mark.parametrize("dtype,d,cap", [(torch.bfloat16, 128, 700), (torch.bfloat16, 64, 700),
                                         (torch.float32, 128, 700), (torch.float32, 64, 129),
                                         (torch.bfloat16, 128, 20000)])
def test_fused_append_decode_equals_the_two_calls(dev, dtype, d, cap):
    """snapkv_append_decode_attend leaves the bytes snapkv_append then snapkv_decode_attend leave
    (cache, new lengths, output), for sequences appending at row 0, row 1, mid-cache and the last
    free row, and a full one (reported, not appended); caches beyond 16384 rows take the two
    kernels in turn."""
    from kv_cache_compression_gb300 import snapkv
    g = torch.Generator().manual_seed(cap + d)
    B, H = 5, 3
    lens = [0, 1, cap // 2, cap - 1, cap]
    kc = torch.randn(B, H, cap, d, generator=g).to(dtype).to(dev)
    vc = torch.randn(B, H, cap, d, generator=g).to(dtype).to(dev)
    q = (torch.randn(B, H, d, generator=g) * 2).to(dtype).to(dev)
    kn = torch.randn(B, H, d, generator=g).to(dtype).to(dev)
    vn = torch.randn(B, H, d, generator=g).to(dtype).to(dev)
    length = torch.tensor(lens, dtype=torch.int32, device=dev)
    kc1, vc1, len1 = kc.clone(), vc.clone(), length.clone()
    st1 = torch.zeros(1, dtype=torch.int32, device=dev)
    snapkv.append(kn, vn, kc1, vc1, len1, dev_status=st1)
    out1 = snapkv.decode_attend(q, kc1, vc1, len1, dev_status=st1)
    kc2, vc2 = kc.clone(), vc.clone()
    st2 = torch.zeros(1, dtype=torch.int32, device=dev)
    out2, len2 = snapkv.append_decode_attend(q, kn, vn, kc2, vc2, length, dev_status=st2)
    torch.cuda.synchronize()
    assert length.cpu().tolist() == lens                   # len_in is only read
    assert len2.cpu().tolist() == len1.cpu().tolist() == [1, 2, cap // 2 + 1, cap, cap]
    assert int(st1.item()) == int(st2.item()) == snapkv.ERR_CAPACITY
    assert torch.equal(kc2, kc1) and torch.equal(vc2, vc1)
    assert torch.equal(out2, out1)
    o = to_numpy_f32(out2)
    for b in (0, 3):
        n = lens[b]
        kref = torch.cat([kc[b, 1, :n], kn[b, 1][None]]).float().cpu().numpy()
        vref = torch.cat([vc[b, 1, :n], vn[b, 1][None]]).float().cpu().numpy()
        check_decode(o[b, 1], orc.decode_attend(q[b, 1].float().cpu().numpy(), kref, vref), dtype == torch.bfloat16,
                     where=f"fused b{b} n{n}")


def test_bench_step_launch_configuration(dev):
    """The benchmark's step as it is timed: the Llama-2-7B-shaped layer compressed into a cache of
    capacity k + L_obs + 1, then one fused decode step filling its last row; every head's output
    against the oracle's decode over that head's cache rows (compression parity is checked on
    every head elsewhere), and the new length."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1]
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, wl.l_prompt, dev)
    cap = wl.budget + wl.l_obs + 1
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, budget=wl.budget, cap=cap, dev_status=status)
    qn, kn, vn = synth.device_decode_tokens(wl, 0, 0, 0, 1, dev)
    out, len_next = snapkv.append_decode_attend(qn, kn, vn, res["k_out"], res["v_out"], res["len"],
                                                dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert res["len"].item() == cap - 1 and len_next.item() == cap
    o = to_numpy_f32(out)
    kc, vc = to_numpy_f32(res["k_out"]), to_numpy_f32(res["v_out"])
    for h in range(wl.heads):
        qh, kh, vh = synth.host_decode_token(wl, 0, 0, h, 0)
        assert np.array_equal(kc[0, h, cap - 1], kh) and np.array_equal(vc[0, h, cap - 1], vh)
        check_decode(o[0, h], orc.decode_attend(qh, kc[0, h], vc[0, h]), True, where=f"head {h}")


def test_append_writes_row_and_advances_length(dev):
    from kv_cache_compression_gb300 import snapkv
    B, H, cap, d = 3, 4, 10, 64
    kc = torch.zeros(B, H, cap, d, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    length = torch.tensor([0, 5, cap], dtype=torch.int32, device=dev)
    kn = torch.randn(B, H, d, device=dev).to(torch.bfloat16)
    vn = torch.randn(B, H, d, device=dev).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    snapkv.append(kn, vn, kc, vc, length, dev_status=status)
    torch.cuda.synchronize()
    assert length.cpu().tolist() == [1, 6, cap]          # the full sequence is left as it was
    assert int(status.item()) == snapkv.ERR_CAPACITY
    assert torch.equal(kc[0, :, 0], kn[0]) and torch.equal(vc[1, :, 5], vn[1])
    assert torch.count_nonzero(kc[2]) == 0
    assert torch.count_nonzero(kc[0, :, 1:]) == 0


def test_uncompressed_cache_decode_equals_full_causal_attention(dev):
    """KV-cache chapter 22.7 on the GPU: with k = L_prefix the compressed cache is the whole prompt,
    and append + decode of each new token gives the oracle's cached-decode rows (which the oracle's
    own pin equates with full causal attention)."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1].with_(heads=2, l_prompt=640, budget=0, ratio_p=1.0, plants=0)
    steps = 6
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, wl.l_prompt, dev)
    res = snapkv.compress(q, k, v, pool_kernel=7, ratio_p=1.0, cap=wl.l_prompt + steps)
    outs = []
    for t in range(steps):
        qn, kn, vn = synth.device_decode_tokens(wl, 0, t, 0, 1, dev)
        snapkv.append(kn, vn, res["k_out"], res["v_out"], res["len"])
        outs.append(snapkv.decode_attend(qn, res["k_out"], res["v_out"], res["len"]))
    torch.cuda.synchronize()
    assert res["len"].item() == wl.l_prompt + steps
    for h in range(wl.heads):
        hi = synth.host_head(wl, 0, 0, h)
        kc, vc = hi.k, hi.v
        for t in range(steps):
            qn, kn, vn = synth.host_decode_token(wl, 0, 0, h, t)
            kc, vc = orc.append(kc, vc, kn, vn)
            check_decode(to_numpy_f32(outs[t][0, h]), orc.decode_attend(qn, kc, vc), True, where=f"h{h} t{t}")


@pytest.mark.parametrize("fused", [False, True], ids=["append+decode", "fused"])
def test_compressed_decode_workload_sampled(dev, fused):
    """The ragged-prompt decode workload on sampled (sequence, layer): compress into a cache of
    capacity 2048 + L_obs + 128, then all 128 decode steps of append + attention (two calls, or the
    fused call with two length arrays in turn), checked against the oracle re-simulating
    compression and every step on sampled heads."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[4]
    lens = wl.prompt_lengths()
    cap = wl.budget + wl.l_obs + wl.decode_steps
    for seq, layer, heads in ((3, 0, [0, 17]), (int(np.argmax(lens)), 31, [31])):
        L = lens[seq]
        q, k, v, _ = synth.device_inputs(wl, layer, seq, 1, L, dev)
        res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, budget=wl.budget, cap=cap)
        del q, k, v
        ws = snapkv.new_workspace(snapkv.decode_workspace_size(1, wl.heads, wl.head_dim, cap), dev)
        outs = []
        len_bufs = [res["len"], torch.empty_like(res["len"])]
        for t in range(wl.decode_steps):
            qn, kn, vn = synth.device_decode_tokens(wl, layer, t, seq, 1, dev)
            if fused:
                o, _ = snapkv.append_decode_attend(qn, kn, vn, res["k_out"], res["v_out"], len_bufs[t % 2],
                                                   len_bufs[(t + 1) % 2], workspace=ws)
            else:
                snapkv.append(kn, vn, res["k_out"], res["v_out"], res["len"])
                o = snapkv.decode_attend(qn, res["k_out"], res["v_out"], res["len"], workspace=ws)
            outs.append(o[0, heads].cpu())
        torch.cuda.synchronize()
        assert len_bufs[wl.decode_steps % 2 if fused else 0].item() == cap
        for j, h in enumerate(heads):
            hi = synth.host_head(wl, layer, seq, h, l_prompt=L)
            ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, budget=wl.budget)
            got_idx = res["idx"][0, h].cpu().numpy()
            # decode continues from the GPU's own kept set (identical unless a boundary tie flipped)
            kc, vc = orc.gather_with_window(hi.k, got_idx, L - wl.l_obs), orc.gather_with_window(hi.v, got_idx, L - wl.l_obs)
            assert np.setxor1d(got_idx, ref.idx).size == 0 or \
                np.all(np.abs(ref.p[np.setxor1d(got_idx, ref.idx)] - ref.tau) <= 1e-5 * ref.tau)
            for t in range(wl.decode_steps):
                qn, kn, vn = synth.host_decode_token(wl, layer, seq, h, t)
                kc, vc = orc.append(kc, vc, kn, vn)
                check_decode(to_numpy_f32(outs[t][j]), orc.decode_attend(qn, kc, vc), True,
                             where=f"seq {seq} layer {layer} head {h} step {t}")


def test_decode_garbage_workspace_shared_across_shapes(dev):
    """The decode workspace is scratch: random contents and reuse by another shape change nothing."""
    from kv_cache_compression_gb300 import snapkv
    g = torch.Generator().manual_seed(11)
    shapes = [(2, 3, 300), (6, 4, 1500), (1, 2, 90)]
    need = max(snapkv.decode_workspace_size(B, H, 128, cap) for B, H, cap in shapes)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, generator=g).to(dev)
    for B, H, cap in shapes * 2:
        kc = torch.randn(B, H, cap, 128, generator=g).to(torch.bfloat16).to(dev)
        vc = torch.randn(B, H, cap, 128, generator=g).to(torch.bfloat16).to(dev)
        q = torch.randn(B, H, 128, generator=g).to(torch.bfloat16).to(dev)
        length = torch.randint(1, cap + 1, (B,), generator=g, dtype=torch.int32).to(dev)
        fresh = snapkv.decode_attend(q, kc, vc, length)
        shared = snapkv.decode_attend(q, kc, vc, length, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(fresh, shared)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_long_cache_split_path(dev, dtype):
    """Caches beyond 16K rows take the split kernel (workspace partials + per-head tickets)."""
    from kv_cache_compression_gb300 import snapkv
    g = torch.Generator().manual_seed(5)
    B, H, d, cap = 2, 2, 128, 17000
    lens = [16999, 9000]
    kc = torch.randn(B, H, cap, d, generator=g).to(dtype)
    vc = torch.randn(B, H, cap, d, generator=g).to(dtype)
    q = (torch.randn(B, H, d, generator=g) * 2).to(dtype)
    out = snapkv.decode_attend(q.to(dev), kc.to(dev), vc.to(dev), torch.tensor(lens, dtype=torch.int32).to(dev))
    torch.cuda.synchronize()
    o = to_numpy_f32(out)
    for b in range(B):
        for h in range(H):
            n = lens[b]
            ref = orc.decode_attend(q[b, h].float().numpy(), kc[b, h, :n].float().numpy(), vc[b, h, :n].float().numpy())
            check_decode(o[b, h], ref, dtype == torch.bfloat16, where=f"b{b} h{h} n{n}")


@pytest.mark.parametrize("extra", [0, 1])
def test_full_16k_cache_decode_sampled(dev, extra):
    """Decode over an uncompressed 16K-row prompt cache (batch 2), the baseline the compressed
    cache is compared with: cap 16384 takes the cluster kernel, cap 16385 the split kernel."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[1]
    B, L = 2, wl.l_prompt
    _, k, v, _ = synth.device_inputs(wl, 0, 0, B, L, dev)
    qn, kn, vn = synth.device_decode_tokens(wl, 0, 0, 0, B, dev)
    cap = L + extra
    kc = torch.zeros((B, wl.heads, cap, wl.head_dim), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    kc[:, :, :L] = k
    vc[:, :, :L] = v
    length = torch.full((B,), L, dtype=torch.int32, device=dev)
    if extra:   # append the new token first, as a decode step does
        snapkv.append(kn, vn, kc, vc, length)
    out = snapkv.decode_attend(qn, kc, vc, length)
    torch.cuda.synchronize()
    n = L + extra
    o = to_numpy_f32(out)
    for b, h in [(0, 0), (1, 17), (1, 31)]:
        ref = orc.decode_attend(to_numpy_f32(qn[b, h]), to_numpy_f32(kc[b, h, :n]), to_numpy_f32(vc[b, h, :n]))
        check_decode(o[b, h], ref, True, where=f"b{b} h{h} n{n}")


def test_prefill_step_launch_configuration(dev):
    """The 32-layer prefill benchmark's per-layer step as it is timed: one layer of B8 x 32 heads
    compressed (p = 0.05) into a cache of capacity k + L_obs + 1, then one fused decode step filling its
    last row (256 heads: one CTA per head); every head's output against the oracle's decode over that
    head's cache rows, the appended rows and the new lengths."""
    from kv_cache_compression_gb300 import snapkv
    wl = synth.WORKLOADS[2]
    B, H, L = wl.batch, wl.heads, wl.l_prompt
    q, k, v, _ = synth.device_inputs(wl, 7, 0, B, L, dev)
    ksel = orc.kept_slots(L - wl.l_obs, ratio_p=wl.ratio_p)
    cap = ksel + wl.l_obs + 1
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p, cap=cap, dev_status=status)
    del q, k, v
    qn, kn, vn = synth.device_decode_tokens(wl, 7, 0, 0, B, dev)
    out, len_next = snapkv.append_decode_attend(qn, kn, vn, res["k_out"], res["v_out"], res["len"],
                                                dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert res["len"].cpu().tolist() == [cap - 1] * B and len_next.cpu().tolist() == [cap] * B
    o = to_numpy_f32(out)
    kc, vc = to_numpy_f32(res["k_out"]), to_numpy_f32(res["v_out"])
    for b in range(B):
        for h in range(H):
            qh, kh, vh = synth.host_decode_token(wl, 7, b, h, 0)
            assert np.array_equal(kc[b, h, cap - 1], kh) and np.array_equal(vc[b, h, cap - 1], vh)
            check_decode(o[b, h], orc.decode_attend(qh, kc[b, h], vc[b, h]), True, where=f"seq {b} head {h}")


def decode_parity_triples(seed=0xC4):
    """64 seeded (sequence, layer, head) triples of the decode workload; layer -> [(sequence, head)]."""
    rng = np.random.default_rng(seed)
    by_layer = {}
    for u in rng.choice(64 * 32 * 32, size=64, replace=False):
        seq, layer, head = int(u // 1024), int((u // 32) % 32), int(u % 32)
        by_layer.setdefault(layer, []).append((seq, head))
    return dict(sorted(by_layer.items()))


def test_decode_workload_64_triples_through_128_steps(dev):
    """The compressed-decode workload in the benchmark's launch configuration: per layer, the 64 ragged
    prompts compressed (budget 2048, one snapkv_compress_varlen call per 16 sequences) into a
    [64, 32, 2208, 128] cache, then 128 fused append + attention steps over all 64 x 32 heads. For 64
    seeded (sequence, layer, head) triples the compression and every step's output are checked
    against the oracle, which re-simulates that head from its own inputs through all 128 steps; the
    cache rows past the compressed length stay untouched until the steps write them."""
    from kv_cache_compression_gb300 import snapkv
    from tests import oracle_pool
    from tests.parity import assert_canary, bf16_bits, canary_like
    wl = synth.WORKLOADS[4]
    B, H, d, lo, steps = wl.batch, wl.heads, wl.head_dim, wl.l_obs, wl.decode_steps
    lengths = wl.prompt_lengths()
    cap = wl.budget + lo + steps
    R = wl.budget + lo
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = snapkv.new_workspace(snapkv.decode_workspace_size(B, H, d, cap), dev)
    jobs = []
    for layer, units in decode_parity_triples().items():
        kc = canary_like((B, H, cap, d), torch.bfloat16, dev)
        vc = canary_like((B, H, cap, d), torch.bfloat16, dev)
        lens = torch.zeros((2, B), dtype=torch.int32, device=dev)
        idx = torch.empty((B, H, wl.budget), dtype=torch.int32, device=dev)
        for c0 in range(0, B, 16):
            ls = lengths[c0:c0 + 16]
            q, k, v = synth.device_inputs_padded(wl, layer, c0, ls, dev, pad_value=0.0)
            res = snapkv.compress_varlen(q, k, v, ls, pool_kernel=wl.pool_kernel, budget=wl.budget,
                                         k_out=kc[c0:c0 + 16], v_out=vc[c0:c0 + 16], len_out=lens[0, c0:c0 + 16],
                                         dev_status=status)
            idx[c0:c0 + 16].copy_(res["idx"])
            del q, k, v
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert lens[0].cpu().tolist() == [R] * B
        assert_canary(kc[:, :, R:], f"layer {layer}: cache rows past the compressed length")
        sel_b = torch.tensor([s for s, _ in units], device=dev)
        sel_h = torch.tensor([h for _, h in units], device=dev)
        kc_bits, vc_bits = bf16_bits(kc[sel_b, sel_h, :R]), bf16_bits(vc[sel_b, sel_h, :R])
        idx_sel = idx[sel_b, sel_h].cpu().numpy()
        outs = torch.empty((steps, len(units), d), dtype=torch.bfloat16, device=dev)
        out = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)
        for t in range(steps):
            qn, kn, vn = synth.device_decode_tokens(wl, layer, t, 0, B, dev)
            snapkv.append_decode_attend(qn, kn, vn, kc, vc, lens[t % 2], lens[(t + 1) % 2], out=out, workspace=ws,
                                        dev_status=status)
            outs[t] = out[sel_b, sel_h]
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert lens[steps % 2].cpu().tolist() == [cap] * B
        out_bits = bf16_bits(outs)
        for i, (s, h) in enumerate(units):
            jobs.append(dict(wl=wl, layer=layer, seq=s, head=h, l_prompt=lengths[s], idx=idx_sel[i],
                             kc_bits=kc_bits[i], vc_bits=vc_bits[i], out_bits=out_bits[:, i],
                             where=f"seq {s} (L {lengths[s]}) layer {layer} head {h}"))
        del kc, vc
    results = oracle_pool.run(oracle_pool.check_decode_run_job, jobs)
    errors = [f"{w}: {e}" for w, _, e in results if e is not None]
    assert not errors, "\n".join(errors[:5])
    assert len(jobs) == 64
    worst = max(r[1] for _, r, _ in results)
    print(f"decode workload: 64 triples x 128 steps, worst |o - o_ref| {worst:.2e}, "
          f"{sum(r[0] for _, r, _ in results)} boundary-excused indices")
