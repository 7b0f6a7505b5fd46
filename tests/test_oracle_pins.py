"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each check compares the oracle with something other than itself: a closed form, an invariant,
a torch library routine, brute-force enumeration, or a value the pages print (tests/golden/).
The ``pin_*`` helpers return the worst error so that ``test_oracle_mutations.py`` can show that
a planted mistake in the oracle makes them fail.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import snapkv_oracle as orc
from tests.conftest import golden


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


# ------------------------------------------------------------------------------------------------
# Pin helpers (return the worst absolute error; the tests assert on it)
# ------------------------------------------------------------------------------------------------

def pin_weights_vs_sdpa(oracle, q_all, k, l_obs):
    """Window rows of torch's full causal attention (queries for every prompt position) equal W.

    torch's scaled_dot_product_attention(is_causal=True) over the whole prompt, with the identity
    as values, returns the attention matrix; its last L_obs rows are the window queries' weights.
    """
    L = k.shape[0]
    qt = torch.from_numpy(q_all)[None, None]
    kt = torch.from_numpy(k)[None, None]
    eye = torch.eye(L, dtype=torch.float64)[None, None]
    w_full = F.scaled_dot_product_attention(qt, kt, eye, is_causal=True)[0, 0].numpy()
    w = oracle.window_weights(q_all[L - l_obs:], k, oracle.PROMPT_CAUSAL)
    return float(np.abs(w - w_full[L - l_obs:]).max())


def pin_prefix_only_vs_torch_softmax(oracle, q_obs, k):
    """PREFIX_ONLY weights equal torch.softmax of the prefix logits (padded with zeros)."""
    l_obs = q_obs.shape[0]
    l_prefix = k.shape[0] - l_obs
    qt, kt = torch.from_numpy(q_obs), torch.from_numpy(k[:l_prefix])
    ref = torch.softmax(qt @ kt.T / math.sqrt(q_obs.shape[1]), dim=-1).numpy()
    w = oracle.window_weights(q_obs, k, oracle.PREFIX_ONLY)
    return max(float(np.abs(w[:, :l_prefix] - ref).max()), float(np.abs(w[:, l_prefix:]).max()))


def pin_pool_vs_torch(oracle, c, kernel):
    ref = F.max_pool1d(torch.from_numpy(c)[None, None], kernel, stride=1, padding=kernel // 2)[0, 0]
    return float(np.abs(oracle.max_pool(c, kernel) - ref.numpy()).max())


def brute_force_topk(p, k):
    """Max-sum k-subset; among equal sums, the lexicographically smallest sorted index tuple."""
    best, best_key = None, None
    for sub in itertools.combinations(range(len(p)), k):
        key = (-sum(p[j] for j in sub), sub)
        if best_key is None or key < best_key:
            best, best_key = sub, key
    return np.array(best, dtype=np.int64)


def pin_decode_vs_full_causal(oracle, x_q, x_k, x_v, l_prompt):
    """Cached decode over an uncompressed cache equals rows of torch's full causal attention.

    Mirrors the KV-cache chapter's section 22.7 check: the prompt's keys/values form the cache,
    then every new token is appended and attended; each output must equal the matching row of
    scaled_dot_product_attention(is_causal=True) over the whole sequence.
    """
    T = x_q.shape[0]
    full = F.scaled_dot_product_attention(torch.from_numpy(x_q)[None, None],
                                          torch.from_numpy(x_k)[None, None],
                                          torch.from_numpy(x_v)[None, None], is_causal=True)[0, 0].numpy()
    k_c, v_c = x_k[:l_prompt].copy(), x_v[:l_prompt].copy()
    worst = 0.0
    for t in range(l_prompt, T):
        k_c, v_c = oracle.append(k_c, v_c, x_k[t], x_v[t])
        o = oracle.decode_attend(x_q[t], k_c, v_c)
        worst = max(worst, float(np.abs(o - full[t]).max()))
    return worst, k_c.shape


# ------------------------------------------------------------------------------------------------
# Split and kept slots
# ------------------------------------------------------------------------------------------------

def test_split_and_kept_slots():
    presets = golden("snapkv_presets.json")
    p = presets["ratio_p"]
    assert orc.prefix_length(1024, 32) == 992
    # k = floor(p * L_prefix): 0.05 * 992 = 49.6 -> 49, 0.05 * 16352 = 817.6 -> 817.
    assert orc.kept_slots(992, ratio_p=p) == 49
    assert orc.kept_slots(16352, ratio_p=p) == 817
    assert orc.kept_slots(1000, ratio_p=p) == 50          # exact product stays exact
    assert orc.kept_slots(19, ratio_p=p) == 0             # k = 0 is allowed
    assert orc.kept_slots(992, ratio_p=1.0) == 992
    for pre in presets["presets"]:
        for cap in pre["max_kept"]:
            assert orc.kept_slots(16352, budget=cap) == min(cap, 16352)
            assert orc.kept_slots(cap // 2, budget=cap) == cap // 2
    with pytest.raises(ValueError):
        orc.prefix_length(32, 32)
    with pytest.raises(ValueError):
        orc.kept_slots(10, ratio_p=1.5)


# ------------------------------------------------------------------------------------------------
# Softmax and vote
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("l_prompt,l_obs,d", [(40, 8, 8), (97, 16, 16), (300, 32, 64), (130, 64, 32)])
def test_weights_match_torch_full_causal_attention(l_prompt, l_obs, d):
    rng = np.random.default_rng(l_prompt * 7 + l_obs)
    q_all, k = _rand(rng, l_prompt, d, scale=1.5), _rand(rng, l_prompt, d)
    assert pin_weights_vs_sdpa(orc, q_all, k, l_obs) < 1e-13


@pytest.mark.parametrize("l_prompt,l_obs,d", [(40, 8, 8), (200, 32, 64)])
def test_prefix_only_weights_match_torch_softmax(l_prompt, l_obs, d):
    rng = np.random.default_rng(5 + l_prompt)
    q, k = _rand(rng, l_obs, d, scale=2.0), _rand(rng, l_prompt, d)
    assert pin_prefix_only_vs_torch_softmax(orc, q, k) < 1e-13


@pytest.mark.parametrize("scope", [orc.PROMPT_CAUSAL, orc.PREFIX_ONLY])
def test_vote_sums_to_window_length(scope):
    """Every row of W sums to 1, so the vote over all visible columns sums to L_obs."""
    rng = np.random.default_rng(11)
    for l_prompt, l_obs, d in [(64, 16, 8), (1024, 32, 64), (500, 64, 128)]:
        q, k = _rand(rng, l_obs, d, scale=3.0), _rand(rng, l_prompt, d)
        c_all = orc.vote_all_columns(q, k, scope)
        assert abs(c_all.sum() - l_obs) < 1e-10 * l_obs
        if scope == orc.PREFIX_ONLY:
            assert abs(orc.vote(q, k, scope).sum() - l_obs) < 1e-10 * l_obs
        assert (c_all >= 0).all()


def test_vote_zero_queries_closed_form():
    """q = 0: row i spreads 1/(L_prefix + i + 1) over its visible columns, so every prefix column
    gets sum_i 1/(L_prefix + i + 1); all pooled values tie and the kept set is 0..k-1."""
    l_prompt, l_obs, d = 300, 16, 8
    l_prefix = l_prompt - l_obs
    k = _rand(np.random.default_rng(3), l_prompt, d)
    c = orc.vote(np.zeros((l_obs, d)), k)
    expect = sum(1.0 / (l_prefix + i + 1) for i in range(l_obs))
    assert np.abs(c - expect).max() < 1e-14
    res = orc.compress_head(np.zeros((l_obs, d)), k, k, pool_kernel=7, budget=40)
    assert res.idx.tolist() == list(range(40))
    # prefix-only: every row spreads uniformly over the L_prefix columns
    c2 = orc.vote(np.zeros((l_obs, d)), k, orc.PREFIX_ONLY)
    assert np.abs(c2 - l_obs / l_prefix).max() < 1e-14


def test_vote_dominant_key_closed_form():
    """A key whose logit dwarfs every other takes all the weight of every row: C_j* = L_obs."""
    l_prompt, l_obs, d = 128, 16, 8
    q = np.zeros((l_obs, d))
    q[:, 0] = 30.0
    k = np.zeros((l_prompt, d))
    k[57, 0] = 30.0
    c = orc.vote(q, k)
    assert abs(c[57] - l_obs) < 1e-12
    assert np.delete(c, 57).max() < 1e-100


def test_vote_window_rows_are_causal():
    """The first window query sees no later window key: its row has no weight past L_prefix."""
    rng = np.random.default_rng(8)
    l_prompt, l_obs, d = 50, 10, 4
    q, k = _rand(rng, l_obs, d), _rand(rng, l_prompt, d)
    w = orc.window_weights(q, k)
    l_prefix = l_prompt - l_obs
    for i in range(l_obs):
        assert np.all(w[i, l_prefix + i + 1:] == 0.0)
        assert np.all(w[i, :l_prefix + i + 1] > 0.0)


# ------------------------------------------------------------------------------------------------
# Max pool
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", [1, 3, 5, 7, 13])
def test_max_pool_matches_torch(kernel):
    rng = np.random.default_rng(kernel)
    for n in (1, 2, 7, 50, 1000):
        c = rng.random(n)
        assert pin_pool_vs_torch(orc, c, kernel) == 0.0


def test_max_pool_identity_and_constant():
    rng = np.random.default_rng(1)
    c = rng.random(40)
    assert np.array_equal(orc.max_pool(c, 1), c)
    assert np.all(orc.max_pool(c, 2 * 40 - 1) == c.max())
    with pytest.raises(ValueError):
        orc.max_pool(c, 4)


# ------------------------------------------------------------------------------------------------
# Top-k
# ------------------------------------------------------------------------------------------------

def test_topk_brute_force_enumeration():
    rng = np.random.default_rng(21)
    for trial in range(60):
        n = int(rng.integers(1, 13))
        p = rng.integers(0, 4, size=n).astype(np.float64)   # many exact ties
        for k in range(0, n + 1):
            got = orc.select_topk(p, k)
            assert got.tolist() == brute_force_topk(p.tolist(), k).tolist()
            assert orc.select_by_sort(p, k).tolist() == got.tolist()


def test_topk_rank_and_sort_agree_with_ties():
    rng = np.random.default_rng(2)
    for n in (10, 333, 3000):
        p = np.round(rng.random(n), 2)
        for k in (0, 1, n // 7, n // 2, n):
            assert np.array_equal(orc.select_by_rank(p, k), orc.select_by_sort(p, k))


def test_topk_matches_torch_on_distinct_values():
    rng = np.random.default_rng(4)
    for n in (5, 100, 5000):
        p = rng.random(n)
        for k in (1, n // 3, n):
            ref = np.sort(torch.topk(torch.from_numpy(p), k).indices.numpy())
            assert np.array_equal(orc.select_topk(p, k), ref)


def test_kth_largest():
    p = np.array([0.5, 0.1, 0.9, 0.5, 0.3])
    assert orc.kth_largest(p, 1) == 0.9
    assert orc.kth_largest(p, 2) == 0.5
    assert orc.kth_largest(p, 3) == 0.5
    assert orc.kth_largest(p, 5) == 0.1


# ------------------------------------------------------------------------------------------------
# Gather + window, whole compression
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("preset", golden("snapkv_presets.json")["presets"], ids=lambda p: p["name"])
def test_compress_invariants(preset):
    rng = np.random.default_rng(preset["l_obs"])
    l_obs, kernel = preset["l_obs"], preset["pool_kernel"]
    l_prompt, d = 700, 32
    l_prefix = l_prompt - l_obs
    q = _rand(rng, l_obs, d).astype(np.float32)
    k = _rand(rng, l_prompt, d).astype(np.float32)
    v = _rand(rng, l_prompt, d).astype(np.float32)
    for kw in (dict(ratio_p=0.05), dict(budget=100), dict(ratio_p=0.0), dict(budget=10 ** 6),
               dict(ratio_p=1.0)):
        res = orc.compress_head(q, k, v, pool_kernel=kernel, **kw)
        kk = orc.kept_slots(l_prefix, **{"ratio_p": 0.0, "budget": 0, **kw})
        assert res.idx.shape == (kk,)
        assert res.k_c.shape == (kk + l_obs, d) and res.v_c.shape == (kk + l_obs, d)
        assert np.all(np.diff(res.idx) > 0) and (kk == 0 or (res.idx[0] >= 0 and res.idx[-1] < l_prefix))
        # the window is always kept, bit for bit, after the kept prefix rows
        assert np.array_equal(res.k_c[kk:], k[l_prefix:]) and np.array_equal(res.v_c[kk:], v[l_prefix:])
        assert np.array_equal(res.k_c[:kk], k[res.idx]) and np.array_equal(res.v_c[:kk], v[res.idx])
        if kk == l_prefix:     # p = 1, or a budget beyond the prefix: the cache is returned whole
            assert np.array_equal(res.k_c, k) and np.array_equal(res.v_c, v)
        if kk > 0:             # every kept pooled value is >= tau, every dropped one <= tau
            dropped = np.setdiff1d(np.arange(l_prefix), res.idx)
            assert res.p[res.idx].min() >= res.tau
            assert dropped.size == 0 or res.p[dropped].max() <= res.tau


def test_strong_planted_keys_are_kept():
    """Keys pushed far along the mean window query are always kept when plants * K_pool <= k."""
    rng = np.random.default_rng(99)
    l_prompt, l_obs, d, kernel = 2048, 32, 64, 7
    l_prefix = l_prompt - l_obs
    q = _rand(rng, l_obs, d)
    k = _rand(rng, l_prompt, d)
    u = q.mean(axis=0)
    u /= np.linalg.norm(u)
    plants = rng.choice(l_prefix, size=8, replace=False)
    k[plants] += 50.0 * u
    res = orc.compress_head(q, k, k, pool_kernel=kernel, budget=8 * kernel)
    assert set(plants.tolist()) <= set(res.idx.tolist())


def test_listing_semantics_prefix_only_with_torch_ops():
    """The restated listing's pipeline, written here with torch ops (softmax over the prefix,
    sum over the window rows, max_pool1d, topk, ascending sort, gather, concatenation), gives the
    oracle's PREFIX_ONLY result on inputs without ties in the pooled scores."""
    rng = np.random.default_rng(17)
    B, H, L, lo, d, kernel, cap = 1, 3, 400, 16, 32, 5, 60
    q = torch.from_numpy(_rand(rng, B, H, L, d))
    k = torch.from_numpy(_rand(rng, B, H, L, d))
    v = torch.from_numpy(_rand(rng, B, H, L, d))
    pfx = L - lo
    w = torch.softmax((q[:, :, pfx:] @ k[:, :, :pfx].transpose(-1, -2)) / math.sqrt(d), dim=-1)
    pooled = F.max_pool1d(w.sum(dim=2), kernel, stride=1, padding=kernel // 2)
    sel = pooled.topk(min(cap, pfx), dim=-1).indices.sort(dim=-1).values
    g = sel[..., None].expand(-1, -1, -1, d)
    k_ref = torch.cat([torch.gather(k[:, :, :pfx], 2, g), k[:, :, pfx:]], dim=2)
    v_ref = torch.cat([torch.gather(v[:, :, :pfx], 2, g), v[:, :, pfx:]], dim=2)
    for h in range(H):
        res = orc.compress_head(q[0, h, pfx:].numpy(), k[0, h].numpy(), v[0, h].numpy(),
                                pool_kernel=kernel, budget=cap, scope=orc.PREFIX_ONLY)
        assert np.allclose(res.p, pooled[0, h].numpy(), rtol=1e-13, atol=0)
        # compare where the k-th value is not tied (pooling plateaus make exact ties)
        if np.sum(res.p == res.tau) == 1:
            assert np.array_equal(res.idx, sel[0, h].numpy())
            assert np.array_equal(res.k_c, k_ref[0, h].numpy())
            assert np.array_equal(res.v_c, v_ref[0, h].numpy())


# ------------------------------------------------------------------------------------------------
# Append + decode attention
# ------------------------------------------------------------------------------------------------

def test_decode_single_row_returns_its_value():
    rng = np.random.default_rng(6)
    k, v = _rand(rng, 1, 16), _rand(rng, 1, 16)
    assert np.abs(orc.decode_attend(_rand(rng, 16, scale=5.0), k, v) - v[0]).max() < 1e-15


def test_decode_zero_query_is_mean_of_values():
    rng = np.random.default_rng(7)
    k, v = _rand(rng, 37, 16), _rand(rng, 37, 16)
    assert np.abs(orc.decode_attend(np.zeros(16), k, v) - v.mean(axis=0)).max() < 1e-14


def test_decode_large_logits_are_stable():
    k = np.zeros((3, 4))
    k[1, 0] = 1.0
    v = np.eye(3, 4)
    q = np.array([4000.0, 0, 0, 0])
    assert np.abs(orc.decode_attend(q, k, v) - v[1]).max() < 1e-15


def test_cached_decode_equals_full_causal_attention():
    """KV-cache chapter, section 22.7, on the chapter's own sizes (golden): batch 2, 7 tokens,
    3 heads of width 4, float64, atol = rtol = 1e-10; plus a SnapKV-sized case with no
    compression (k = L_prefix) followed by decode steps."""
    g = golden("cached_decode_equivalence.json")
    gen = torch.Generator().manual_seed(22)
    B, T, W, H = g["batch"], g["tokens"], g["model_width"], g["heads"]
    dh = W // H
    x = torch.randn(B, T, W, dtype=torch.float64, generator=gen)
    wq, wk, wv = (torch.randn(W, W, dtype=torch.float64, generator=gen) for _ in range(3))

    def heads(t):
        return t.view(B, T, H, dh).transpose(1, 2).numpy()
    q, k, v = heads(x @ wq), heads(x @ wk), heads(x @ wv)
    for b in range(B):
        for h in range(H):
            worst, shape = pin_decode_vs_full_causal(orc, q[b, h], k[b, h], v[b, h], l_prompt=0)
            assert worst <= g["atol"]
            assert shape == tuple(g["cache_shape"][2:])

    rng = np.random.default_rng(23)
    l_prompt, l_obs, steps, d = 120, 16, 9, 16
    xq, xk, xv = (_rand(rng, l_prompt + steps, d) for _ in range(3))
    res = orc.compress_head(xq[l_prompt - l_obs:l_prompt], xk[:l_prompt], xv[:l_prompt],
                            pool_kernel=7, ratio_p=1.0)
    assert np.array_equal(res.k_c, xk[:l_prompt])
    worst, shape = pin_decode_vs_full_causal(orc, xq, xk, xv, l_prompt)
    assert worst <= 1e-10 and shape == (l_prompt + steps, d)


def test_kv_cache_bytes_matches_worked_example():
    g = golden("kv_cache_memory.json")
    per_token = orc.kv_cache_bytes(g["batch"], 1, g["layers"], g["kv_heads"], g["head_dim"], g["elem_bytes"])
    assert per_token == g["bytes_per_token"]
    assert orc.kv_cache_bytes(g["batch"], g["tokens"], g["layers"], g["kv_heads"], g["head_dim"],
                              g["elem_bytes"]) == g["bytes_at_tokens"]
    for s, b in g["extrapolated"].items():
        assert orc.kv_cache_bytes(1, int(s), 32, 32, 128, 2) == b


# ------------------------------------------------------------------------------------------------
# Hit rate ([SnapKV] Hit Rate（適中率）の定式化)
# ------------------------------------------------------------------------------------------------

def test_hit_count_threshold_zero_counts_every_prefix_position():
    """theta = 0: every prefix weight is positive, so M_threshold covers the prefix and the hits are
    exactly the kept positions."""
    rng = np.random.default_rng(41)
    k = _rand(rng, 40, 16)
    q = _rand(rng, 16)
    idx = np.array([1, 5, 9, 30])
    h = orc.hit_count(q, k, 33, idx, theta=0.0)
    assert (h.total, h.hits) == (33, 4)


def test_hit_count_keeping_the_whole_prefix_hits_everything():
    rng = np.random.default_rng(42)
    k = _rand(rng, 50, 8, scale=3.0)
    q = _rand(rng, 8)
    h = orc.hit_count(q, k, 45, np.arange(45), theta=0.01)
    assert h.total > 0 and h.hits == h.total


def test_hit_count_uniform_weights_and_strict_threshold():
    """q = 0 gives every cached row the weight 1/len exactly (len = 64 is a power of two): the mask
    keeps weights strictly above theta, so theta = 1/len marks nothing and just below it everything."""
    k = np.random.default_rng(43).standard_normal((64, 8))
    q = np.zeros(8)
    assert orc.hit_count(q, k, 60, np.arange(10), theta=1.0 / 64).total == 0
    h = orc.hit_count(q, k, 60, np.arange(10), theta=1.0 / 64 - 1e-12)
    assert (h.total, h.hits) == (60, 10)


def test_hit_count_dominant_key_and_prefix_restriction():
    """One key aligned with a long query takes almost all the weight: it is the only position above
    theta. Inside the prefix it counts (a hit only if kept); in the window it does not count."""
    rng = np.random.default_rng(44)
    d, n, l_prefix = 16, 48, 40
    k = _rand(rng, n, d, scale=0.1)
    q = np.zeros(d)
    q[0] = 50.0
    for jstar, kept, want in [(7, [7, 20], (1, 1)), (7, [3, 20], (0, 1)), (44, [3, 20], (0, 0))]:
        kk = k.copy()
        kk[jstar, 0] = 5.0
        h = orc.hit_count(q, kk, l_prefix, np.array(kept), theta=0.05)
        assert (h.hits, h.total) == want, (jstar, kept)


# ------------------------------------------------------------------------------------------------
# Grouped-query attention (the KV head's vote sums its query heads' votes)
# ------------------------------------------------------------------------------------------------

def test_gqa_single_query_head_is_plain_compression():
    rng = np.random.default_rng(51)
    q, k, v = _rand(rng, 8, 16), _rand(rng, 100, 16), _rand(rng, 100, 16)
    a = orc.compress_kv_head_gqa(q[None], k, v, pool_kernel=5, budget=20)
    b = orc.compress_head(q, k, v, pool_kernel=5, budget=20)
    assert np.array_equal(a.idx, b.idx) and np.allclose(a.c, b.c, rtol=0, atol=0)


def test_gqa_identical_query_heads_scale_the_vote():
    """G copies of one query head: the vote is exactly G times the single head's (a sum of equal
    terms), so pooling and selection are unchanged."""
    rng = np.random.default_rng(52)
    q, k, v = _rand(rng, 8, 16), _rand(rng, 120, 16), _rand(rng, 120, 16)
    one = orc.compress_head(q, k, v, pool_kernel=7, budget=30)
    four = orc.compress_kv_head_gqa(np.stack([q] * 4), k, v, pool_kernel=7, budget=30)
    assert np.allclose(four.c, 4 * one.c, rtol=1e-15, atol=0)
    assert np.array_equal(four.idx, one.idx)


def test_gqa_vote_sum_over_prompt_is_group_times_window():
    """Each query head's rows sum to one over the keys they see, so the group's votes over every
    prompt column sum to G * L_obs (and the prefix columns alone carry less)."""
    rng = np.random.default_rng(53)
    qg, k = _rand(rng, 3, 8, 16, scale=2.0), _rand(rng, 90, 16)
    tot = sum(orc.vote_all_columns(qg[g], k).sum() for g in range(3))
    assert abs(tot - 24.0) < 1e-12
    gq = orc.compress_kv_head_gqa(qg, k, k, pool_kernel=3, budget=10)
    assert gq.c.sum() < 24.0
