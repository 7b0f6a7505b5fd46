"""CPU oracle for SnapKV compression and for decode attention over the compressed cache.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import or run anything under ``oracle/``. The product path (the C-ABI library and its
Python binding) never calls it and shares no code with it.

Plain, slow and literal: numpy in float64, one (layer, sequence, head) at a time, every step in
the order the pages give it. A library primitive (matmul, exp, max, sort) serves as a step; there
is no tiling, fusion or reordering.

Sources (page title, section / equation):
  [SnapKV]   "論文解説: SnapKV — アテンションパターン観測によるKVキャッシュ圧縮"
             (0h-n0.github.io, posts/paper-2404-14469): sections プロンプトの分割 (prompt split),
             投票メカニズム (vote C = sum_i W_obs[:, i, :], I = Top_k(C, k), k = floor(p L_prefix)),
             クラスタリングによる文脈保持 (1D max pooling before top-k), アルゴリズム (the
             restated Algorithm 1: softmax of Q_obs K^T / sqrt(d_k), sum over the window rows,
             max_pool1d(kernel, padding=kernel//2, stride=1), k = min(max_cap, L_prefix),
             ascending indices, per-head gather, concatenation with the window),
             実装のポイント (per-head independent selection).
  [KVcache]  "第22章 KV Cache" (waylandz.com, llm-transformer-book-ja/chapter-22-kv-cache):
             section 22.2 (append K_cache <- [K_cache; k_t], o_t = softmax(q_t K_cache^T / sqrt(d_h))
             V_cache, every cached position visible), 22.4 (M_KV = 2 B S L H_KV d_h b),
             22.7 (cached decode equals full causal attention, float64, atol = rtol = 1e-10).

Readings where the pages are open:
  * Softmax scope: rows are normalised over every prompt column the window query can see (all
    prefix columns plus the window columns up to and including its own position); the vote keeps
    the prefix columns. The restated listing normalises over the prefix columns only; that
    variant is kept as ``scope=PREFIX_ONLY``.
  * The vote sums exactly L_obs rows (the printed upper bound of the sum is off by one).
  * k = floor(p * L_prefix) evaluated in IEEE double, or min(budget, L_prefix) with a fixed budget.
  * Max-pool padding is -inf, so the window is clipped to [0, L_prefix); the kernel is odd.
  * Top-k ties go to the lower index; the kept indices are emitted in ascending order, then the
    window rows follow in their original order.

Every function below is pinned by a ``-m "not gpu"`` test against something other than itself
(closed forms, invariants, torch library routines, brute-force enumeration, the KV-cache
chapter's equivalence check); none is "parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

PROMPT_CAUSAL = "prompt_causal"
PREFIX_ONLY = "prefix_only"


def prefix_length(l_prompt: int, l_obs: int) -> int:
    """[SnapKV] プロンプトの分割: L_prompt = L_prefix + L_obs; the window is the last L_obs tokens."""
    if not (1 <= l_obs < l_prompt):
        raise ValueError(f"need 1 <= L_obs < L_prompt (got L_obs={l_obs}, L_prompt={l_prompt})")
    return l_prompt - l_obs


def kept_slots(l_prefix: int, ratio_p: float = 0.0, budget: int = 0) -> int:
    """Number k of prefix positions kept per head.

    [SnapKV] 投票メカニズム: k = floor(p * L_prefix); アルゴリズム: k = min(max_cap, L_prefix) with a
    fixed per-head budget. ``budget > 0`` selects the budget form.
    """
    if budget > 0:
        return min(int(budget), int(l_prefix))
    if not (0.0 <= ratio_p <= 1.0):
        raise ValueError("p must lie in [0, 1]")
    return int(math.floor(ratio_p * float(l_prefix)))


def window_logits(q_obs: np.ndarray, k: np.ndarray) -> np.ndarray:
    """s_ij = (q_i . k_j) / sqrt(d) for every window query i and prompt key j ([L_obs, L_prompt]).

    [SnapKV] アルゴリズム: matmul(q_obs, k^T) / d_k ** 0.5.
    """
    q64 = np.asarray(q_obs, dtype=np.float64)
    k64 = np.asarray(k, dtype=np.float64)
    return (q64 @ k64.T) / math.sqrt(q64.shape[1])


def visible(l_obs: int, l_prompt: int, scope: str = PROMPT_CAUSAL) -> np.ndarray:
    """Mask of the (i, j) pairs that enter row i's softmax ([L_obs, L_prompt] bool).

    PROMPT_CAUSAL: window query i sits at prompt position L_prefix + i and sees j <= L_prefix + i.
    PREFIX_ONLY: every row sees exactly the prefix columns j < L_prefix (the restated listing).
    """
    l_prefix = prefix_length(l_prompt, l_obs)
    i = np.arange(l_obs)[:, None]
    j = np.arange(l_prompt)[None, :]
    if scope == PROMPT_CAUSAL:
        return j <= l_prefix + i
    if scope == PREFIX_ONLY:
        return np.broadcast_to(j < l_prefix, (l_obs, l_prompt)).copy()
    raise ValueError(f"unknown softmax scope {scope!r}")


def window_weights(q_obs: np.ndarray, k: np.ndarray, scope: str = PROMPT_CAUSAL) -> np.ndarray:
    """W[i, j] = exp(s_ij - m_i) / Z_i on visible (i, j), 0 elsewhere ([L_obs, L_prompt]).

    m_i = max of row i's visible logits, Z_i = sum of exp(s_ij - m_i) over them.
    """
    s = window_logits(q_obs, k)
    mask = visible(s.shape[0], s.shape[1], scope)
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.where(mask, np.exp(s - m), 0.0)
    z = e.sum(axis=1, keepdims=True)
    return e / z


def vote_all_columns(q_obs: np.ndarray, k: np.ndarray, scope: str = PROMPT_CAUSAL) -> np.ndarray:
    """Column sums of W over the L_obs window rows for every prompt column ([L_prompt])."""
    return window_weights(q_obs, k, scope).sum(axis=0)


def vote(q_obs: np.ndarray, k: np.ndarray, scope: str = PROMPT_CAUSAL) -> np.ndarray:
    """[SnapKV] 投票メカニズム: C_j = sum over the L_obs window rows i of W_obs[i, j], j < L_prefix."""
    l_prefix = prefix_length(k.shape[0], q_obs.shape[0])
    return vote_all_columns(q_obs, k, scope)[:l_prefix]


def max_pool(c: np.ndarray, kernel: int) -> np.ndarray:
    """[SnapKV] クラスタリングによる文脈保持: P_j = max of C over |j' - j| <= kernel // 2.

    Stride 1, padding kernel // 2 filled with -inf, so the window is clipped to the valid range
    and the output has the input's length. The kernel must be odd.
    """
    if kernel < 1 or kernel % 2 == 0:
        raise ValueError("pool kernel must be odd and >= 1")
    c = np.asarray(c, dtype=np.float64)
    r = kernel // 2
    n = c.shape[0]
    padded = np.concatenate([np.full(r, -np.inf), c, np.full(r, -np.inf)])
    out = np.full(n, -np.inf)
    for shift in range(kernel):
        out = np.maximum(out, padded[shift:shift + n])
    return out


def select_by_rank(p: np.ndarray, k: int) -> np.ndarray:
    """Top-k by its definition: rank_j = #{P_j' > P_j} + #{j' < j : P_j' = P_j}; keep rank_j < k.

    Ties go to the lower index. O(L^2); for small inputs. Returns the kept indices ascending.
    """
    p = np.asarray(p, dtype=np.float64)
    n = p.shape[0]
    idx = np.arange(n)
    rank = np.empty(n, dtype=np.int64)
    block = 2048
    for s in range(0, n, block):
        pj = p[s:s + block, None]
        jj = idx[s:s + block, None]
        rank[s:s + block] = (p[None, :] > pj).sum(axis=1) + ((p[None, :] == pj) & (idx[None, :] < jj)).sum(axis=1)
    return np.nonzero(rank < k)[0].astype(np.int64)


def select_by_sort(p: np.ndarray, k: int) -> np.ndarray:
    """Top-k by a stable order on (-P_j, j): the first k positions, returned ascending."""
    p = np.asarray(p, dtype=np.float64)
    order = np.lexsort((np.arange(p.shape[0]), -p))
    return np.sort(order[:k]).astype(np.int64)


def select_topk(p: np.ndarray, k: int) -> np.ndarray:
    """[SnapKV] I = Top_k(P, k), lower index first on ties, emitted ascending."""
    if not (0 <= k <= p.shape[0]):
        raise ValueError("k out of range")
    return select_by_rank(p, k) if p.shape[0] <= 4096 else select_by_sort(p, k)


def kth_largest(p: np.ndarray, k: int) -> float:
    """tau = the k-th largest pooled value (k >= 1)."""
    return float(np.sort(np.asarray(p, dtype=np.float64))[::-1][k - 1])


def gather_with_window(x: np.ndarray, idx: np.ndarray, l_prefix: int) -> np.ndarray:
    """[SnapKV] アルゴリズム: [x[idx]; x[L_prefix:L_prompt]] — kept prefix rows, then the window."""
    x = np.asarray(x)
    return np.concatenate([x[np.asarray(idx, dtype=np.int64)], x[l_prefix:]], axis=0)


@dataclass
class Compressed:
    c: np.ndarray        # vote over the prefix columns, float64 [L_prefix]
    p: np.ndarray        # pooled vote, float64 [L_prefix]
    idx: np.ndarray      # kept prefix positions, ascending, int64 [k]
    tau: float           # k-th largest pooled value (nan when k == 0)
    k_c: np.ndarray      # [k + L_obs, d] compressed keys (input dtype)
    v_c: np.ndarray      # [k + L_obs, d] compressed values


def compress_head(q_obs: np.ndarray, k: np.ndarray, v: np.ndarray, *, pool_kernel: int,
                  ratio_p: float = 0.0, budget: int = 0, scope: str = PROMPT_CAUSAL) -> Compressed:
    """SnapKV compression of one (layer, sequence, head), every step in the pages' order.

    q_obs: the L_obs window queries [L_obs, d]; k, v: the whole prompt [L_prompt, d].
    """
    l_obs = q_obs.shape[0]
    l_prefix = prefix_length(k.shape[0], l_obs)
    k_sel = kept_slots(l_prefix, ratio_p, budget)
    c = vote(q_obs, k, scope)
    p = max_pool(c, pool_kernel)
    idx = select_topk(p, k_sel)
    tau = kth_largest(p, k_sel) if k_sel > 0 else float("nan")
    return Compressed(c=c, p=p, idx=idx, tau=tau, k_c=gather_with_window(k, idx, l_prefix),
                      v_c=gather_with_window(v, idx, l_prefix))


def compress_kv_head_gqa(q_obs_group: np.ndarray, k: np.ndarray, v: np.ndarray, *, pool_kernel: int,
                         ratio_p: float = 0.0, budget: int = 0, scope: str = PROMPT_CAUSAL) -> Compressed:
    """SnapKV compression of one KV head shared by G query heads (grouped-query attention).

    The pages are silent on grouped heads; the reading taken: every query head of the group votes
    with its own row softmax over the shared keys, the KV head's vote is the sum of the G votes,
    and pooling, selection and gather then run once on the KV head as for a single head.
    q_obs_group: [G, L_obs, d] window queries of the group; k, v: the KV head's prompt [L_prompt, d].
    """
    l_obs = q_obs_group.shape[1]
    l_prefix = prefix_length(k.shape[0], l_obs)
    k_sel = kept_slots(l_prefix, ratio_p, budget)
    c = np.zeros(l_prefix)
    for g in range(q_obs_group.shape[0]):
        c = c + vote(q_obs_group[g], k, scope)
    p = max_pool(c, pool_kernel)
    idx = select_topk(p, k_sel)
    tau = kth_largest(p, k_sel) if k_sel > 0 else float("nan")
    return Compressed(c=c, p=p, idx=idx, tau=tau, k_c=gather_with_window(k, idx, l_prefix),
                      v_c=gather_with_window(v, idx, l_prefix))


def append(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray, v_new: np.ndarray):
    """[KVcache] 22.2: K_cache <- [K_cache; k_t], V_cache <- [V_cache; v_t]."""
    return (np.concatenate([k_cache, np.asarray(k_new)[None, :]], axis=0),
            np.concatenate([v_cache, np.asarray(v_new)[None, :]], axis=0))


def decode_attend(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray) -> np.ndarray:
    """[KVcache] 22.2: o = softmax(q K_cache^T / sqrt(d_h)) V_cache over every cached row (float64)."""
    q64 = np.asarray(q, dtype=np.float64)
    s = (np.asarray(k_cache, dtype=np.float64) @ q64) / math.sqrt(q64.shape[0])
    w = np.exp(s - s.max())
    w = w / w.sum()
    return w @ np.asarray(v_cache, dtype=np.float64)


@dataclass
class HitCount:
    hits: int       # sum of O = M_threshold AND M_vote over the prefix positions
    total: int      # sum of M_threshold
    weights: np.ndarray   # A_cur over the prefix positions (float64), for boundary checks


def hit_count(q: np.ndarray, k_cache: np.ndarray, l_prefix: int, idx: np.ndarray, theta: float = 0.05) -> HitCount:
    """[SnapKV] Hit Rate（適中率）の定式化, for one head and one generation-time query.

    A_cur is the query's attention over every cached row (softmax of q K^T / sqrt(d), the decode
    attention of [KVcache] 22.2) taken at the prefix positions j < l_prefix; M_threshold marks
    A_cur > theta, M_vote marks the kept positions idx, O = M_threshold AND M_vote, and the hit
    rate is H = sum(O) / sum(M_threshold) (summed over heads by the caller).
    """
    q64 = np.asarray(q, dtype=np.float64)
    s = (np.asarray(k_cache, dtype=np.float64) @ q64) / math.sqrt(q64.shape[0])
    w = np.exp(s - s.max())
    w = w / w.sum()
    a_cur = w[:l_prefix]
    m_thr = a_cur > theta
    m_vote = np.zeros(a_cur.shape[0], dtype=bool)
    m_vote[np.asarray(idx, dtype=np.int64)] = True
    return HitCount(hits=int(np.sum(m_thr & m_vote)), total=int(np.sum(m_thr)), weights=a_cur)


def kv_cache_bytes(batch: int, seq: int, layers: int, kv_heads: int, head_dim: int,
                   elem_bytes: int) -> int:
    """[KVcache] 22.4: M_KV = 2 B S L H_KV d_h b (dense cache, keys and values)."""
    return 2 * batch * seq * layers * kv_heads * head_dim * elem_bytes
