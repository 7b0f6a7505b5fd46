"""Plant a mistake in the oracle (on the CPU, via monkeypatch) and check that a pin catches it.

Shows that the pins in test_oracle_pins.py are sensitive to the plausible mistakes: a dropped
scale, an off-by-one causal mask, a wrong pool radius, the wrong tie rule, a wrong sum bound,
a transposed decode operand, an inclusive hit-rate threshold, hit-rate attention counted
outside the prefix.
"""
import math

import numpy as np

from oracle import snapkv_oracle as orc
from tests import test_oracle_pins as pins


def _case(seed=0, l_prompt=90, l_obs=16, d=8):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((l_prompt, d)) * 1.5, rng.standard_normal((l_prompt, d)), l_obs


def test_dropped_scale_is_caught(monkeypatch):
    q_all, k, l_obs = _case()
    monkeypatch.setattr(orc, "window_logits", lambda q, kk: np.asarray(q, float) @ np.asarray(kk, float).T)
    assert pins.pin_weights_vs_sdpa(orc, q_all, k, l_obs) > 1e-3


def test_off_by_one_causal_mask_is_caught(monkeypatch):
    q_all, k, l_obs = _case(1)

    def bad_visible(lo, lp, scope=orc.PROMPT_CAUSAL):
        i = np.arange(lo)[:, None]
        j = np.arange(lp)[None, :]
        return j < (lp - lo) + i if scope == orc.PROMPT_CAUSAL else j < lp - lo
    # a query that cannot see itself: rows i >= 1 differ (row 0 keeps the full prefix)
    monkeypatch.setattr(orc, "visible", bad_visible)
    assert pins.pin_weights_vs_sdpa(orc, q_all, k, l_obs) > 1e-3


def test_wrong_pool_radius_is_caught(monkeypatch):
    c = np.random.default_rng(2).random(60)
    real = orc.max_pool
    monkeypatch.setattr(orc, "max_pool", lambda x, kernel: real(x, max(1, kernel - 2)))
    assert pins.pin_pool_vs_torch(orc, c, 7) > 0.0


def test_wrong_tie_rule_is_caught(monkeypatch):
    def upper_index_first(p, k):
        p = np.asarray(p, float)
        order = np.lexsort((-np.arange(p.shape[0]), -p))
        return np.sort(order[:k])
    monkeypatch.setattr(orc, "select_topk", upper_index_first)
    p = np.array([1.0, 2.0, 2.0, 0.0, 2.0])
    assert orc.select_topk(p, 2).tolist() != pins.brute_force_topk(p.tolist(), 2).tolist()


def test_short_vote_sum_is_caught(monkeypatch):
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((16, 8)), rng.standard_normal((100, 8))
    monkeypatch.setattr(orc, "vote_all_columns",
                        lambda qq, kk, scope=orc.PROMPT_CAUSAL: orc.window_weights(qq, kk, scope)[:-1].sum(axis=0))
    assert abs(orc.vote_all_columns(q, k).sum() - 16) > 0.5


def test_transposed_decode_operand_is_caught(monkeypatch):
    rng = np.random.default_rng(4)
    x = [rng.standard_normal((12, 12)) for _ in range(3)]

    def bad_decode(q, kc, vc):
        s = (np.asarray(vc) @ q) / math.sqrt(q.shape[0])      # values used as keys
        w = np.exp(s - s.max())
        return (w / w.sum()) @ np.asarray(kc)
    monkeypatch.setattr(orc, "decode_attend", bad_decode)
    worst, _ = pins.pin_decode_vs_full_causal(orc, x[0], x[1], x[2], l_prompt=3)
    assert worst > 1e-3


def _hit_count_variant(inclusive=False, whole_cache=False):
    """hit_count with a planted mistake: >= theta instead of > theta, or no restriction to the prefix."""
    def bad(q, k_cache, l_prefix, idx, theta=0.05):
        q64 = np.asarray(q, dtype=np.float64)
        s = (np.asarray(k_cache, dtype=np.float64) @ q64) / math.sqrt(q64.shape[0])
        w = np.exp(s - s.max())
        w = w / w.sum()
        a_cur = w if whole_cache else w[:l_prefix]
        m_thr = a_cur >= theta if inclusive else a_cur > theta
        m_vote = np.zeros(a_cur.shape[0], dtype=bool)
        m_vote[np.asarray(idx, dtype=np.int64)] = True
        return orc.HitCount(hits=int(np.sum(m_thr & m_vote)), total=int(np.sum(m_thr)), weights=a_cur)
    return bad


def test_inclusive_hit_threshold_is_caught(monkeypatch):
    monkeypatch.setattr(orc, "hit_count", _hit_count_variant(inclusive=True))
    try:
        pins.test_hit_count_uniform_weights_and_strict_threshold()
    except AssertionError:
        return
    raise AssertionError("the pin did not catch an inclusive threshold")


def test_hit_count_over_the_window_is_caught(monkeypatch):
    monkeypatch.setattr(orc, "hit_count", _hit_count_variant(whole_cache=True))
    try:
        pins.test_hit_count_dominant_key_and_prefix_restriction()
    except AssertionError:
        return
    raise AssertionError("the pin did not catch attention counted outside the prefix")
