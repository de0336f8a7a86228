"""GrowPage's boundary policy in fp64: working sets, decision, kept set.

Test infrastructure only (see the package docstring).

Source: "GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning
Serving", evolve.pub review, Summary -- at each PagedAttention capacity
boundary the Top-p attention working-set sizes induced by the short and the
long query summary are compared; a larger recent (short) working set
allocates one more physical page, otherwise historical KV is compacted within
the current allocation using the maximum of the two importance scores.  The
review's FAQ section gives Top-p 0.99, demand threshold tau = 0 and a local
retention quota of 64 tokens.
"""
from __future__ import annotations

import numpy as np


def softmax(u: np.ndarray) -> np.ndarray:
    """softmax over the last axis in fp64 (max-shifted)."""
    u = np.asarray(u, dtype=np.float64)
    e = np.exp(u - u.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def topp_count(p: np.ndarray, top_p: float) -> int:
    """Top-p working-set size of a probability vector.

    W = min { k : sum of the k largest probabilities >= top_p * sum(p) }.
    Reading: ">=" (the set reaches the mass), ties in value do not change W.
    """
    p = np.asarray(p, dtype=np.float64)
    srt = np.sort(p)[::-1]
    cs = np.cumsum(srt)
    thr = float(top_p) * cs[-1]
    return int(np.searchsorted(cs, thr, side="left")) + 1 if thr > 0 else 1


def topp_range(p: np.ndarray, top_p: float, rel: float = 1e-5):
    """(W at top_p*(1-rel), W at min(1, top_p*(1+rel))): the near-tie band."""
    lo = topp_count(p, top_p * (1.0 - rel))
    hi = topp_count(p, min(1.0, top_p * (1.0 + rel)))
    return lo, hi


def demand_delta(w_short, w_long) -> int:
    """Delta = sum over (layer, kv head) of (W_short - W_long).

    Reading: the pages say only that a larger recent working set triggers
    growth; summing the per-head differences over all layers and kv heads
    gives one signal per request, and any positive normalisation would give
    the same sign at tau = 0.
    """
    return int(np.sum(np.asarray(w_short, dtype=np.int64) - np.asarray(w_long, dtype=np.int64)))


def wants_grow(delta: int, tau: float) -> bool:
    """Grow iff Delta > tau (strict: Delta == 0 compacts)."""
    return float(delta) > float(tau)


def importance(p_short: np.ndarray, p_long: np.ndarray) -> np.ndarray:
    """Per-token importance: the maximum of the two summaries' probabilities."""
    return np.maximum(np.asarray(p_short, np.float64), np.asarray(p_long, np.float64))


def private_importance(u_short: np.ndarray, u_long: np.ndarray, prefix_len: int) -> np.ndarray:
    """Importance of the private tokens from both summaries' scores.

    u_short, u_long: scores of every resident token, prefix first.  Each
    summary's probabilities are one softmax over the whole resident set
    (prefix included: the prefix is part of the attention distribution the
    summary induces); the private tokens' entries are then taken, and the
    importance is the larger of the two probabilities.  Reading: the review's
    Summary says compaction ranks history by "the maximum of both temporal
    importance scores"; normalising each over the same resident set keeps the
    two scores comparable.
    """
    ps = softmax(u_short)[prefix_len:]
    pl = softmax(u_long)[prefix_len:]
    return importance(ps, pl)


def delta_range(band_short: np.ndarray, band_long: np.ndarray):
    """Smallest and largest Delta when every W may take any value of its band.

    band_*: [..., 2] integer (W at Top-p*(1-1e-5), W at Top-p*(1+1e-5)) per
    (layer, kv head).  Delta is smallest with every short W at its low end
    and every long W at its high end, and largest the other way round.
    """
    bs = np.asarray(band_short, dtype=np.int64)
    bl = np.asarray(band_long, dtype=np.int64)
    return int(np.sum(bs[..., 0] - bl[..., 1])), int(np.sum(bs[..., 1] - bl[..., 0]))


def drop_set(imp: np.ndarray, pos: np.ndarray, n_drop: int) -> np.ndarray:
    """Indices of the n_drop candidates ranked lowest by (importance, position).

    Ascending importance; at equal importance the older (smaller position)
    token goes first, i.e. the more recent one is kept.
    """
    order = np.lexsort((np.asarray(pos), np.asarray(imp)))
    return order[:n_drop]


def compaction_plan(imp_priv: np.ndarray, pos_priv: np.ndarray, pos_now: int,
                    capacity: int, page_size: int, recent_window: int, n_free: int = None):
    """Which private tokens a compaction drops, and the near-tie gap at the cut.

    The request holds ``capacity`` private tokens (all its pages full).  It
    keeps capacity - n_free of them (n_free = page_size by default: one
    page-worth of slots free within the same allocation): the most recent
    W = min(recent_window, capacity - n_free) tokens always, plus the best of
    the older ones by importance.  Returns (indices dropped, relative gap at
    the cut or inf).
    """
    n = len(pos_priv)
    assert n == capacity
    if n_free is None:
        n_free = page_size
    w_eff = min(recent_window, capacity - n_free)
    keep_total = capacity - n_free
    recent = pos_priv >= pos_now - w_eff
    assert int(recent.sum()) == w_eff, (int(recent.sum()), w_eff)
    cand = np.nonzero(~recent)[0]
    n_drop = len(cand) - (keep_total - w_eff)
    assert n_drop == n_free
    order = np.lexsort((pos_priv[cand], imp_priv[cand]))
    dropped = cand[order[:n_drop]]
    gap = np.inf
    if len(cand) > n_drop and n_drop > 0:
        a = imp_priv[cand[order[n_drop - 1]]]   # largest dropped
        b = imp_priv[cand[order[n_drop]]]       # smallest kept
        gap = abs(b - a) / max(b, 1e-300)
    return dropped, gap


def may_shrink(pages: int, page_size: int, recent_window: int) -> bool:
    """Whether the SHRINK ablation may release a page at this boundary.

    Reading: the review names a SHRINK ablation (Tables 8-9) that isolates
    "the cost of irreversible shrinking" and gives no rule.  Here, a
    boundary that does not want to grow releases the request's last private
    page instead of compacting in place: it drops two pages' worth of tokens
    by the compaction rule, so that the remaining pages - 1 pages again have
    one page of free slots.  A page is released only while the kept set
    still holds the whole recent window, (pages - 2) * page_size >=
    recent_window; otherwise the boundary compacts as GrowPage does.
    """
    return pages >= 2 and (pages - 2) * page_size >= recent_window


MASK64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    """SplitMix64 output for state x (Steele, Lea and Flood, "Fast splittable
    pseudorandom number generators", OOPSLA 2014), in exact integer arithmetic."""
    z = (x + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def random_grow(slot: int, boundaries_seen: int, rate: float) -> bool:
    """Frequency-matched random policy: grow iff u < rate, u = the top 53
    bits of SplitMix64(slot << 32 | boundaries seen so far) scaled to [0, 1).

    Reading: the review's GROWPAGE-RANDOM (Tables 8-9) draws decisions at the
    measured grow frequency; the pages do not say how, so a counter-based
    generator keyed by the request and its boundary count is used."""
    x = ((slot & 0xFFFFFFFF) << 32) | (boundaries_seen & 0xFFFFFFFF)
    u = (splitmix64(x) >> 11) * 2.0 ** -53
    return u < float(rate)
