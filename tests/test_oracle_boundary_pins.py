"""Pins of the oracle's boundary wiring: how ``OraclePool.step`` assembles
the summary scores, the importance used by compaction and the near-tie
exemption of a decision.

Source: "GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning
Serving", evolve.pub review, Summary -- Top-p working sets of the short and
the long query summary (kept pre-RoPE) are compared at each capacity
boundary; compaction keeps history by the maximum of both importance scores.

Each pin recomputes one piece from its definition, with code that shares
nothing with the oracle: rotary embedding by complex multiplication, the EMA
by its closed form, Top-p by a plain sort, the kept set by ranking Python
tuples, the exemption by enumerating every combination of working-set sizes
inside their bands.  Each pin is paired with a test that plants the
plausible mistake in the oracle (on the CPU) and shows that the pin fails.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import policy as pol
from oracle.pool import OracleConfig, OraclePool, COMPACT, GROW, STARVED


def _rope_c(x, pos, theta):
    """Rotate-half RoPE of the last axis by complex multiplication (fp64)."""
    x = np.asarray(x, dtype=np.float64)
    if theta == 0.0:
        return x.copy()
    d = x.shape[-1]
    h = d // 2
    w = np.exp(-np.arange(h) * 2.0 / d * np.log(theta))
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * pos * w)
    return np.concatenate([z.real, z.imag], axis=-1)


def _probs(u):
    e = np.exp(np.asarray(u, np.float64) - np.max(u))
    return e / e.sum()


def _topp_sorted(p, top_p):
    """Smallest k whose k largest probabilities reach top_p of the mass."""
    srt = sorted((float(x) for x in p), reverse=True)
    tot = sum(srt)
    acc = 0.0
    for k, x in enumerate(srt, 1):
        acc += x
        if acc >= top_p * tot:
            return k
    return len(srt)


def _ema_closed_form(qbars, beta):
    """s_t = beta^(t-1) qbar_1 + (1 - beta) sum_{s >= 2} beta^(t-s) qbar_s."""
    t = len(qbars)
    s = beta ** (t - 1) * qbars[0]
    for j in range(1, t):
        s = s + (1.0 - beta) * beta ** (t - 1 - j) * qbars[j]
    return s


class _Tracker:
    """Drives one request through an OraclePool and keeps, independently of
    the pool, the raw inputs: resident keys with their positions, and the
    query group means of every step."""

    def __init__(self, cfg, prefix_k, prompt_k, budget, keep_logits=True):
        L, hk, d = cfg.num_layers, cfg.num_kv_heads, cfg.head_dim
        self.cfg = cfg
        self.pool = OraclePool(cfg, keep_logits=keep_logits)
        plen = 0 if prefix_k is None else prefix_k.shape[1]
        pid = -1
        if prefix_k is not None:
            pid = self.pool.add_prefix(prefix_k, np.zeros_like(prefix_k))
        n = prompt_k.shape[1]
        self.pool.add_request(0, prompt_k, np.zeros_like(prompt_k), budget, pid)
        # stored keys by position: [L][Hk][d] each
        self.keys = {}
        for j in range(plen):
            self.keys[j] = _rope_c(prefix_k[:, j], j, cfg.rope_theta)
        for j in range(n):
            self.keys[plen + j] = _rope_c(prompt_k[:, j], plen + j, cfg.rope_theta)
        self.plen = plen
        self.pos = plen + n
        self.qbars = []          # [L][Hk][d] fp64 per step

    def step(self, q, k):
        """q [L][Hq][d], k [L][Hk][d] raw; returns (record or None, pos_t)."""
        cfg = self.cfg
        L, hk, d = cfg.num_layers, cfg.num_kv_heads, cfg.head_dim
        G = cfg.num_q_heads // hk
        pos_t = self.pos
        self.qbars.append(np.asarray(q, np.float32).astype(np.float64)
                          .reshape(L, hk, G, d).mean(axis=2))
        res = self.pool.step([0], q[None], k[None], np.zeros((1, L, hk, d)))
        self.keys[pos_t] = _rope_c(k, pos_t, cfg.rope_theta)
        self.pos += 1
        return res["records"].get(0), pos_t

    def summaries(self):
        """(short, long) summaries after the last step, fp64 closed forms."""
        bs = float(np.float32(self.cfg.beta_s))
        bl = float(np.float32(self.cfg.beta_l))
        return _ema_closed_form(self.qbars, bs), _ema_closed_form(self.qbars, bl)

    def scores(self, positions, pos_t):
        """u[l][g][X][j] = RoPE(s_X, pos_t) . k_j / sqrt(d) over `positions`."""
        cfg = self.cfg
        d = cfg.head_dim
        K = np.stack([self.keys[p] for p in positions], axis=2)      # [L][Hk][R][d]
        out = []
        for s in self.summaries():
            sr = _rope_c(s, pos_t, cfg.rope_theta)                   # [L][Hk][d]
            out.append(np.einsum("lgrd,lgd->lgr", K, sr) / math.sqrt(d))
        return np.stack(out, axis=2)                                 # [L][Hk][2][R]


def _expected_kept(u_short, u_long, positions, plen, pos_t, capacity, page_size, window):
    """Private positions kept by a compaction, from the definition: each
    summary's probabilities over the whole resident set, importance = the
    larger one, the most recent min(window, capacity - P) private tokens
    always, then the best older ones by (importance, position)."""
    ps, pl = _probs(u_short), _probs(u_long)
    priv = [(positions[j], max(ps[j], pl[j])) for j in range(plen, len(positions))]
    keep_n = capacity - page_size
    w_eff = min(window, keep_n)
    recent = {p for p, _ in priv if p >= pos_t - w_eff}
    older = sorted(((imp, p) for p, imp in priv if p not in recent), reverse=True)
    kept = set(recent) | {p for _, p in older[:keep_n - w_eff]}
    gap = np.inf
    if len(older) > keep_n - w_eff > 0:
        a, b = older[keep_n - w_eff - 1][0], older[keep_n - w_eff][0]
        gap = abs(a - b) / max(a, 1e-300)
    return kept, gap


# ------------------------------------------------ summary scores (A4) ----

def _scenario_scores(seed=0):
    """One layer, 2 kv heads x 2 query heads, d = 32, RoPE theta 1e4; a
    16-token prefix and a 20-token prompt in 2 pages of 16: the request's
    private pages fill after 12 steps, so step 13 is its first boundary.
    beta_S = 0 (the short summary is the step's query mean) and beta_L = 0.5;
    tau is huge, so the boundary compacts."""
    cfg = OracleConfig(num_layers=1, num_q_heads=4, num_kv_heads=2, head_dim=32, page_size=16,
                       num_pages=64, max_pages_per_req=8, dtype="f32", rope_theta=10000.0,
                       top_p=0.9, recent_window=4, beta_s=0.0, beta_l=0.5, tau=1e9)
    rng = np.random.default_rng(seed)
    L, hk, hq, d = 1, 2, 4, 32
    tr = _Tracker(cfg, rng.standard_normal((L, 16, hk, d)), rng.standard_normal((L, 20, hk, d)), 2)
    for t in range(13):
        q = 2.0 * rng.standard_normal((L, hq, d))
        k = rng.standard_normal((L, hk, d))
        rec, pos_t = tr.step(q, k)
        if rec is not None:
            return tr, rec, pos_t
    raise AssertionError("no boundary")


def _check_scores(tr, rec, pos_t):
    """The pin: the oracle's boundary scores, working sets and kept set equal
    their recomputation from the definition."""
    cfg = tr.cfg
    positions = list(range(pos_t))           # prefix + private; the staged token excluded
    assert rec.logits.shape[-1] == len(positions)
    u = tr.scores(positions, pos_t)
    scale = np.max(np.abs(u))
    assert np.max(np.abs(rec.logits - u)) <= 1e-5 * scale
    for g in range(cfg.num_kv_heads):
        for X, W in ((0, rec.w_short), (1, rec.w_long)):
            if not rec.w_near_tie[0, g, X]:
                assert W[0, g] == _topp_sorted(_probs(u[0, g, X]), cfg.top_p)
    assert rec.decision == COMPACT
    kp = tr.pool.kept_positions(0)
    for g in range(cfg.num_kv_heads):
        kept, gap = _expected_kept(u[0, g, 0], u[0, g, 1], positions, tr.plen, pos_t,
                                   2 * cfg.page_size, cfg.page_size, cfg.recent_window)
        assert gap > 1e-5
        assert sorted(kept | {pos_t}) == kp[0, g].tolist()


def test_summary_scores_rotated_to_current_position():
    tr, rec, pos_t = _scenario_scores()
    assert pos_t == 16 + 20 + 12
    _check_scores(tr, rec, pos_t)


@pytest.mark.parametrize("mistake", ["unrotated", "previous_position", "unscaled"])
def test_score_pin_fails_on_a_planted_mistake(monkeypatch, mistake):
    # the plausible mistakes in assembling the scores, planted in the oracle:
    # each makes the pin above fail
    def planted(self, Kres, s, pos_t, scale):
        s64 = np.asarray(s, np.float64)
        if mistake == "unrotated":
            sr = s64
        elif mistake == "previous_position":
            sr = _rope_c(s64, pos_t - 1, self.cfg.rope_theta)
        else:
            sr, scale = _rope_c(s64, pos_t, self.cfg.rope_theta), 1.0
        return np.matmul(Kres, sr[:, :, None])[:, :, 0] * scale

    monkeypatch.setattr(OraclePool, "_summary_scores", planted)
    tr, rec, pos_t = _scenario_scores()
    with pytest.raises(AssertionError):
        _check_scores(tr, rec, pos_t)


# --------------------------------------- importance normalisation (A8) ----

def _scenario_importance():
    """No RoPE, one kv head, d = 16.  Steps 1..12 query along A, step 13 along
    B (A orthogonal to B); the 16 prefix keys lie along B.  The short summary
    (beta 0: the step's query) puts almost all its mass on the prefix, the
    long one (beta 0.9) little.  Normalised over prefix + private, the private
    tokens' short probabilities are tiny and their ranking follows the long
    summary; normalised over the private tokens alone it would not."""
    cfg = OracleConfig(num_layers=1, num_q_heads=1, num_kv_heads=1, head_dim=16, page_size=16,
                       num_pages=64, max_pages_per_req=8, dtype="f32", rope_theta=0.0,
                       top_p=0.9, recent_window=4, beta_s=0.0, beta_l=0.9, tau=1e9)
    rng = np.random.default_rng(3)
    d = 16
    A = np.zeros(d); A[0] = 1.0
    B = np.zeros(d); B[1] = 1.0
    pre = 3.0 * B[None, None, None, :] + 0.1 * rng.standard_normal((1, 16, 1, d))
    prompt = rng.standard_normal((1, 20, 1, d))
    tr = _Tracker(cfg, pre, prompt, 2)
    for t in range(13):
        q = (3.0 * (B if t == 12 else A) + 0.3 * rng.standard_normal(d))[None, None, :]
        rec, pos_t = tr.step(q, rng.standard_normal((1, 1, d)))
        if rec is not None:
            return tr, rec, pos_t
    raise AssertionError("no boundary")


def _private_only_kept(u_short, u_long, positions, plen, pos_t, capacity, P, window):
    """The kept set if each summary were normalised over private tokens only."""
    big = 1e9
    us = np.concatenate([np.full(plen, -big), u_short[plen:]])
    ul = np.concatenate([np.full(plen, -big), u_long[plen:]])
    return _expected_kept(us, ul, positions, plen, pos_t, capacity, P, window)[0]


def _check_importance(tr, rec, pos_t):
    cfg = tr.cfg
    positions = list(range(pos_t))
    u = tr.scores(positions, pos_t)
    kept, gap = _expected_kept(u[0, 0, 0], u[0, 0, 1], positions, tr.plen, pos_t, 32,
                               cfg.page_size, cfg.recent_window)
    assert gap > 1e-5
    assert sorted(kept | {pos_t}) == tr.pool.kept_positions(0)[0, 0].tolist()


def test_importance_normalised_over_prefix_and_private():
    tr, rec, pos_t = _scenario_importance()
    assert rec.decision == COMPACT and tr.plen == 16
    positions = list(range(pos_t))
    u = tr.scores(positions, pos_t)
    # the scenario discriminates: the other normalisation keeps another set
    right = _expected_kept(u[0, 0, 0], u[0, 0, 1], positions, 16, pos_t, 32, 16, 4)[0]
    wrong = _private_only_kept(u[0, 0, 0], u[0, 0, 1], positions, 16, pos_t, 32, 16, 4)
    assert right != wrong
    _check_importance(tr, rec, pos_t)


def test_importance_pin_fails_on_private_only_normalisation(monkeypatch):
    def planted(u_short, u_long, prefix_len):
        return pol.importance(pol.softmax(np.asarray(u_short)[prefix_len:]),
                              pol.softmax(np.asarray(u_long)[prefix_len:]))

    monkeypatch.setattr(pol, "private_importance", planted)
    tr, rec, pos_t = _scenario_importance()
    with pytest.raises(AssertionError):
        _check_importance(tr, rec, pos_t)


# ------------------------------------------------ near-tie exemption ----

def _scenario_band(seed):
    """No RoPE, 2 kv heads (one query head each), d = 16, Top-p 0.5, a
    20-token prompt in 2 pages: first boundary at step 13 with 32 resident
    tokens.  Every key of head 0 is the same vector, so both summaries see
    uniform scores over 32 tokens: Top-p 0.5 is reached exactly at 16 tokens
    and W sits on a tie (band 16..17).  Head 1 has random keys; for even
    seeds every step has the same query, so both summaries stay (nearly)
    equal and head 1 adds little to Delta."""
    cfg = OracleConfig(num_layers=1, num_q_heads=2, num_kv_heads=2, head_dim=16, page_size=16,
                       num_pages=64, max_pages_per_req=8, dtype="f32", rope_theta=0.0,
                       top_p=0.5, recent_window=4, beta_s=0.9, beta_l=0.999, tau=0.0)
    rng = np.random.default_rng(100 + seed)
    d = 16
    k0 = rng.standard_normal(d)
    prompt = rng.standard_normal((1, 20, 2, d))
    prompt[0, :, 0] = k0
    tr = _Tracker(cfg, None, prompt, 2)
    q_const = 2.0 * rng.standard_normal((1, 2, d))
    for t in range(13):
        q = q_const if seed % 2 == 0 else 2.0 * rng.standard_normal((1, 2, d))
        k = rng.standard_normal((1, 2, d))
        k[0, 0] = k0
        rec, pos_t = tr.step(q, k)
        if rec is not None:
            return tr, rec, pos_t
    raise AssertionError("no boundary")


def _band(p, top_p, rel=1e-5):
    return _topp_sorted(p, top_p * (1 - rel)), _topp_sorted(p, min(1.0, top_p * (1 + rel)))


def _exempt_brute(bands, tau):
    """Whether the grow decision (Delta > tau) can come out both ways when
    every W takes any value inside its band: all combinations enumerated."""
    ranges = [range(lo, hi + 1) for lo, hi in bands]
    outcomes = set()
    for combo in itertools.product(*ranges):
        delta = sum(combo[0::2]) - sum(combo[1::2])   # (short, long) per head, in order
        outcomes.add(delta > tau)
    return len(outcomes) > 1


def _check_exemption(tr, rec, pos_t):
    """Returns the brute-force exemption; asserts the oracle agrees."""
    cfg = tr.cfg
    u = tr.scores(list(range(pos_t)), pos_t)
    bands = []
    for g in range(2):
        for X in (0, 1):
            b = _band(_probs(u[0, g, X]), cfg.top_p)
            assert tuple(rec.w_band[0, g, X]) == b
            bands.append(b)
    assert bands[0] == bands[1] == (16, 17)       # head 0: uniform scores, on the tie
    ex = _exempt_brute(bands, cfg.tau)
    assert rec.decision_exempt == ex
    return ex


def test_near_tie_exemption_matches_enumeration():
    seen = set()
    for seed in range(12):
        tr, rec, pos_t = _scenario_band(seed)
        seen.add(_check_exemption(tr, rec, pos_t))
    assert seen == {True, False}   # both outcomes occur among the cases


def test_exemption_pin_fails_on_a_planted_mistake(monkeypatch):
    # the band ends paired the wrong way round (short low with long low)
    def planted(band_short, band_long):
        bs, bl = np.asarray(band_short), np.asarray(band_long)
        return int(np.sum(bs[..., 0] - bl[..., 0])), int(np.sum(bs[..., 1] - bl[..., 1]))

    monkeypatch.setattr(pol, "delta_range", planted)
    failed = 0
    for seed in range(12):
        tr, rec, pos_t = _scenario_band(seed)
        try:
            _check_exemption(tr, rec, pos_t)
        except AssertionError:
            failed += 1
    assert failed > 0


# ---------------------------------------------------- full-KV page cap ----

def test_full_kv_stops_at_the_page_cap():
    # full KV with a cap of 3 private pages: the first boundary grows to 3,
    # every later one cannot grow and drops its token (starved), exactly as a
    # boundary with no free page does
    cfg = OracleConfig(num_layers=1, num_q_heads=2, num_kv_heads=1, head_dim=16, page_size=16,
                       num_pages=64, max_pages_per_req=3, dtype="f32", rope_theta=0.0,
                       top_p=0.9, recent_window=4, full_kv=True)
    rng = np.random.default_rng(7)
    pool = OraclePool(cfg)
    pool.add_request(0, rng.standard_normal((1, 32, 1, 16)), rng.standard_normal((1, 32, 1, 16)), 2)
    decs = []
    for t in range(60):
        res = pool.step([0], rng.standard_normal((1, 1, 2, 16)), rng.standard_normal((1, 1, 1, 16)),
                        rng.standard_normal((1, 1, 1, 16)))
        pool.check_invariants()
        if 0 in res["records"]:
            decs.append((t, res["records"][0].decision))
    r = pool.req[0]
    assert decs[0] == (0, GROW)
    assert [d for _, d in decs[1:]] == [STARVED] * (len(decs) - 1) and len(decs) > 10
    assert len(r.pages) == 3 and r.toks.n == 48 and r.pos == 32 + 60
    assert pool.starved == len(decs) - 1 and len(pool.free) == 61
