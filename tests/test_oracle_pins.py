"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one oracle function against mathematics or an independent
library routine: closed forms, brute force on tiny inputs, exact rational
rounding, torch's own SDPA.  None of them needs a GPU.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import numerics as nm
from oracle import policy as pol
from oracle.pool import OracleConfig, OraclePool, GROW, COMPACT, COMPACT_DENIED, SHRINK

HERE = os.path.dirname(os.path.abspath(__file__))


# ------------------------------------------------------------------ EMA ----

def _closed_form(qbars, beta):
    """s_t = beta^(t-1) qbar_1 + (1-beta) sum_{s=2..t} beta^(t-s) qbar_s (fp64)."""
    t = len(qbars)
    s = beta ** (t - 1) * qbars[0].astype(np.float64)
    for j in range(1, t):
        s = s + (1 - beta) * beta ** (t - 1 - j) * qbars[j].astype(np.float64)
    return s


@pytest.mark.parametrize("beta", [0.9, 0.999, 0.5])
def test_ema_recurrence_matches_closed_form(beta):
    rng = np.random.default_rng(1)
    qb = [rng.standard_normal(64).astype(np.float32) for _ in range(300)]
    s = qb[0].copy()
    for x in qb[1:]:
        s = nm.ema_fold(s, x, beta)
    ref = _closed_form(qb, float(np.float32(beta)))
    err = np.max(np.abs(s - ref)) / np.max(np.abs(ref))
    assert err < 3e-5, err


def test_ema_beta_zero_is_current_query():
    rng = np.random.default_rng(2)
    s = rng.standard_normal(32).astype(np.float32)
    x = rng.standard_normal(32).astype(np.float32)
    assert np.array_equal(nm.ema_fold(s, x, 0.0), x)


def test_group_mean_close_to_fp64_mean():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 128)).astype(np.float32)
    m = nm.group_mean_f32(q)
    ref = q.astype(np.float64).mean(axis=0)
    assert np.max(np.abs(m - ref)) < 1e-6


# ----------------------------------------------------------------- RoPE ----

def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(4)
    d, theta = 128, 500000.0
    tab = nm.RopeTable(theta, d)
    for pos in (0, 1, 17, 1000, 32767):
        x = rng.standard_normal(d)
        y = nm.rope_apply(x, tab, pos)
        h = d // 2
        w = np.exp(-np.arange(h) * 2.0 / d * np.log(theta))   # theta^(-2i/d)
        z = (x[:h] + 1j * x[h:]) * np.exp(1j * pos * w)
        assert np.allclose(y[:h], z.real, rtol=0, atol=1e-9 * max(1, pos) ** 0.5)
        assert np.allclose(y[h:], z.imag, rtol=0, atol=1e-9 * max(1, pos) ** 0.5)
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12 * d


def test_rope_relative_position_identity():
    rng = np.random.default_rng(5)
    d = 64
    tab = nm.RopeTable(10000.0, d)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    for m, n in ((5, 3), (100, 1), (777, 700)):
        lhs = nm.rope_apply(q, tab, m) @ nm.rope_apply(k, tab, n)
        rhs = nm.rope_apply(q, tab, m - n) @ k
        assert abs(lhs - rhs) < 1e-10


def test_rope_theta_zero_is_identity():
    x = np.arange(8.0)
    assert np.array_equal(nm.rope_apply(x, nm.RopeTable(0.0, 8), 123), x)


# ------------------------------------------------------- bf16 rounding ----

def _exact_bf16(x: float) -> float:
    """Nearest-even bf16 value of x by exact rational arithmetic."""
    if x == 0.0:
        return x
    fx = Fraction(x)
    a = abs(fx)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e - 7, -133)
    step = Fraction(2) ** q
    m = a / step
    lo = math.floor(m)
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    r = lo * step
    if r > Fraction(float.fromhex("0x1.fep127")):
        return math.copysign(math.inf, x)
    return math.copysign(float(r), x)


def test_round_bf16_exact_rational():
    rng = np.random.default_rng(6)
    xs = list(rng.standard_normal(2000) * np.exp(rng.uniform(-20, 20, 2000)))
    xs += [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 2 ** -130, 3 * 2 ** -134,
           2 ** -134, float.fromhex("0x1.ffp127"), float.fromhex("0x1.fdp127"), 1e-300]
    got = nm.round_bf16(np.array(xs))
    for x, g in zip(xs, got):
        assert g == _exact_bf16(float(x)), (x, g, _exact_bf16(float(x)))


def test_round_bf16_matches_torch_cast_on_fp32_values():
    rng = np.random.default_rng(7)
    x32 = (rng.standard_normal(10000) * 3).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(nm.round_bf16(x32.astype(np.float64)), ref)


# ---------------------------------------------------------------- Top-p ----

def _brute_topp(p, top_p):
    """Smallest size of ANY subset whose mass reaches top_p * total."""
    n = len(p)
    tot = float(np.sum(p))
    for size in range(1, n + 1):
        for sub in itertools.combinations(range(n), size):
            if float(np.sum(p[list(sub)])) >= top_p * tot:
                return size
    return n


def test_topp_brute_force_subsets():
    rng = np.random.default_rng(8)
    for trial in range(150):
        n = int(rng.integers(1, 10))
        u = rng.standard_normal(n) * rng.uniform(0.1, 4)
        p = pol.softmax(u)
        tp = float(rng.choice([0.5, 0.9, 0.99, float(np.float32(0.9))]))
        assert pol.topp_count(p, tp) == _brute_topp(p, tp), (p, tp)


def test_topp_uniform_and_one_hot():
    for n in (7, 64, 1000):
        p = np.full(n, 1.0 / n)
        tp = 0.9
        if abs(tp * n - round(tp * n)) > 1e-6:
            assert pol.topp_count(p, tp) == math.ceil(tp * n)
    u = np.zeros(100)
    u[37] = 50.0
    assert pol.topp_count(pol.softmax(u), 0.99) == 1


def test_demand_rule_strict():
    assert pol.wants_grow(1, 0.0)
    assert not pol.wants_grow(0, 0.0)
    assert not pol.wants_grow(-3, 0.0)
    assert pol.demand_delta([[3, 1]], [[1, 2]]) == 1


# ------------------------------------------------------ kept-set choice ----

@pytest.mark.parametrize("pages_freed", [1, 2])
def test_compaction_plan_brute_force(pages_freed):
    rng = np.random.default_rng(9 + pages_freed)
    P = 4
    n_free = pages_freed * P
    for trial in range(200):
        cap = P * int(rng.integers(pages_freed + 1, 6 + pages_freed))
        window = int(rng.integers(0, cap + 2))
        pos = np.sort(rng.choice(np.arange(0, 3 * cap), size=cap, replace=False))
        pos_now = int(pos[-1]) + 1
        # force the most recent tokens to be contiguous up to pos_now
        w_eff = min(window, cap - n_free)
        pos[cap - w_eff:] = np.arange(pos_now - w_eff, pos_now)
        pos = np.sort(pos)
        if len(set(pos.tolist())) != cap:
            continue
        imp = rng.choice([0.1, 0.2, 0.3, 0.5], size=cap) * rng.choice([1, 1, 2], size=cap)
        dropped, _ = pol.compaction_plan(imp, pos, pos_now, cap, P, window, n_free)
        kept = set(range(cap)) - set(dropped.tolist())
        recent = {j for j in range(cap) if pos[j] >= pos_now - w_eff}
        older = sorted((j for j in range(cap) if j not in recent),
                       key=lambda j: (imp[j], pos[j]), reverse=True)
        want = recent | set(older[:cap - n_free - w_eff])
        assert kept == want
        assert len(kept) == cap - n_free


# ------------------------------------------- attention vs dense SDPA ----

def _small_cfg(**kw):
    base = dict(num_layers=2, num_q_heads=8, num_kv_heads=2, head_dim=32,
                page_size=16, num_pages=64, max_pages_per_req=64, dtype="f32",
                rope_theta=10000.0, top_p=0.9, recent_window=16)
    base.update(kw)
    return OracleConfig(**base)


def _rope_complex(x, pos, theta):
    """Rotate-half RoPE by complex multiplication (independent of the oracle)."""
    d = x.shape[-1]
    h = d // 2
    w = np.exp(-np.arange(h) * 2.0 / d * np.log(theta))
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * pos * w)
    return np.concatenate([z.real, z.imag], axis=-1)


@pytest.mark.parametrize("G", [1, 4])
@pytest.mark.parametrize("full_kv", [True, False])
def test_attention_without_compaction_is_dense_sdpa(G, full_kv):
    torch.manual_seed(0)
    hk = 2
    cfg = _small_cfg(num_q_heads=hk * G, num_kv_heads=hk, full_kv=full_kv)
    pool = OraclePool(cfg)
    L, d = cfg.num_layers, cfg.head_dim
    plen = 21
    kp = torch.randn(L, plen, hk, d).numpy()
    vp = torch.randn(L, plen, hk, d).numpy()
    # a large budget so that no boundary is reached in GrowPage mode
    pool.add_request(3, kp, vp, budget_pages=8)
    Ks = [[_rope_complex(kp[l, j], j, cfg.rope_theta) for j in range(plen)] for l in range(L)]
    Vs = [[vp[l, j] for j in range(plen)] for l in range(L)]
    for t in range(12):
        pos = plen + t
        q = torch.randn(1, L, hk * G, d).numpy()
        k = torch.randn(1, L, hk, d).numpy()
        v = torch.randn(1, L, hk, d).numpy()
        res = pool.step([3], q, k, v)
        for l in range(L):
            Ks[l].append(_rope_complex(k[0, l], pos, cfg.rope_theta))
            Vs[l].append(v[0, l])
            K = torch.from_numpy(np.stack(Ks[l], 1))            # [Hk][R][d]
            V = torch.from_numpy(np.stack(Vs[l], 1)).double()
            Q = torch.from_numpy(_rope_complex(q[0, l], pos, cfg.rope_theta))[:, None, :]
            Kr = K.repeat_interleave(G, 0)
            Vr = V.repeat_interleave(G, 0)
            ref = torch.nn.functional.scaled_dot_product_attention(Q, Kr, Vr)[:, 0]
            # stored keys are fp32-rounded in the oracle; allow that rounding
            assert np.allclose(res["out"][0, l], ref.numpy(), rtol=0, atol=2e-6)
    pool.check_invariants()


# ------------------------------------------------------- pool behaviour ----

def _run_tiny(cfg, steps, budget=2, plen=32, seed=0, slots=(0,)):
    rng = np.random.default_rng(seed)
    pool = OraclePool(cfg)
    L, hk, hq, d = cfg.num_layers, cfg.num_kv_heads, cfg.num_q_heads, cfg.head_dim
    for s in slots:
        pool.add_request(s, rng.standard_normal((L, plen, hk, d)),
                         rng.standard_normal((L, plen, hk, d)), budget_pages=budget)
    recs = []
    for t in range(steps):
        n = len(slots)
        res = pool.step(list(slots), rng.standard_normal((n, L, hq, d)),
                        rng.standard_normal((n, L, hk, d)),
                        rng.standard_normal((n, L, hk, d)))
        recs.append(res["records"])
        pool.check_invariants()
    return pool, recs


def test_equal_summaries_always_compact_and_tau_negative_always_grows():
    # beta_s == beta_l makes both summaries identical: Delta == 0 at every
    # boundary, so the strict rule compacts; with tau < 0 it always grows.
    cfg = _small_cfg(beta_s=0.95, beta_l=0.95, num_pages=40)
    pool, recs = _run_tiny(cfg, 64)
    decs = [r.decision for rr in recs for r in rr.values()]
    assert decs and all(x == COMPACT for x in decs)
    assert all(r.delta == 0 for rr in recs for r in rr.values())
    n = pool.req[0].toks.n
    assert n <= 2 * 16 and len(pool.req[0].pages) == 2
    cfg2 = _small_cfg(beta_s=0.95, beta_l=0.95, tau=-1.0, num_pages=40)
    pool2, recs2 = _run_tiny(cfg2, 64)
    decs2 = [r.decision for rr in recs2 for r in rr.values()]
    assert decs2 and all(x == GROW for x in decs2)
    assert pool2.req[0].toks.n == 32 + 64


def test_boundary_every_page_size_steps_and_window_kept():
    cfg = _small_cfg(num_pages=40)
    pool, recs = _run_tiny(cfg, 80)
    steps_with_b = [t for t, rr in enumerate(recs) if rr]
    # prompt 32 = 2 pages exactly -> boundary at the first step, then every 16
    assert steps_with_b == list(range(0, 80, 16))
    r = pool.req[0]
    pos = np.sort(r.toks.pos[:, :, :r.toks.n], axis=-1)
    # the most recent tokens are always resident
    assert np.all(pos[..., -16:] == np.arange(r.pos - 16, r.pos))


def test_full_kv_never_compacts_and_grows_one_page_per_boundary():
    cfg = _small_cfg(full_kv=True, num_pages=64)
    pool, recs = _run_tiny(cfg, 70)
    r = pool.req[0]
    assert r.toks.n == 32 + 70
    assert len(r.pages) == 2 + len([1 for rr in recs if rr])
    assert len(r.pages) * 16 >= r.toks.n


def test_pool_exhaustion_compacts_instead():
    cfg = _small_cfg(tau=-1.0, num_pages=3)
    pool, recs = _run_tiny(cfg, 40)
    decs = [r.decision for rr in recs for r in rr.values()]
    assert decs[0] == GROW and all(x == COMPACT_DENIED for x in decs[1:])
    assert not pool.free


def test_allocator_order_prefix_refcounts_and_free():
    cfg = _small_cfg(num_pages=20)
    rng = np.random.default_rng(11)
    pool = OraclePool(cfg)
    L, hk, d = cfg.num_layers, cfg.num_kv_heads, cfg.head_dim
    pid = pool.add_prefix(rng.standard_normal((L, 32, hk, d)),
                          rng.standard_normal((L, 32, hk, d)))
    assert pool.prefixes[pid].pages == [0, 1]
    pool.add_request(0, np.zeros((L, 5, hk, d)), np.zeros((L, 5, hk, d)), 2, pid)
    pool.add_request(4, np.zeros((L, 0, hk, d)), np.zeros((L, 0, hk, d)), 3, pid)
    assert pool.block_table(0) == [0, 1, 2, 3]
    assert pool.block_table(4) == [0, 1, 4, 5, 6]
    pool.check_invariants()
    pool.free_request(0)           # pushes 2, 3 -> next pops 3, 2
    pool.add_request(1, np.zeros((L, 1, hk, d)), np.zeros((L, 1, hk, d)), 2)
    assert pool.block_table(1) == [3, 2]
    pool.release_prefix(pid)
    assert pid in pool.prefixes    # still used by slot 4
    pool.free_request(4)
    assert pid not in pool.prefixes
    pool.check_invariants()
    assert len(pool.free) == 18


def test_growpage_run_with_prefix_keeps_invariants():
    cfg = _small_cfg(num_pages=64, num_layers=1)
    rng = np.random.default_rng(12)
    pool = OraclePool(cfg)
    L, hk, hq, d = 1, cfg.num_kv_heads, cfg.num_q_heads, cfg.head_dim
    pid = pool.add_prefix(rng.standard_normal((L, 16, hk, d)), rng.standard_normal((L, 16, hk, d)))
    pool.add_request(0, rng.standard_normal((L, 30, hk, d)), rng.standard_normal((L, 30, hk, d)), 2, pid)
    pool.add_request(2, rng.standard_normal((L, 32, hk, d)), rng.standard_normal((L, 32, hk, d)), 2, -1)
    nb = 0
    for t in range(100):
        res = pool.step([0, 2], rng.standard_normal((2, L, hq, d)),
                        rng.standard_normal((2, L, hk, d)), rng.standard_normal((2, L, hk, d)))
        nb += len(res["records"])
        pool.check_invariants()
        for s in (0, 2):
            kp = pool.kept_positions(s)
            assert kp.shape[-1] == pool.req[s].toks.n
            assert np.all(kp >= pool.req[s].prefix_len)      # prefix never a candidate
    assert nb > 5


def test_paper_hyperparameters_fixture():
    with open(os.path.join(HERE, "golden", "paper_hyperparameters.json")) as f:
        g = json.load(f)
    c = OracleConfig(num_layers=1, num_q_heads=1, num_kv_heads=1, head_dim=2,
                     page_size=g["kv_block_size"], num_pages=1, max_pages_per_req=1,
                     dtype="f32", rope_theta=0.0, top_p=g["top_p"],
                     recent_window=g["local_retention_quota"], tau=g["tau"])
    assert (c.beta_s, c.beta_l) == (g["beta_short"], g["beta_long"])
    for name, row in g["throughput_tok_s_full_kv_vs_growpage"].items():
        if name.startswith("_"):
            continue
        full, gp, pct = row
        # The review prints +64.3% next to 1472 -> 2417 tok/s, whose ratio is
        # +64.2%: the percentage is presumably averaged per benchmark.
        assert abs((gp / full - 1) * 100 - pct) < 0.15


def test_pool_summaries_follow_closed_form_of_group_means():
    # The pool folds the mean of each kv head's query group once per step;
    # its summaries must match the fp64 closed form of those means.
    cfg = _small_cfg(num_layers=1, num_q_heads=8, num_kv_heads=2, num_pages=64)
    rng = np.random.default_rng(13)
    pool = OraclePool(cfg)
    L, hk, hq, d = 1, 2, 8, cfg.head_dim
    pool.add_request(0, rng.standard_normal((L, 8, hk, d)), rng.standard_normal((L, 8, hk, d)), 4)
    qs = []
    for t in range(60):
        q = rng.standard_normal((1, L, hq, d)).astype(np.float32)
        qs.append(q[0, 0].reshape(hk, 4, d).astype(np.float64).mean(axis=1))
        res = pool.step([0], q, rng.standard_normal((1, L, hk, d)), rng.standard_normal((1, L, hk, d)))
    for X, beta in ((0, cfg.beta_s), (1, cfg.beta_l)):
        ref = _closed_form(qs, float(np.float32(beta)))
        got = res["summaries"][0, 0, :, X]
        assert np.max(np.abs(got - ref)) < 2e-5 * np.max(np.abs(ref))


# ----------------------------------------------------- ablation policies ----

def test_splitmix64_published_outputs():
    with open(os.path.join(HERE, "golden", "splitmix64.json")) as f:
        g = json.load(f)
    golden = 0x9E3779B97F4A7C15
    for k, want in enumerate(g["outputs_from_state_0"]):
        # next() advances the state by the golden gamma, then mixes
        assert pol.splitmix64((k * golden) & pol.MASK64) == int(want, 16)


def test_random_policy_frequency():
    for rate in (0.0, 0.3, 1.0):
        n = 20000
        grows = sum(pol.random_grow(s, b, rate) for s in range(40) for b in range(n // 40))
        if rate in (0.0, 1.0):
            assert grows == int(rate * n)
        else:
            assert abs(grows / n - rate) < 4 * math.sqrt(rate * (1 - rate) / n)


def _first_decision(policy, seed=21, **kw):
    cfg = _small_cfg(num_pages=40, policy=policy, **kw)
    rng = np.random.default_rng(seed)
    pool = OraclePool(cfg)
    L, hk, hq, d = cfg.num_layers, cfg.num_kv_heads, cfg.num_q_heads, cfg.head_dim
    # 20 prompt tokens in a 2-page budget: the first boundary comes at step
    # 13, after the summaries have diverged
    pool.add_request(0, rng.standard_normal((L, 20, hk, d)), rng.standard_normal((L, 20, hk, d)), 2)
    for t in range(40):
        res = pool.step([0], rng.standard_normal((1, L, hq, d)), rng.standard_normal((1, L, hk, d)),
                        rng.standard_normal((1, L, hk, d)))
        if res["records"]:
            return res["records"][0]
    raise AssertionError("no boundary")


def test_inverse_and_fixed_policies_at_the_first_boundary():
    # the three policies see the same inputs up to their first boundary,
    # hence the same scores and the same Delta
    g = _first_decision("growpage")
    inv = _first_decision("inverse")
    fx = _first_decision("fixed")
    assert g.delta == inv.delta == fx.delta != 0
    assert (g.decision == GROW) == (g.delta > 0)
    assert (inv.decision == GROW) == (inv.delta < 0)
    assert fx.decision == COMPACT


def test_shrink_policy_releases_pages_down_to_the_window():
    # equal smoothing makes Delta == 0 at every boundary: never a grow.  With
    # 8 pages of 16 tokens and a 16-token window, SHRINK releases one page per
    # boundary while (pages - 2) * 16 >= 16, i.e. down to 2 pages, then
    # compacts in place.
    cfg = _small_cfg(beta_s=0.95, beta_l=0.95, num_pages=40, policy="shrink")
    rng = np.random.default_rng(5)
    pool = OraclePool(cfg)
    L, hk, hq, d, P = cfg.num_layers, cfg.num_kv_heads, cfg.num_q_heads, cfg.head_dim, 16
    pool.add_request(0, rng.standard_normal((L, 128, hk, d)), rng.standard_normal((L, 128, hk, d)),
                     budget_pages=8)
    decs, pages = [], []
    for t in range(130):
        before = list(pool.req[0].pages)
        res = pool.step([0], rng.standard_normal((1, L, hq, d)), rng.standard_normal((1, L, hk, d)),
                        rng.standard_normal((1, L, hk, d)))
        pool.check_invariants()
        rec = res["records"].get(0)
        r = pool.req[0]
        if rec is None:
            continue
        assert t % P == 0               # the cadence of boundaries is unchanged
        decs.append(rec.decision)
        pages.append(len(r.pages))
        if rec.decision == SHRINK:
            # the last private page went back on top of the free stack
            assert r.pages == before[:-1] and pool.free[-1] == before[-1]
            assert r.toks.n == (len(before) - 2) * P + 1   # kept + the staged token
        # the most recent tokens are always resident
        pos = np.sort(r.toks.pos[:, :, :r.toks.n], axis=-1)
        assert np.all(pos[..., -16:] == np.arange(r.pos - 16, r.pos))
    assert decs == [SHRINK] * 6 + [COMPACT] * (len(decs) - 6)
    assert pages[:7] == [7, 6, 5, 4, 3, 2, 2]


def test_shrink_policy_grows_like_growpage():
    # tau < 0: every boundary wants to grow, so SHRINK never releases a page
    cfg = _small_cfg(beta_s=0.95, beta_l=0.95, tau=-1.0, num_pages=40, policy="shrink")
    pool, recs = _run_tiny(cfg, 64)
    decs = [r.decision for rr in recs for r in rr.values()]
    assert decs and all(x == GROW for x in decs)
    assert pool.req[0].toks.n == 32 + 64


def test_may_shrink_floor():
    assert pol.may_shrink(6, 16, 64) and not pol.may_shrink(5, 16, 64)
    assert pol.may_shrink(2, 16, 0) and not pol.may_shrink(1, 16, 0)


def test_topp_near_tie_band():
    # uniform mass over 10 tokens: Top-p 0.3 reaches its mass exactly at 3
    # tokens, so a relative move of 1e-5 either way changes W (a near tie);
    # at Top-p 0.35 the threshold sits mid-token and the band is one value
    p = np.full(10, 0.1)
    assert pol.topp_count(p, 0.3) in (3, 4)
    lo, hi = pol.topp_range(p, 0.3)
    assert (lo, hi) == (3, 4)
    assert pol.topp_range(p, 0.35) == (4, 4)
    # a dominant token: W = 1 for any Top-p up to its mass
    q = np.array([0.97, 0.01, 0.01, 0.01])
    assert pol.topp_range(q, 0.9) == (1, 1)


def test_shrink_with_prefix_and_several_requests_keeps_invariants():
    # SHRINK with a shared prefix and three requests at boundaries in the same
    # steps: request 1 sees one constant query, so its two summaries stay
    # equal (Delta = 0) and it releases pages, while the other two see random
    # queries and grow.  Every page is owned once, prefix tokens are never
    # dropped, and pages released in a step go on the stack after the step's
    # pops, in ascending slot order.
    cfg = _small_cfg(num_pages=80, num_layers=1, policy="shrink", recent_window=16)
    rng = np.random.default_rng(21)
    pool = OraclePool(cfg)
    L, hk, hq, d = 1, cfg.num_kv_heads, cfg.num_q_heads, cfg.head_dim
    pid = pool.add_prefix(rng.standard_normal((L, 32, hk, d)), rng.standard_normal((L, 32, hk, d)))
    for s, pre in enumerate([pid, -1, pid]):
        pool.add_request(s, rng.standard_normal((L, 96, hk, d)), rng.standard_normal((L, 96, hk, d)),
                         6, pre)
    q_const = rng.standard_normal((L, hq, d))
    mixed = 0
    for t in range(160):
        before = {s: list(pool.req[s].pages) for s in range(3)}
        q = rng.standard_normal((3, L, hq, d))
        q[1] = q_const
        res = pool.step([0, 1, 2], q, rng.standard_normal((3, L, hk, d)),
                        rng.standard_normal((3, L, hk, d)))
        pool.check_invariants()
        recs = res["records"]
        released = [before[s][-1] for s in sorted(recs) if recs[s].decision == SHRINK]
        grown = [pool.req[s].pages[-1] for s in sorted(recs) if recs[s].decision == GROW]
        if released:
            assert pool.free[-len(released):] == released
            assert not set(released) & set(grown)
            mixed += bool(grown)
        if 1 in recs and len(before[1]) >= 3:
            assert recs[1].delta == 0 and recs[1].decision == SHRINK
        for s in range(3):
            assert np.all(pool.kept_positions(s) >= pool.req[s].prefix_len)
    assert mixed >= 2
