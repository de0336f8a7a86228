"""Step-by-step fp64 simulation of a GrowPage page pool under decoding.

Test infrastructure only (see the package docstring).

Sources ("GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning
Serving"):
* abstract: capacity boundaries; "compresses KV states within the current
  allocation or acquires an additional physical page"; integration with
  PagedAttention's page-level memory; continuous batching and prefix caching
  are preserved.
* evolve.pub review, Summary: Top-p working sets of the short / long query
  summaries (beta 0.9 / 0.999, kept pre-RoPE); one extra physical page when
  the recent working set is larger, else compaction by the maximum of both
  importance scores.
* evolve.pub review, FAQ: Top-p, tau = 0, local retention quota.

Readings this module takes (the pages leave them open):
* Boundary: a request is at a capacity boundary when, at the start of a
  step, all its private pages are full (private tokens == pages * page size).
  Pages are allocated when a request is admitted (its initial budget) and
  one at a time by growth.
* Step order: stage the new token (its key rotated to its position, rounded
  once to the storage dtype), fold q_t into both summaries, attend over the
  resident tokens plus the staged one; at a boundary, score both summaries,
  rotated to the current position, against every resident key (prefix
  included, staged token excluded); decide; grow or compact; then append the
  staged token.
* Summaries are per kv head, over the mean of its query heads; first fold
  sets s = qbar.
* Delta = sum over layers and kv heads of (W_short - W_long); grow iff
  Delta > tau and a page is free (and the request is below its page cap);
  otherwise compact.  Compaction keeps capacity - page_size private tokens:
  the most recent min(window, capacity - page_size) plus the highest by
  importance (ties: the more recent is kept).  Selection is per (layer, kv
  head), so every (layer, head) keeps the same count.
* Allocator: a stack whose pops return 0, 1, 2, ... initially; growth is
  served in ascending slot order; freeing pushes a request's private pages in
  block-table order, and a prefix's pages once its reference count is 0.
  Pages released by the SHRINK ablation are pushed after every growth of the
  step has popped, in ascending slot order.
* Full-KV mode: the same steps, every boundary grows, nothing is compacted;
  a boundary that cannot get a page (none free, or the request already holds
  max_pages_per_req) drops the step's token ("starved").
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

from . import numerics as nm
from . import policy as pol

GROW, COMPACT, COMPACT_DENIED, STARVED, SHRINK = 1, 2, 3, 4, 5


@dataclasses.dataclass
class OracleConfig:
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    max_pages_per_req: int
    dtype: str
    rope_theta: float
    top_p: float
    recent_window: int
    beta_s: float = 0.9
    beta_l: float = 0.999
    tau: float = 0.0
    full_kv: bool = False
    # grow decision at a boundary: "growpage" (Delta > tau), "fixed" (never),
    # "inverse" (-Delta > tau), "random" (see policy.random_grow) or "shrink"
    # (Delta > tau grows; otherwise a page is released, see policy.may_shrink)
    policy: str = "growpage"
    random_grow_rate: float = 0.0

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    @staticmethod
    def from_workload(w, full_kv=False, **over):  # noqa: D401
        kw = dict(num_layers=w.num_layers, num_q_heads=w.num_q_heads,
                  num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                  page_size=w.page_size, num_pages=w.num_pages,
                  max_pages_per_req=w.max_pages_per_req, dtype=w.dtype,
                  rope_theta=w.rope_theta, top_p=w.top_p,
                  recent_window=w.recent_window, beta_s=w.beta_s,
                  beta_l=w.beta_l, tau=w.tau, full_kv=full_kv)
        kw.update(over)
        return OracleConfig(**kw)


class _Grow:
    """Row-growable per-(layer, head) token arrays."""

    def __init__(self, L, hk, d):
        self.cap = 64
        self.n = 0
        self.K = np.zeros((L, hk, self.cap, d))
        self.V = np.zeros((L, hk, self.cap, d))
        self.pos = np.zeros((L, hk, self.cap), dtype=np.int64)

    def append(self, k, v, pos):
        if self.n == self.cap:
            self.cap *= 2
            for name in ("K", "V", "pos"):
                a = getattr(self, name)
                b = np.zeros(a.shape[:2] + (self.cap,) + a.shape[3:], dtype=a.dtype)
                b[:, :, :self.n] = a[:, :, :self.n]
                setattr(self, name, b)
        self.K[:, :, self.n] = k
        self.V[:, :, self.n] = v
        self.pos[:, :, self.n] = pos
        self.n += 1


@dataclasses.dataclass
class OracleRequest:
    slot: int
    prefix_id: int
    prefix_len: int
    pages: List[int]
    pos: int
    steps: int
    toks: _Grow
    s_short: np.ndarray     # fp32 [L][Hk][d]
    s_long: np.ndarray
    boundaries: int = 0     # capacity boundaries met so far


@dataclasses.dataclass
class OraclePrefix:
    pages: List[int]
    length: int
    K: np.ndarray           # [L][Hk][len][d] stored (rounded) keys, fp64
    V: np.ndarray
    refs: int               # requests using it + 1 while its creator holds it
    held: bool = True


@dataclasses.dataclass
class BoundaryRecord:
    slot: int
    delta: int
    decision: int
    decision_exempt: bool
    w_short: np.ndarray          # [L][Hk]
    w_long: np.ndarray
    w_near_tie: np.ndarray       # [L][Hk][2] bool: W moves inside the band
    cut_gap: Optional[np.ndarray]  # [L][Hk] relative gap at the kept-set cut
    logits: Optional[np.ndarray] = None  # [L][Hk][2][R] when kept
    w_band: Optional[np.ndarray] = None  # [L][Hk][2][2]: W at Top-p*(1-1e-5), *(1+1e-5)


class OraclePool:
    def __init__(self, cfg: OracleConfig, keep_logits: bool = False):
        self.cfg = cfg
        self.free = list(range(cfg.num_pages - 1, -1, -1))  # pop() -> 0, 1, ...
        self.req: Dict[int, OracleRequest] = {}
        self.prefixes: Dict[int, OraclePrefix] = {}
        self.next_prefix = 0
        self.rope = nm.RopeTable(cfg.rope_theta, cfg.head_dim)
        self.keep_logits = keep_logits
        self.starved = 0

    # ------------------------------------------------------------ admin ----
    def _store_keys(self, k_raw, positions):
        """Rotate raw keys [L][len][Hk][d] to their positions, round once."""
        k = np.asarray(k_raw, dtype=np.float64)
        out = np.empty_like(k)
        for j, p in enumerate(positions):
            out[:, j] = nm.to_storage(nm.rope_apply(k[:, j], self.rope, p), self.cfg.dtype)
        return out

    def add_prefix(self, k, v) -> int:
        c = self.cfg
        length = k.shape[1]
        assert length % c.page_size == 0
        npg = length // c.page_size
        if len(self.free) < npg:
            raise MemoryError("no pages")
        pages = [self.free.pop() for _ in range(npg)]
        ks = self._store_keys(k, range(length))
        vs = np.asarray(v, dtype=np.float64)
        pid = self.next_prefix
        self.next_prefix += 1
        self.prefixes[pid] = OraclePrefix(pages, length, ks.transpose(0, 2, 1, 3).copy(),
                                          vs.transpose(0, 2, 1, 3).copy(), refs=1)
        return pid

    def release_prefix(self, pid: int):
        pf = self.prefixes[pid]
        assert pf.held
        pf.held = False
        self._unref(pid)

    def _unref(self, pid):
        pf = self.prefixes[pid]
        pf.refs -= 1
        if pf.refs == 0:
            for pg in pf.pages:
                self.free.append(pg)
            del self.prefixes[pid]

    def add_request(self, slot, k_prompt, v_prompt, budget_pages, prefix_id=-1):
        c = self.cfg
        assert slot not in self.req
        plen = self.prefixes[prefix_id].length if prefix_id >= 0 else 0
        n = k_prompt.shape[1]
        if n > budget_pages * c.page_size or budget_pages > c.max_pages_per_req or budget_pages < 1:
            raise ValueError("prompt does not fit the budget")
        if len(self.free) < budget_pages:
            raise MemoryError("no pages")
        pages = [self.free.pop() for _ in range(budget_pages)]
        if prefix_id >= 0:
            self.prefixes[prefix_id].refs += 1
        toks = _Grow(c.num_layers, c.num_kv_heads, c.head_dim)
        ks = self._store_keys(k_prompt, range(plen, plen + n))
        vs = np.asarray(v_prompt, dtype=np.float64)
        for j in range(n):
            toks.append(ks[:, j], vs[:, j], plen + j)
        z = np.zeros((c.num_layers, c.num_kv_heads, c.head_dim), np.float32)
        self.req[slot] = OracleRequest(slot, prefix_id, plen, pages, plen + n, 0,
                                       toks, z.copy(), z.copy())

    def free_request(self, slot):
        r = self.req.pop(slot)
        for pg in r.pages:
            self.free.append(pg)
        if r.prefix_id >= 0:
            self._unref(r.prefix_id)

    # ------------------------------------------------------------- step ----
    def _summary_scores(self, Kres, s, pos_t, scale):
        """Summary scores of one layer: u_j = RoPE(s, pos_t) . k_j / sqrt(d).

        Kres: [Hk][R][d] resident keys (prefix first, then private; the step's
        staged token is not among them), stored rotated to their own
        positions.  s: [Hk][d] fp32 summary, kept pre-RoPE.  Reading: the
        review keeps the summaries pre-RoPE, so a summary is rotated to the
        current position before it meets the rotated cache, as a query of
        that position would be.
        """
        sr = nm.rope_apply(np.asarray(s, dtype=np.float64), self.rope, pos_t)
        return np.matmul(Kres, sr[:, :, None])[:, :, 0] * scale

    def step(self, slots, q, k, v, arbiter=None):
        """One decode step for the requests ``slots`` (ascending).

        q: [n][L][Hq][d], k, v: [n][L][Hk][d] (storage-dtype values).
        Returns a dict: out [n][L][Hq][d] fp64, staged_k [n][L][Hk][d] (the
        stored key of the step's token), summaries [n][L][Hk][2][d] fp32,
        boundary records by slot.

        ``arbiter`` (optional) lets a checker resynchronise the simulation
        at near-ties, where more than one outcome is correct.  It is asked
        only at two points and only after the oracle has computed its own
        choice: ``arbiter.decision(slot, record)`` may return another
        decision for a boundary whose record is ``decision_exempt``, and
        ``arbiter.dropped(slot, layer, head, pos_priv, dropped, gap)`` may
        return another set of dropped indices when the relative importance
        gap at the cut is at most 1e-5.  Anything else it returns is
        rejected.  The arithmetic of the step does not change.
        """
        c = self.cfg
        L, hk, hq, d, G, P = (c.num_layers, c.num_kv_heads, c.num_q_heads,
                              c.head_dim, c.group, c.page_size)
        assert list(slots) == sorted(slots) and len(set(slots)) == len(slots)
        n = len(slots)
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        out = np.zeros((n, L, hq, d))
        staged_k = np.zeros((n, L, hk, d))
        summ = np.zeros((n, L, hk, 2, d), np.float32)
        records = {}
        scale = 1.0 / math.sqrt(d)
        boundary_logits = {}
        for i, slot in enumerate(slots):
            r = self.req[slot]
            cap = len(r.pages) * P
            at_b = r.toks.n == cap
            pos_t = r.pos
            # A2: fold q_t into both summaries (fp32, before any scoring).
            qbar = nm.group_mean_f32(q[i].reshape(L, hk, G, d))
            if r.steps == 0:
                r.s_short = qbar.copy()
                r.s_long = qbar.copy()
            else:
                r.s_short = nm.ema_fold(r.s_short, qbar, c.beta_s)
                r.s_long = nm.ema_fold(r.s_long, qbar, c.beta_l)
            summ[i, :, :, 0] = r.s_short
            summ[i, :, :, 1] = r.s_long
            # A1: stage the step's key (rotated to pos_t, one rounding).
            ks = nm.to_storage(nm.rope_apply(k[i], self.rope, pos_t), c.dtype)
            staged_k[i] = ks
            pf = self.prefixes[r.prefix_id] if r.prefix_id >= 0 else None
            npriv = r.toks.n
            lg = np.zeros((L, hk, 2, (pf.length if pf else 0) + npriv)) if at_b else None
            for l in range(L):
                Kres = r.toks.K[l, :, :npriv]
                Vres = r.toks.V[l, :, :npriv]
                if pf is not None:
                    Kres = np.concatenate([pf.K[l], Kres], axis=1)
                    Vres = np.concatenate([pf.V[l], Vres], axis=1)
                # A3: attention over resident tokens + the staged token.
                qr = nm.rope_apply(q[i, l], self.rope, pos_t).reshape(hk, G, d)
                logits = np.concatenate(
                    [np.matmul(qr, Kres.transpose(0, 2, 1)),
                     np.matmul(qr, ks[l][:, :, None])], axis=2) * scale   # [Hk][G][R+1]
                p = pol.softmax(logits)
                o = np.matmul(p[:, :, :-1], Vres) + p[:, :, -1:] * v[i, l][:, None, :]
                out[i, l] = o.reshape(hq, d)
                # A4: summary logits against every resident key.
                if at_b and not c.full_kv:
                    for X, s in ((0, r.s_short[l]), (1, r.s_long[l])):
                        lg[l, :, X] = self._summary_scores(Kres, s, pos_t, scale)
            if at_b:
                boundary_logits[slot] = lg
        # A5/A6: working sets and decisions; A7: growth in ascending slot order.
        decisions = {}
        for slot in slots:
            r = self.req[slot]
            cap = len(r.pages) * P
            if r.toks.n != cap:
                continue
            if c.full_kv:
                if self.free and len(r.pages) < c.max_pages_per_req:
                    r.pages.append(self.free.pop())
                    decisions[slot] = GROW
                else:
                    decisions[slot] = STARVED
                    self.starved += 1
                records[slot] = BoundaryRecord(slot, 0, decisions[slot], False,
                                               np.zeros((L, hk), np.int64),
                                               np.zeros((L, hk), np.int64),
                                               np.zeros((L, hk, 2), bool), None)
                continue
            lg = boundary_logits[slot]
            ws = np.zeros((L, hk), np.int64)
            wl = np.zeros((L, hk), np.int64)
            band = np.zeros((L, hk, 2, 2), np.int64)
            for l in range(L):
                for g in range(hk):
                    for X, W in ((0, ws), (1, wl)):
                        pr = pol.softmax(lg[l, g, X])
                        W[l, g] = pol.topp_count(pr, c.top_p)
                        band[l, g, X] = pol.topp_range(pr, c.top_p)
            delta = pol.demand_delta(ws, wl)
            dmin, dmax = pol.delta_range(band[:, :, 0], band[:, :, 1])
            if c.policy in ("growpage", "shrink"):
                want = pol.wants_grow(delta, c.tau)
                exempt = pol.wants_grow(dmin, c.tau) != pol.wants_grow(dmax, c.tau)
            elif c.policy == "inverse":
                want = pol.wants_grow(-delta, c.tau)
                exempt = pol.wants_grow(-dmin, c.tau) != pol.wants_grow(-dmax, c.tau)
            elif c.policy == "fixed":
                want, exempt = False, False
            elif c.policy == "random":
                want = pol.random_grow(slot, r.boundaries, c.random_grow_rate)
                exempt = False
            else:
                raise ValueError(c.policy)
            r.boundaries += 1
            can = len(r.pages) < c.max_pages_per_req
            if arbiter is not None and exempt:
                # near-tie: the checker may adopt the other side of the rule
                rec0 = BoundaryRecord(slot, delta, None, exempt, ws, wl, None, None)
                forced = arbiter.decision(slot, rec0)
                if forced is not None:
                    want = bool(forced)
            if want and can and self.free:
                r.pages.append(self.free.pop())
                dec = GROW
            elif want:
                dec = COMPACT_DENIED
            elif c.policy == "shrink" and pol.may_shrink(len(r.pages), P, c.recent_window):
                dec = SHRINK
            else:
                dec = COMPACT
            decisions[slot] = dec
            near = band[:, :, :, 0] != band[:, :, :, 1]
            records[slot] = BoundaryRecord(slot, delta, dec, exempt, ws, wl, near, None,
                                           lg if self.keep_logits else None, band)
        # SHRINK releases the last private page of each shrinking request, in
        # ascending slot order, after every growth of the step has popped.
        for slot in sorted(decisions):
            if decisions[slot] == SHRINK:
                self.free.append(self.req[slot].pages[-1])
        # A8/A9: compaction of the requests that did not grow.
        for slot, dec in decisions.items():
            if dec not in (COMPACT, COMPACT_DENIED, SHRINK):
                continue
            r = self.req[slot]
            cap = len(r.pages) * P
            lg = boundary_logits[slot]
            plen = r.prefix_len
            gaps = np.full((L, hk), np.inf)
            n_free = 2 * P if dec == SHRINK else P
            keep_n = cap - n_free
            newK = np.zeros((L, hk, r.toks.cap, d))
            newV = np.zeros_like(newK)
            newpos = np.zeros((L, hk, r.toks.cap), np.int64)
            for l in range(L):
                for g in range(hk):
                    imp = pol.private_importance(lg[l, g, 0], lg[l, g, 1], plen)
                    posp = r.toks.pos[l, g, :cap]
                    dropped, gap = pol.compaction_plan(imp, posp, r.pos, cap, P,
                                                       c.recent_window, n_free)
                    if arbiter is not None and gap <= 1e-5:
                        alt = arbiter.dropped(slot, l, g, posp.copy(), dropped.copy(), gap)
                        if alt is not None:
                            alt = np.asarray(alt, dtype=np.int64)
                            w_eff = min(c.recent_window, cap - n_free)
                            ok = (len(set(alt.tolist())) == len(dropped)
                                  and np.all(posp[alt] < r.pos - w_eff))
                            if not ok:
                                raise ValueError("arbiter returned an invalid dropped set")
                            dropped = alt
                    gaps[l, g] = gap
                    keep = np.ones(cap, bool)
                    keep[dropped] = False
                    newK[l, g, :keep_n] = r.toks.K[l, g, :cap][keep]
                    newV[l, g, :keep_n] = r.toks.V[l, g, :cap][keep]
                    newpos[l, g, :keep_n] = posp[keep]
            r.toks.K, r.toks.V, r.toks.pos = newK, newV, newpos
            r.toks.n = keep_n
            if dec == SHRINK:
                r.pages.pop()
            records[slot].cut_gap = gaps
        # A10: commit the staged token.
        for i, slot in enumerate(slots):
            r = self.req[slot]
            if decisions.get(slot) != STARVED:
                r.toks.append(staged_k[i], v[i], r.pos)
            r.pos += 1
            r.steps += 1
        return dict(out=out, staged_k=staged_k, summaries=summ, records=records)

    # ------------------------------------------------------- inspection ----
    def kept_positions(self, slot):
        """Sorted private positions per (layer, head): [L][Hk][n] int64."""
        r = self.req[slot]
        return np.sort(r.toks.pos[:, :, :r.toks.n], axis=-1)

    def block_table(self, slot):
        r = self.req[slot]
        pre = self.prefixes[r.prefix_id].pages if r.prefix_id >= 0 else []
        return list(pre) + list(r.pages)

    def check_invariants(self):
        """Pool invariants: ownership, counts, capacity.  Raises on violation."""
        c = self.cfg
        owned = []
        for pid, pf in self.prefixes.items():
            owned += pf.pages
            users = sum(1 for r in self.req.values() if r.prefix_id == pid)
            assert pf.refs == users + int(pf.held), "prefix refcount"
            assert pf.refs > 0
        for r in self.req.values():
            owned += r.pages
            assert r.toks.n <= len(r.pages) * c.page_size
            assert len(r.pages) <= c.max_pages_per_req
        assert len(owned) == len(set(owned)), "page owned twice"
        assert not (set(owned) & set(self.free)), "page both owned and free"
        assert len(owned) + len(self.free) == c.num_pages, "page leaked"
        assert len(set(self.free)) == len(self.free)
