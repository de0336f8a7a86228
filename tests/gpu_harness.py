"""Step-by-step comparison of the CUDA path with the CPU oracle.

Both sides get the same seeded inputs (``synth.RequestStream``).  Every step
runs on the GPU first, then in the oracle; the oracle computes its own
result and may adopt the GPU's choice only at a near-tie (a decision whose
sign flips when Top-p moves by 1e-5 relative, or a compaction cut whose
importance gap is at most 1e-5 relative).  Every such adoption is counted.

Compared each step, per request:
  * attention output: max-abs error / max-abs oracle value per (request,
    layer) within ``tol`` (1e-4 for fp32 storage, 2e-2 for bf16);
  * both summaries and the staged (rotated, rounded) key: bit-exact;
  * position, pages held, private tokens, block table: exact;
  * at a boundary: the decision and Delta exact (Delta only when no W sits
    in its near-tie band), each W exact outside its band and inside the band
    otherwise; after a compaction, the kept positions per (layer, kv head)
    exact.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch

from demand_paged_kv_gqa_b300 import growpage as gpb
from demand_paged_kv_gqa_b300 import synth
from oracle.pool import OracleConfig, OraclePool, GROW, COMPACT, COMPACT_DENIED, STARVED, SHRINK


@dataclasses.dataclass
class Report:
    steps: int = 0
    boundaries: int = 0
    grows: int = 0
    compacts: int = 0
    shrinks: int = 0
    decision_resyncs: int = 0
    cut_resyncs: int = 0
    w_in_band: int = 0
    max_out_err: float = 0.0
    failures: List[str] = dataclasses.field(default_factory=list)

    def fail(self, msg):
        if len(self.failures) < 20:
            self.failures.append(msg)


class _Arbiter:
    """Offers the oracle the GPU's choice at near-ties (and counts them)."""

    def __init__(self, rep: Report):
        self.rep = rep
        self.gpu_dec: Dict[int, int] = {}
        self.gpu_kept: Dict[int, np.ndarray] = {}   # slot -> [L][Hk] sets

    def decision(self, slot, rec):
        g = self.gpu_dec.get(slot)
        if g is None:
            return None
        want = g in (GROW, COMPACT_DENIED)
        self.rep.decision_resyncs += 1
        return want

    def dropped(self, slot, l, h, pos_priv, dropped, gap):
        kept = self.gpu_kept.get(slot)
        if kept is None:
            return None
        ks = kept[l][h]
        gd = np.array([j for j in range(len(pos_priv)) if int(pos_priv[j]) not in ks], dtype=np.int64)
        if sorted(gd.tolist()) == sorted(dropped.tolist()):
            return None
        self.rep.cut_resyncs += 1
        return gd


def oracle_config(w, mode, num_pages, random_grow_rate=0.0):
    """The oracle's configuration for a GPU pool mode."""
    policy = {gpb.GP_MODE_GROWPAGE: "growpage", gpb.GP_MODE_FULL_KV: "growpage",
              gpb.GP_MODE_FIXED: "fixed", gpb.GP_MODE_INVERSE: "inverse",
              gpb.GP_MODE_RANDOM: "random", gpb.GP_MODE_SHRINK: "shrink"}[mode]
    return OracleConfig.from_workload(w, full_kv=mode == gpb.GP_MODE_FULL_KV, num_pages=num_pages,
                                      policy=policy, random_grow_rate=random_grow_rate)


def _private_positions(tok_pos, bt_priv: List[int], n: int, L: int, hk: int, P: int):
    """[L][Hk][n] positions of the first n private slots (block-table order).

    ``tok_pos`` is the host copy of the whole region, or the device tensor
    itself, in which case only the request's own pages are copied."""
    npg = -(-n // P)
    if isinstance(tok_pos, torch.Tensor):
        idx = torch.tensor(bt_priv[:npg], dtype=torch.long, device=tok_pos.device)
        rows = tok_pos.index_select(0, idx).cpu().numpy()        # [npg][L][Hk][P]
    else:
        rows = tok_pos[bt_priv[:npg]]
    out = np.zeros((L, hk, n), np.int64)
    for s in range(n):
        out[:, :, s] = rows[s // P, :, :, s % P]
    return out


class Harness:
    def __init__(self, w: synth.Workload, n_req: int, mode=gpb.GP_MODE_GROWPAGE,
                 num_pages: Optional[int] = None, max_seq_len: Optional[int] = None,
                 tol: Optional[float] = None, budget_pages: Optional[int] = None,
                 random_grow_rate: float = 0.0):
        self.w = w
        self.n = n_req
        self.full_kv = mode == gpb.GP_MODE_FULL_KV
        npages = num_pages or w.num_pages
        self.cfg = gpb.config_for(w, mode=mode, max_requests=n_req, num_pages=npages,
                                  max_seq_len=max_seq_len, random_grow_rate=random_grow_rate)
        self.pool = gpb.Pool(self.cfg)
        self.ora = OraclePool(oracle_config(w, mode, npages, random_grow_rate))
        self.tol = tol if tol is not None else (1e-4 if w.dtype == "f32" else 2e-2)
        self.rep = Report()
        self.arb = _Arbiter(self.rep)
        self.budget = budget_pages or w.budget_pages
        self.lens = synth.draw_lengths(w, n_req)
        self.streams = []
        self.slots = list(range(n_req))
        dev = torch.device("cuda")
        self.dev = dev
        for rid, (pl, T) in enumerate(self.lens):
            st = synth.RequestStream(w, rid, T)
            self.streams.append(st)
            k, v = st.prompt(pl)
            self.pool.add_request(rid, k.to(dev).contiguous(), v.to(dev).contiguous(), self.budget)
            self.ora.add_request(rid, k.double().numpy(), v.double().numpy(), self.budget)
        self.slots_dev = torch.tensor(self.slots, dtype=torch.int32, device=dev)
        L, hq, d = w.num_layers, w.num_q_heads, w.head_dim
        self.outs = [torch.empty(n_req, hq, d, dtype=w.torch_dtype, device=dev) for _ in range(L)]

    # -------------------------------------------------------------------
    def step(self, check=True, after_layer=None):
        """One step on both sides; ``after_layer(l)`` (optional) runs after
        the GPU call of layer l, before the next one."""
        w, rep = self.w, self.rep
        L, hk, hq, d, P = w.num_layers, w.num_kv_heads, w.num_q_heads, w.head_dim, w.page_size
        qs, ks, vs = [], [], []
        for st in self.streams:
            q, k, v = st.next_step()
            qs.append(q); ks.append(k); vs.append(v)
        q = torch.stack(qs)
        k = torch.stack(ks)
        v = torch.stack(vs)
        qd, kd, vd = q.to(self.dev), k.to(self.dev), v.to(self.dev)
        for l in range(L):
            self.pool.decode_step(l, self.slots_dev, qd[:, l].contiguous(), kd[:, l].contiguous(),
                                  vd[:, l].contiguous(), self.outs[l])
            if after_layer is not None:
                after_layer(l)
        self.pool.boundary(self.slots_dev)
        self.pool.sync()
        # GPU state after the step
        metas, bts = {}, {}
        for s in self.slots:
            m, bt = self.pool.request(s)
            metas[s], bts[s] = m, bt
        tok_pos = None
        self.arb.gpu_dec = {}
        self.arb.gpu_kept = {}
        for s in self.slots:
            m = metas[s]
            if m.steps > 0 and m.n_boundaries > 0 and self._had_boundary(s, m):
                self.arb.gpu_dec[s] = m.last_decision
                if m.last_decision in (COMPACT, COMPACT_DENIED, SHRINK):
                    if tok_pos is None:
                        tok_pos = self.pool.region("tok_pos").cpu().numpy()
                    npre = m.n_pre_pages
                    pos = _private_positions(tok_pos, bts[s][npre:], m.seq_priv - 1, L, hk, P)
                    self.arb.gpu_kept[s] = [[set(pos[l, h].tolist()) for h in range(hk)]
                                            for l in range(L)]
        res = self.ora.step(self.slots, q.double().numpy(), k.double().numpy(),
                            v.double().numpy(), arbiter=self.arb)
        rep.steps += 1
        if check:
            self._compare(res, metas, bts, tok_pos)
        self._prev = {s: (metas[s].n_boundaries) for s in self.slots}
        return res

    def _had_boundary(self, s, m):
        prev = getattr(self, "_prev", {}).get(s, 0)
        return m.n_boundaries > prev

    def _compare(self, res, metas, bts, tok_pos):
        w, rep = self.w, self.rep
        L, hk, d, P = w.num_layers, w.num_kv_heads, w.head_dim, w.page_size
        t = rep.steps
        out_g = torch.stack([o.float().cpu() for o in self.outs], 1).double().numpy()  # [n][L][Hq][d]
        out_o = res["out"]
        for i in range(self.n):
            for l in range(L):
                ref = out_o[i, l]
                err = np.max(np.abs(out_g[i, l] - ref)) / max(np.max(np.abs(ref)), 1e-30)
                rep.max_out_err = max(rep.max_out_err, float(err))
                if not err <= self.tol:
                    rep.fail(f"step {t} req {i} layer {l}: output rel err {err:.3g} > {self.tol}")
        summ = self.pool.region("summary")[: self.n].cpu().numpy()
        if not np.array_equal(summ, res["summaries"]):
            bad = np.argwhere(summ != res["summaries"])
            rep.fail(f"step {t}: summaries differ at {bad[:3].tolist()}")
        stg = self.pool.region("staging")[: self.n, :, :, 0].float().cpu().double().numpy()
        if not np.array_equal(stg, res["staged_k"]):
            bad = np.argwhere(stg != res["staged_k"])
            rep.fail(f"step {t}: staged keys differ at {bad[:3].tolist()}")
        wset = None
        for i, s in enumerate(self.slots):
            m, r = metas[s], self.ora.req[s]
            if m.pos != r.pos or m.n_pages != len(r.pages) or m.seq_priv != r.toks.n:
                rep.fail(f"step {t} slot {s}: pos/pages/seq {m.pos},{m.n_pages},{m.seq_priv} "
                         f"vs {r.pos},{len(r.pages)},{r.toks.n}")
            if bts[s] != self.ora.block_table(s):
                rep.fail(f"step {t} slot {s}: block table {bts[s]} vs {self.ora.block_table(s)}")
            rec = res["records"].get(s)
            if rec is None:
                continue
            rep.boundaries += 1
            if m.last_decision != rec.decision:
                rep.fail(f"step {t} slot {s}: decision {m.last_decision} vs {rec.decision} "
                         f"(delta {m.delta} vs {rec.delta}, exempt {rec.decision_exempt})")
            if rec.decision == GROW:
                rep.grows += 1
            elif rec.decision in (COMPACT, COMPACT_DENIED):
                rep.compacts += 1
            elif rec.decision == SHRINK:
                rep.shrinks += 1
            if self.full_kv:
                continue
            if wset is None:
                wset = self.pool.region("wset").cpu().numpy()
            wg = wset[s]  # [L][Hk][2]
            wo = np.stack([rec.w_short, rec.w_long], -1)
            near = rec.w_near_tie
            if not np.array_equal(wg[~near], wo[~near]):
                bad = np.argwhere((wg != wo) & ~near)
                rep.fail(f"step {t} slot {s}: W differs outside near-tie at {bad[:3].tolist()}: "
                         f"{[(int(wg[tuple(b)]), int(wo[tuple(b)])) for b in bad[:3]]}")
            rep.w_in_band += int(np.sum(near & (wg != wo)))
            if not near.any() and m.delta != rec.delta:
                rep.fail(f"step {t} slot {s}: delta {m.delta} vs {rec.delta}")
            if rec.decision in (COMPACT, COMPACT_DENIED, SHRINK):
                if tok_pos is None:
                    tok_pos = self.pool.region("tok_pos").cpu().numpy()
                npre = m.n_pre_pages
                pos = _private_positions(tok_pos, bts[s][npre:], m.seq_priv, L, hk, P)
                got = np.sort(pos, axis=-1)
                want = self.ora.kept_positions(s)
                if not np.array_equal(got, want):
                    rep.fail(f"step {t} slot {s}: kept positions differ")

    def run(self, steps, check_every=1, after_layer=None):
        for t in range(steps):
            self.step(check=(t % check_every == 0), after_layer=after_layer)
            if self.rep.failures:
                break
        return self.rep


class Scenario:
    """A GPU pool and the oracle driven through admissions, steps and frees.

    ``compare_all``: the oracle holds every request and the same pool, so
    block tables are compared exactly.  Otherwise only the requests admitted
    with ``compare=True`` are simulated (each needs nothing from the others
    as long as the GPU pool never runs short of pages, which is checked), and
    page counts, positions and kept-token sets are compared instead of page
    ids.  Inputs come from ``synth.RequestStream`` on ``gen_device``.
    """

    def __init__(self, w, max_requests, num_pages, mode=gpb.GP_MODE_GROWPAGE, compare_all=True,
                 gen_device="cpu", max_seq_len=None, max_prefixes=0, tol=None, oracle_pages=None,
                 side=None, record=False):
        """``side``: a second torch stream; steps then end with
        gp_boundary_async on it.  ``record``: keep every step's slot list,
        inputs and outputs (device tensors) in ``self.trace``."""
        self.side = side
        self.trace = [] if record else None
        self.w = w
        self.full_kv = mode == gpb.GP_MODE_FULL_KV
        self.cfg = gpb.config_for(w, mode=mode, max_requests=max_requests, num_pages=num_pages,
                                  max_seq_len=max_seq_len, max_prefixes=max_prefixes)
        self.pool = gpb.Pool(self.cfg)
        self.compare_all = compare_all
        opages = num_pages if compare_all else (oracle_pages or num_pages)
        self.ora = OraclePool(OracleConfig.from_workload(w, full_kv=self.full_kv, num_pages=opages))
        self.tol = tol if tol is not None else (1e-4 if w.dtype == "f32" else 2e-2)
        self.rep = Report()
        self.arb = _Arbiter(self.rep)
        self.gen = torch.device(gen_device)
        self.dev = torch.device("cuda")
        self.active = {}          # slot -> RequestStream
        self.cmp = set()          # compared slots
        self.gpid, self.opid = {}, {}
        self.prev_nb = {}

    def add_prefix(self, index, compare=True):
        k, v = synth.prefix_tensors(self.w, index, device=self.gen)
        self.gpid[index] = self.pool.add_prefix(k.to(self.dev).contiguous(), v.to(self.dev).contiguous())
        if compare:
            self.opid[index] = self.ora.add_prefix(k.double().cpu().numpy(), v.double().cpu().numpy())
        return self.gpid[index]

    def release_prefix(self, index):
        self.pool.release_prefix(self.gpid.pop(index))
        if index in self.opid:
            self.ora.release_prefix(self.opid.pop(index))

    def admit(self, slot, rid, compare=True, prefix=None, budget_pages=None):
        w = self.w
        pl, T = synth.draw_lengths(w, 1, rid)[0]
        st = synth.RequestStream(w, rid, T, device=self.gen)
        k, v = st.prompt(pl)
        budget = budget_pages or max(w.budget_pages, -(-pl // w.page_size))
        gp = self.gpid[prefix] if prefix is not None else -1
        self.pool.add_request(slot, k.to(self.dev).contiguous() if pl else None,
                              v.to(self.dev).contiguous() if pl else None, budget, gp)
        if compare:
            op = self.opid[prefix] if prefix is not None else -1
            self.ora.add_request(slot, k.double().cpu().numpy(), v.double().cpu().numpy(), budget, op)
            self.cmp.add(slot)
        self.active[slot] = st
        self.prev_nb[slot] = 0
        return T

    def free(self, slot):
        self.pool.free(slot)
        del self.active[slot]
        if slot in self.cmp:
            self.ora.free_request(slot)
            self.cmp.discard(slot)

    def step(self, check=True, exclude=()):
        """One step of the active requests not in ``exclude``; returns the
        slots that were at a boundary (of the compared requests)."""
        w, rep = self.w, self.rep
        L, hk, hq, d, P = w.num_layers, w.num_kv_heads, w.num_q_heads, w.head_dim, w.page_size
        slots = sorted(s for s in self.active if s not in exclude)
        if not slots:
            if self.side is not None:   # an empty step still counts as a step
                empty = torch.zeros(0, dtype=torch.int32, device=self.dev)
                for l in range(L):
                    self.pool.decode_step(l, empty, None, None, None, None)
                self.pool.boundary_async(empty, self.side)
                if self.trace is not None:
                    self.trace.append(([], None, None, None, []))
            return set()
        qs, ks, vs = [], [], []
        for s in slots:
            q, k, v = self.active[s].next_step()
            qs.append(q); ks.append(k); vs.append(v)
        q = torch.stack(qs).to(self.dev)
        k = torch.stack(ks).to(self.dev)
        v = torch.stack(vs).to(self.dev)
        slots_dev = torch.tensor(slots, dtype=torch.int32, device=self.dev)
        outs = []
        for l in range(L):
            o = torch.empty(len(slots), hq, d, dtype=w.torch_dtype, device=self.dev)
            self.pool.decode_step(l, slots_dev, q[:, l].contiguous(), k[:, l].contiguous(),
                                  v[:, l].contiguous(), o)
            outs.append(o)
        if self.side is not None:
            self.pool.boundary_async(slots_dev, self.side)
        else:
            self.pool.boundary(slots_dev)
        if self.trace is not None:
            self.trace.append((list(slots), q, k, v, outs))
        self.pool.sync()
        cslots = sorted(s for s in self.cmp if s in slots)
        idx = [slots.index(s) for s in cslots]
        metas, bts = {}, {}
        for s in cslots:
            metas[s], bts[s] = self.pool.request(s)
        st = self.pool.stats()
        if not self.compare_all and st.denied:
            rep.fail("the GPU pool ran short of pages: sampled comparison no longer valid")
        tok_pos = None
        self.arb.gpu_dec, self.arb.gpu_kept = {}, {}
        for s in cslots:
            m = metas[s]
            if m.n_boundaries > self.prev_nb[s]:
                self.arb.gpu_dec[s] = m.last_decision
                if m.last_decision in (COMPACT, COMPACT_DENIED, SHRINK):
                    tok_pos = self.pool.region("tok_pos")
                    pos = _private_positions(tok_pos, bts[s][m.n_pre_pages:], m.seq_priv - 1, L, hk, P)
                    self.arb.gpu_kept[s] = [[set(pos[l, h].tolist()) for h in range(hk)] for l in range(L)]
        bnd = set()
        if cslots:
            qc = q[idx].double().cpu().numpy()
            kc = k[idx].double().cpu().numpy()
            vc = v[idx].double().cpu().numpy()
            res = self.ora.step(cslots, qc, kc, vc, arbiter=self.arb)
            rep.steps += 1
            bnd = set(res["records"])
            if check:
                out_g = torch.stack([o[idx].float().cpu() for o in outs], 1).double().numpy()
                self._compare(res, cslots, out_g, metas, bts, tok_pos)
        for s in cslots:
            self.prev_nb[s] = metas[s].n_boundaries
        return bnd

    def _compare(self, res, cslots, out_g, metas, bts, tok_pos):
        w, rep = self.w, self.rep
        L, hk, P = w.num_layers, w.num_kv_heads, w.page_size
        t = rep.steps
        for ci, s in enumerate(cslots):
            for l in range(L):
                ref = res["out"][ci, l]
                err = np.max(np.abs(out_g[ci, l] - ref)) / max(np.max(np.abs(ref)), 1e-30)
                rep.max_out_err = max(rep.max_out_err, float(err))
                if not err <= self.tol:
                    rep.fail(f"step {t} slot {s} layer {l}: output rel err {err:.3g} > {self.tol}")
        summ = self.pool.region("summary")[cslots].cpu().numpy()
        if not np.array_equal(summ, res["summaries"]):
            rep.fail(f"step {t}: summaries differ")
        stg = self.pool.region("staging")[cslots][:, :, :, 0].float().cpu().double().numpy()
        if not np.array_equal(stg, res["staged_k"]):
            rep.fail(f"step {t}: staged keys differ")
        wset = None
        for s in cslots:
            m, r = metas[s], self.ora.req[s]
            if m.pos != r.pos or m.n_pages != len(r.pages) or m.seq_priv != r.toks.n:
                rep.fail(f"step {t} slot {s}: pos/pages/seq {m.pos},{m.n_pages},{m.seq_priv} "
                         f"vs {r.pos},{len(r.pages)},{r.toks.n}")
            if self.compare_all and bts[s] != self.ora.block_table(s):
                rep.fail(f"step {t} slot {s}: block table {bts[s]} vs {self.ora.block_table(s)}")
            rec = res["records"].get(s)
            if rec is None:
                continue
            rep.boundaries += 1
            if m.last_decision != rec.decision:
                rep.fail(f"step {t} slot {s}: decision {m.last_decision} vs {rec.decision}")
            if rec.decision == GROW:
                rep.grows += 1
            elif rec.decision in (COMPACT, COMPACT_DENIED):
                rep.compacts += 1
            elif rec.decision == SHRINK:
                rep.shrinks += 1
            if self.full_kv:
                continue
            if wset is None:
                wset = self.pool.region("wset").cpu().numpy()
            wg = wset[s]
            wo = np.stack([rec.w_short, rec.w_long], -1)
            near = rec.w_near_tie
            if not np.array_equal(wg[~near], wo[~near]):
                rep.fail(f"step {t} slot {s}: W differs outside near-ties")
            rep.w_in_band += int(np.sum(near & (wg != wo)))
            if not near.any() and m.delta != rec.delta:
                rep.fail(f"step {t} slot {s}: delta {m.delta} vs {rec.delta}")
            if rec.decision in (COMPACT, COMPACT_DENIED, SHRINK):
                pos = _private_positions(self.pool.region("tok_pos"), bts[s][m.n_pre_pages:],
                                         m.seq_priv, L, hk, P)
                if not np.array_equal(np.sort(pos, axis=-1), self.ora.kept_positions(s)):
                    rep.fail(f"step {t} slot {s}: kept positions differ")
