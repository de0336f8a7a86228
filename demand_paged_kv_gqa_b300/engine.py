"""Host-side decode loop around the C-ABI library: continuous batching.

The pages ("GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning
Serving", abstract) keep continuous batching and prefix caching on top of
PagedAttention's page-level memory.  This module is the host half of that:
it admits requests into free slots when the pool has their initial budget,
runs one decode step (all layers, then the boundary call) for the active
slots, retires requests that reached their output length and refills their
slots.  Every arithmetic step of the decode path runs in the library's
kernels; this module only decides which slots take part.

Full-KV mode (every boundary grows) cannot compact when the pool runs dry.
There the engine preempts, as a PagedAttention server does by recomputation:
before a step whose boundaries need more pages than are free, the most
recently admitted requests release their pages and go back to the head of
the queue; the tokens they had produced are subtracted from the count.
In full-KV mode page use is a function of the step count alone, so the host
tracks it exactly without reading the device.

Inputs are drawn on the device by ``synth.BatchStream`` (the workload's
recipe, batched); this module does not time anything itself but exposes
hooks (``before_step`` / ``after_layer`` / ``after_step``) for events.
"""
from __future__ import annotations

import collections
import dataclasses
from typing import Callable, Dict, List, Optional

import torch

from . import growpage as gpb
from . import synth


@dataclasses.dataclass
class Req:
    rid: int
    prompt_len: int
    out_len: int
    produced: int = 0
    produced_timed: int = 0
    n_pages: int = 0       # full-KV bookkeeping only
    seq_priv: int = 0
    prefix_id: int = -1


class Engine:
    def __init__(self, w: synth.Workload, mode=gpb.GP_MODE_GROWPAGE, device="cuda",
                 num_pages: Optional[int] = None, batch: Optional[int] = None,
                 seed_offset: int = 0, max_seq_len: Optional[int] = None,
                 random_grow_rate: float = 0.0):
        self.w = w
        self.mode = mode
        self.full_kv = mode == gpb.GP_MODE_FULL_KV
        self.device = torch.device(device)
        self.batch = batch or w.batch
        self.cfg = gpb.config_for(w, mode=mode, max_requests=self.batch,
                                  num_pages=num_pages or w.num_pages, max_seq_len=max_seq_len,
                                  random_grow_rate=random_grow_rate)
        self.pool = gpb.Pool(self.cfg, device=self.device)
        self.num_pages = self.cfg.num_pages
        self.P = w.page_size
        self.seed_offset = seed_offset
        self.slots: List[Optional[Req]] = [None] * self.batch
        self.admit_order: List[int] = []          # slots, oldest first
        self.queue: collections.deque = collections.deque()
        self.next_rid = seed_offset * 1_000_000
        self.lengths_cache: Dict[int, tuple] = {}
        self.gen = synth.BatchStream(w, self.batch, [1] * self.batch, device=self.device,
                                     seed=seed_offset)
        self.free_pages = self.num_pages          # full-KV: exact; else refreshed
        self.tokens = 0
        self.tokens_timed = 0
        self.preempted = 0
        self.finished = 0
        self.steps = 0
        self._slots_dev = None
        self._active_key = None
        L, hq, hk, d = w.num_layers, w.num_q_heads, w.num_kv_heads, w.head_dim
        dt = w.torch_dtype
        self.q = torch.empty(L, self.batch, hq, d, dtype=dt, device=self.device)
        self.k = torch.empty(L, self.batch, hk, d, dtype=dt, device=self.device)
        self.v = torch.empty(L, self.batch, hk, d, dtype=dt, device=self.device)
        self.out = torch.empty(L, self.batch, hq, d, dtype=dt, device=self.device)

    # ------------------------------------------------------------ admission
    def _lengths(self, rid):
        if rid not in self.lengths_cache:
            self.lengths_cache[rid] = synth.draw_lengths(self.w, 1, rid)[0]
        return self.lengths_cache[rid]

    def _new_rid(self):
        rid = self.next_rid
        self.next_rid += 1
        return rid

    def _refresh_free(self):
        if not self.full_kv:
            self.free_pages = int(self.pool.stats().free_top)

    def _admit(self, slot, rid) -> bool:
        w = self.w
        pl, T = self._lengths(rid)
        budget = max(w.budget_pages, -(-pl // self.P))
        if self.free_pages < budget:
            return False
        st = synth.RequestStream(w, rid, T, device=self.device)
        k, v = st.prompt(pl)
        self.pool.add_request(slot, k.contiguous(), v.contiguous(), budget)
        self.slots[slot] = Req(rid, pl, T, n_pages=budget, seq_priv=pl)
        self.admit_order.append(slot)
        self.free_pages -= budget
        self.gen.reset_request(slot, T)
        return True

    def fill(self):
        """Admit queued or new requests into every free slot that fits."""
        for slot in range(self.batch):
            if self.slots[slot] is not None:
                continue
            if not self.queue:
                self.queue.append(self._new_rid())
            if not self._admit(slot, self.queue[0]):
                break
            self.queue.popleft()

    def _release(self, slot):
        r = self.slots[slot]
        self.pool.free(slot)
        self.slots[slot] = None
        self.admit_order.remove(slot)
        if self.full_kv:
            self.free_pages += r.n_pages
        return r

    # ------------------------------------------------------------- stepping
    def active(self) -> List[int]:
        return [s for s in range(self.batch) if self.slots[s] is not None]

    def _preempt_for_step(self):
        """Full-KV: free the newest requests until this step's grows fit."""
        while True:
            need = sum(1 for s in self.active()
                       if self.slots[s].seq_priv == self.slots[s].n_pages * self.P)
            if need <= self.free_pages or not self.admit_order:
                return
            slot = self.admit_order[-1]
            r = self._release(slot)
            self.tokens -= r.produced
            self.tokens_timed -= r.produced_timed
            self.preempted += 1
            self.queue.appendleft(r.rid)

    def prepare_inputs(self):
        """Draw the next step's q, k, v for every slot (device, layer-major)."""
        q, k, v = self.gen.next_step()           # [n][L][H][d]
        self.q.copy_(q.transpose(0, 1))
        self.k.copy_(k.transpose(0, 1))
        self.v.copy_(v.transpose(0, 1))

    def _slot_tensor(self, act):
        key = tuple(act)
        if key != self._active_key:
            self._slots_dev = torch.tensor(act, dtype=torch.int32, device=self.device)
            self._active_key = key
        return self._slots_dev

    def step(self, timed=False, before_step: Optional[Callable] = None,
             after_layer: Optional[Callable] = None, after_step: Optional[Callable] = None,
             before_layer: Optional[Callable] = None):
        """One decode step for the active slots; returns the number of tokens."""
        if self.full_kv:
            self._preempt_for_step()
        act = self.active()
        n = len(act)
        if n == 0:
            return 0
        slots_dev = self._slot_tensor(act)
        if n == self.batch:
            q, k, v = self.q, self.k, self.v
        else:  # gather the active rows before the step starts
            idx = torch.tensor(act, device=self.device)
            q, k, v = self.q[:, idx], self.k[:, idx], self.v[:, idx]
        L = self.w.num_layers
        if before_step:
            before_step()
        for l in range(L):
            if before_layer:
                before_layer(l)
            self.pool.decode_step(l, slots_dev, q[l], k[l], v[l], self.out[l, :n])
            if after_layer:
                after_layer(l)
        self.pool.boundary(slots_dev)
        if after_step:
            after_step()
        # host bookkeeping
        self.steps += 1
        self.tokens += n
        if timed:
            self.tokens_timed += n
        done = []
        for s in act:
            r = self.slots[s]
            r.produced += 1
            if timed:
                r.produced_timed += 1
            if self.full_kv:
                if r.seq_priv == r.n_pages * self.P:
                    r.n_pages += 1
                    self.free_pages -= 1
                r.seq_priv += 1
            if r.produced >= r.out_len:
                done.append(s)
        for s in done:
            self._release(s)
            self.finished += 1
        if done or self.queue:
            self._refresh_free()
            self.fill()
        return n
