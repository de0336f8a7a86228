"""Host-side decode loop around the C-ABI library: continuous batching.

The pages ("GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning
Serving", abstract) keep continuous batching and prefix caching on top of
PagedAttention's page-level memory.  This module is the host half of that:
it admits requests into free slots when the pool has their initial budget,
runs one decode step (all layers, then the boundary call) for the active
slots, retires requests that reached their output length and refills their
slots.  Every arithmetic step of the decode path runs in the library's
kernels; this module only decides which slots take part.

Arrivals.  A workload with an arrival rate draws Poisson arrival times on a
virtual clock of ``step_seconds`` per decode step (``synth.poisson_arrivals``)
and admits arrived requests first come, first served, up to its slot count
and ``total_requests``.  Without a rate, a new request is always waiting.

Shared prefixes.  A workload with ``prefix_len`` > 0 gives each group of
``prefix_group`` consecutive requests one shared prefix (prefix caching):
the first member to be admitted stores it (``gp_add_prefix``), every member
references it, and the engine drops its creator reference once every member
has been admitted, so the prefix's pages return to the pool when its last
member leaves.  A preempted member re-admitted later re-creates it if needed.

Boundaries.  Both outcomes of a boundary (grow, or compact within the
allocation) leave P - 1 free private slots after the step's token is
appended, so the host knows, without reading the device, how many steps
each request has until its next boundary.  The engine counts the requests
at a boundary in each step (``last_boundaries``).

Full-KV mode (every boundary grows) cannot compact when the pool runs dry.
There the engine preempts, as a PagedAttention server does by recomputation:
before a step whose boundaries need more pages than are free, the most
recently admitted requests release their pages and go back to the head of
the queue; the tokens they had produced are subtracted from the count.
In full-KV mode page use is a function of the step count alone, so the host
tracks it exactly without reading the device.  Its page cap per request is
raised to hold the longest request, so that a request never starves at it.

Graphs.  With ``use_graph``, a step in which every slot takes part is
captured once as a CUDA graph (all layers and the boundary call) and
replayed: the slot list and the q / k / v / out buffers are then the same
tensors every step, and everything else the step reads lives in the pool's
device state.  This removes the host's launch cost from steps too short to
hide it (a single layer).

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
    n_pages: int = 0       # private pages (full-KV bookkeeping)
    seq_priv: int = 0      # private tokens (full-KV bookkeeping)
    free_slots: int = 0    # private slots left: 0 = at a boundary at step start
    group: int = -1        # shared-prefix group (-1: none)


@dataclasses.dataclass
class _Group:
    pid: int = -1          # device prefix id, -1 while not stored
    members: int = 0       # admitted members still holding it
    held: bool = False     # the engine's creator reference
    admitted: int = 0      # members admitted at least once


class Engine:
    def __init__(self, w: synth.Workload, mode=gpb.GP_MODE_GROWPAGE, device="cuda",
                 num_pages: Optional[int] = None, batch: Optional[int] = None,
                 seed_offset: int = 0, max_seq_len: Optional[int] = None,
                 random_grow_rate: float = 0.0, async_boundary: bool = False,
                 use_graph: bool = False):
        self.w = w
        self.mode = mode
        self.full_kv = mode == gpb.GP_MODE_FULL_KV
        self.device = torch.device(device)
        self.batch = batch or w.batch
        self.P = w.page_size
        max_out = max(w.decode_steps, w.out_max)
        cap = None
        if self.full_kv:
            cap = max(w.max_pages_per_req, -(-(w.prompt_max + max_out) // self.P) + 1)
        self.grp = w.prefix_group if w.prefix_len > 0 else 0
        self.cfg = gpb.config_for(w, mode=mode, max_requests=self.batch,
                                  num_pages=num_pages or w.num_pages, max_seq_len=max_seq_len,
                                  random_grow_rate=random_grow_rate, max_pages_per_req=cap,
                                  max_prefixes=(self.batch + 2) if self.grp else None)
        self.pool = gpb.Pool(self.cfg, device=self.device)
        self.num_pages = self.cfg.num_pages
        self.seed_offset = seed_offset
        self.slots: List[Optional[Req]] = [None] * self.batch
        self.admit_order: List[int] = []          # slots, oldest first
        self.queue: collections.deque = collections.deque()
        self.rid0 = seed_offset * 1_000_000
        self.next_rid = self.rid0
        self.total = w.total_requests or None
        self.arrivals = (synth.poisson_arrivals(w, self.total or 1 << 16)
                         if w.arrival_rate > 0 else None)
        self.clock = 0                            # decode steps on the virtual clock
        self.lengths_cache: Dict[int, tuple] = {}
        self.groups: Dict[int, _Group] = {}
        self.prefix_pages = w.prefix_len // self.P
        self.gen = synth.BatchStream(w, self.batch, [1] * self.batch, device=self.device,
                                     seed=seed_offset)
        self.free_pages = self.num_pages          # full-KV: exact; else refreshed
        self.tokens = 0
        self.tokens_timed = 0
        self.preempted = 0
        self.finished = 0
        self.steps = 0
        self.last_boundaries = 0
        # asynchronous boundary work: the requests at a boundary in a step get
        # their boundary work on a second stream and sit out the next step
        self.side = torch.cuda.Stream(device=self.device) if async_boundary else None
        self.out_of_step = set()
        self.use_graph = use_graph and not async_boundary
        self._graph = None
        self.graph_launches = 0     # library launches replayed through the graph
        self._graph_per_step = 0
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

    def _arrive(self):
        """Queue the requests that have arrived by the current clock."""
        if self.arrivals is None:
            return                                # no clock: made on demand in fill()
        while self.total is None or self.next_rid - self.rid0 < self.total:
            if self.arrivals[self.next_rid - self.rid0] > self.clock:
                return
            self.queue.append(self.next_rid)
            self.next_rid += 1

    def _take_new(self) -> bool:
        """Without an arrival clock a new request is always waiting."""
        if self.arrivals is not None:
            return False
        if self.total is not None and self.next_rid - self.rid0 >= self.total:
            return False
        self.queue.append(self.next_rid)
        self.next_rid += 1
        return True

    def _refresh_free(self):
        if not self.full_kv:
            self.free_pages = int(self.pool.stats().free_top)

    def _group_of(self, rid):
        return (rid - self.rid0) // self.grp if self.grp else -1

    def _admit(self, slot, rid) -> bool:
        w = self.w
        pl, T = self._lengths(rid)
        budget = max(w.budget_pages, -(-pl // self.P))
        g = self._group_of(rid)
        grp = self.groups.setdefault(g, _Group()) if g >= 0 else None
        need = budget + (self.prefix_pages if grp is not None and grp.pid < 0 else 0)
        if self.full_kv:
            # keep one page per running request for its next grow, so that a
            # request preempted for pages is not re-admitted straight away
            need += len(self.admit_order)
        if self.free_pages < need:
            return False
        st = synth.RequestStream(w, rid, T, device=self.device)
        pid = -1
        if grp is not None:
            if grp.pid < 0:
                pk, pv = synth.prefix_tensors(w, g, device=self.device)
                grp.pid = self.pool.add_prefix(pk.contiguous(), pv.contiguous())
                grp.held = True
                self.free_pages -= self.prefix_pages
            pid = grp.pid
        if pl > 0:
            k, v = st.prompt(pl)
            self.pool.add_request(slot, k.contiguous(), v.contiguous(), budget, pid)
        else:
            self.pool.add_request(slot, None, None, budget, pid)
        self.slots[slot] = Req(rid, pl, T, n_pages=budget, seq_priv=pl,
                               free_slots=budget * self.P - pl, group=g)
        self.admit_order.append(slot)
        self.free_pages -= budget
        self.gen.reset_request(slot, T)
        if grp is not None:
            grp.members += 1
            grp.admitted += 1
            size = self.grp if self.total is None else min(self.grp, self.total - g * self.grp)
            if grp.held and grp.admitted >= size:
                self.pool.release_prefix(grp.pid)   # members keep it alive
                grp.held = False
        return True

    def fill(self):
        """Admit arrived requests, first come first served, into free slots."""
        self._arrive()
        for slot in range(self.batch):
            if self.slots[slot] is not None:
                continue
            if not self.queue and not self._take_new():
                break
            if not self._admit(slot, self.queue[0]):
                break
            self.queue.popleft()

    def _release(self, slot):
        r = self.slots[slot]
        self.pool.free(slot)
        self.slots[slot] = None
        self.admit_order.remove(slot)
        self.out_of_step.discard(slot)
        if self.full_kv:
            self.free_pages += r.n_pages
        if r.group >= 0:
            grp = self.groups[r.group]
            grp.members -= 1
            if grp.members == 0 and not grp.held:   # its last reference went
                grp.pid = -1
                if self.full_kv:
                    self.free_pages += self.prefix_pages
        return r

    # ------------------------------------------------------------- stepping
    def active(self) -> List[int]:
        return [s for s in range(self.batch) if self.slots[s] is not None]

    def stepping(self) -> List[int]:
        """Active slots that take part in the next step."""
        return [s for s in self.active() if s not in self.out_of_step]

    def at_boundary(self) -> List[int]:
        """Slots of the next step whose private pages are full at its start."""
        return [s for s in self.stepping() if self.slots[s].free_slots == 0]

    def _preempt_for_step(self):
        """Full-KV: free the newest requests until this step's grows fit."""
        while True:
            need = len(self.at_boundary())
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

    def _replay(self, slots_dev):
        """One full step through the captured graph (captured on first use)."""
        if self._graph is None:
            L = self.w.num_layers
            home = self.pool.stream
            g = torch.cuda.CUDAGraph()
            n0 = self.pool.launch_count()
            with torch.cuda.graph(g):
                self.pool.set_stream(torch.cuda.current_stream())
                for l in range(L):
                    self.pool.decode_step(l, slots_dev, self.q[l], self.k[l], self.v[l], self.out[l])
                self.pool.boundary(slots_dev)
            self.pool.set_stream(home)
            self._graph = g
            self._graph_per_step = self.pool.launch_count() - n0
        self._graph.replay()
        self.graph_launches += self._graph_per_step

    def drained(self) -> bool:
        """No request active, queued or still to arrive."""
        return (not self.active() and not self.queue and self.total is not None
                and self.next_rid - self.rid0 >= self.total)

    def step(self, timed=False, before_step: Optional[Callable] = None,
             after_layer: Optional[Callable] = None, after_step: Optional[Callable] = None,
             before_layer: Optional[Callable] = None):
        """One decode step for the active slots; returns the number of tokens.

        The virtual clock advances by one step even when no request is active
        (requests still to arrive)."""
        if self.full_kv:
            self._preempt_for_step()
        act = self.stepping()
        n = len(act)
        self.clock += 1
        if n == 0:
            if self.side is not None and self.out_of_step:
                # the library counts steps by calls: a step with no request
                # still separates the boundary work from the requests' return
                empty = torch.zeros(0, dtype=torch.int32, device=self.device)
                for l in range(self.w.num_layers):
                    self.pool.decode_step(l, empty, None, None, None, None)
                self.pool.boundary_async(empty, self.side)
            self.last_boundaries = 0
            self.out_of_step = set()
            self._refresh_free()
            self.fill()
            return 0
        self.last_boundaries = sum(1 for s in act if self.slots[s].free_slots == 0)
        slots_dev = self._slot_tensor(act)
        if n == self.batch:
            q, k, v = self.q, self.k, self.v
        else:  # gather the active rows before the step starts
            idx = torch.tensor(act, device=self.device)
            q, k, v = self.q[:, idx], self.k[:, idx], self.v[:, idx]
        L = self.w.num_layers
        if before_step:
            before_step()
        if self.use_graph and n == self.batch and not (before_layer or after_layer):
            self._replay(slots_dev)
        else:
            for l in range(L):
                if before_layer:
                    before_layer(l)
                self.pool.decode_step(l, slots_dev, q[l], k[l], v[l], self.out[l, :n])
                if after_layer:
                    after_layer(l)
            if self.side is not None:
                self.pool.boundary_async(slots_dev, self.side)
            else:
                self.pool.boundary(slots_dev)
        if after_step:
            after_step()
        if self.side is not None:
            self.out_of_step = {s for s in act if self.slots[s].free_slots == 0}
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
            if r.free_slots == 0:                # a boundary: P - 1 slots left either way
                r.free_slots = self.P - 1
                if self.full_kv:
                    r.n_pages += 1
                    self.free_pages -= 1
            else:
                r.free_slots -= 1
            r.seq_priv += 1
            if r.produced >= r.out_len:
                done.append(s)
        for s in done:
            self._release(s)
            self.finished += 1
        # admit when a slot was freed or a request arrived; a request waiting
        # for pages is retried every P steps (pages move only at boundaries)
        queued = len(self.queue)
        self._arrive()
        if done or len(self.queue) > queued or (queued and self.clock % self.P == 0):
            self._refresh_free()
            self.fill()
        return n
