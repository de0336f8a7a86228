"""The engine's host logic (no GPU): admission, retirement and refill, and
full-KV preemption, against a fake pool that keeps the same page books as the
device and refuses any step the pool could not serve."""
import pytest
import torch

from demand_paged_kv_gqa_b300 import engine as engmod
from demand_paged_kv_gqa_b300 import growpage as gpb
from demand_paged_kv_gqa_b300 import synth


class FakePool:
    def __init__(self, cfg, device=None):
        self.cfg = cfg
        self.P = cfg.page_size
        self.free_top = cfg.num_pages
        self.req = {}           # slot -> [pages, seq, prefix id]
        self.prefixes = {}      # prefix id -> [pages, references]
        self.next_pid = 0
        self.stream = None
        self.steps = 0

    def add_prefix(self, k, v):
        npg = k.shape[1] // self.P
        assert npg <= self.free_top
        self.free_top -= npg
        pid = self.next_pid
        self.next_pid += 1
        self.prefixes[pid] = [npg, 1]
        return pid

    def _unref(self, pid):
        pf = self.prefixes[pid]
        pf[1] -= 1
        if pf[1] == 0:
            self.free_top += pf[0]
            del self.prefixes[pid]

    def release_prefix(self, pid):
        self._unref(pid)

    def add_request(self, slot, k, v, budget, prefix_id=-1):
        n = 0 if k is None else k.shape[1]
        assert slot not in self.req and budget <= self.free_top
        self.free_top -= budget
        self.req[slot] = [budget, n, prefix_id]
        if prefix_id >= 0:
            self.prefixes[prefix_id][1] += 1

    def free(self, slot):
        pages, _, pid = self.req.pop(slot)
        self.free_top += pages
        if pid >= 0:
            self._unref(pid)

    def stats(self):
        class S:
            pass
        s = S()
        s.free_top = self.free_top
        return s

    def decode_step(self, layer, slots, q, k, v, out):
        assert q.shape[0] == slots.numel() == out.shape[0]

    def boundary(self, slots):
        self.steps += 1
        full_kv = self.cfg.mode == gpb.GP_MODE_FULL_KV
        for s in slots.tolist():
            pages, seq, pid = self.req[s]
            if seq == pages * self.P:
                if full_kv:
                    if self.free_top == 0:
                        raise AssertionError("full-KV step with no free page: engine did not preempt")
                    self.free_top -= 1
                    pages += 1
                else:
                    seq -= self.P      # compaction frees one page of slots
            self.req[s] = [pages, seq + 1, pid]


@pytest.fixture
def fake(monkeypatch):
    monkeypatch.setattr(gpb, "Pool", FakePool)


def _workload():
    # 4 slots of the tiny shapes with short outputs, so requests retire
    return synth.WORKLOADS["tiny"].replace(batch=4, prompt_min=20, prompt_max=40,
                                           out_median=60, out_sigma=0.5, out_min=30,
                                           out_max=120, budget_pages=3)


def test_growpage_refills_slots_and_counts_tokens(fake):
    w = _workload()
    eng = engmod.Engine(w, mode=gpb.GP_MODE_GROWPAGE, device="cpu", num_pages=40)
    eng.fill()
    assert len(eng.active()) == 4
    total = 0
    for _ in range(300):
        eng.prepare_inputs()
        total += eng.step()
    assert eng.finished > 4                  # requests retired and slots were refilled
    assert eng.tokens == total
    produced = sum(r.produced for r in eng.slots if r is not None)
    assert total >= produced
    # books agree with the pool's: every active slot holds its pages
    held = sum(p for p, _, _ in eng.pool.req.values())
    assert held + eng.pool.free_top == 40


def test_full_kv_preempts_newest_and_requeues(fake):
    w = _workload()
    eng = engmod.Engine(w, mode=gpb.GP_MODE_FULL_KV, device="cpu", num_pages=18)
    eng.fill()
    total = 0
    for _ in range(400):
        eng.prepare_inputs()
        total += eng.step()
        # the host's exact page count matches the pool's
        assert eng.free_pages == eng.pool.free_top
    assert eng.preempted > 0
    # preempted requests lose their produced tokens from the count
    assert eng.tokens <= total
    assert eng.finished > 0


def _boundaries_match(eng):
    # the host's free-slot count equals the pool's for every active request
    for s in eng.active():
        pages, seq, _ = eng.pool.req[s]
        assert eng.slots[s].free_slots == pages * eng.P - seq


@pytest.mark.parametrize("mode", [gpb.GP_MODE_GROWPAGE, gpb.GP_MODE_FULL_KV])
def test_poisson_arrivals_and_shared_prefixes(fake, mode):
    # requests arrive on the virtual clock and are admitted first come first
    # served; each group of 3 shares one prefix, which lives while any member
    # does; the run drains completely and every page comes back
    w = synth.WORKLOADS["tiny"].replace(batch=5, prompt_min=0, prompt_max=0, prefix_len=32,
                                        prefix_group=3, arrival_rate=4.0, step_seconds=0.02,
                                        total_requests=14, out_median=50, out_sigma=0.5,
                                        out_min=20, out_max=120, budget_pages=2)
    eng = engmod.Engine(w, mode=mode, device="cpu", num_pages=30)
    arrivals = eng.arrivals
    eng.fill()
    seen = set()
    for t in range(2000):
        if eng.drained():
            break
        eng.prepare_inputs()
        eng.step()
        _boundaries_match(eng)
        for s in eng.active():
            r = eng.slots[s]
            if r.rid not in seen:
                seen.add(r.rid)
                assert arrivals[r.rid] <= eng.clock       # never admitted before arriving
        live = {g for g, grp in eng.groups.items() if grp.pid >= 0}
        assert len(live) == len(eng.pool.prefixes)
        for g in live:
            users = sum(1 for s in eng.active() if eng.slots[s].group == g)
            pf = eng.pool.prefixes[eng.groups[g].pid]
            assert pf[1] == users + int(eng.groups[g].held)
        if mode == gpb.GP_MODE_FULL_KV:
            assert eng.free_pages == eng.pool.free_top
    assert eng.drained() and eng.finished == 14
    assert not eng.pool.prefixes and eng.pool.free_top == 30
    # arrivals are spread out: about 0.08 per step
    assert 100 < arrivals[13] < 400


def test_at_boundary_counts_lockstep_requests(fake):
    # prompts of exactly the budget: every request is at a boundary on the
    # first step and every P steps after it
    w = synth.WORKLOADS["tiny"].replace(batch=4, prompt_min=32, prompt_max=32, budget_pages=2,
                                        decode_steps=100)
    eng = engmod.Engine(w, device="cpu", num_pages=40)
    eng.fill()
    counts = []
    for _ in range(40):
        eng.prepare_inputs()
        eng.step()
        counts.append(eng.last_boundaries)
        _boundaries_match(eng)
    assert counts == [4 if t % 16 == 0 else 0 for t in range(40)]
