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
        self.req = {}           # slot -> [pages, seq]
        self.stream = None
        self.steps = 0

    def add_request(self, slot, k, v, budget):
        assert slot not in self.req and budget <= self.free_top
        self.free_top -= budget
        self.req[slot] = [budget, k.shape[1]]

    def free(self, slot):
        pages, _ = self.req.pop(slot)
        self.free_top += pages

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
            pages, seq = self.req[s]
            if seq == pages * self.P:
                if full_kv:
                    if self.free_top == 0:
                        raise AssertionError("full-KV step with no free page: engine did not preempt")
                    self.free_top -= 1
                    pages += 1
                else:
                    seq -= self.P      # compaction frees one page of slots
            self.req[s] = [pages, seq + 1]


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
    held = sum(p for p, _ in eng.pool.req.values())
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
