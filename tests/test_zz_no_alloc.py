"""The read-ceiling entry point that needs no caller scratch.

gp_kv_read_ceiling_static is for callers that cannot allocate device memory
at the point of the call (a fixed memory arena, an allocator that must not be
entered there): its per-call scratch is a static device array of the
library.  It must read exactly what gp_kv_read_ceiling reads, and, since it
leaves the pool's own scratch alone, calling it between two layers of a step
must not change that step.  This file is collected last, so a failure here
comes after every other test has run.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _sink_result(sink):
    s = [int(x) & 0xFFFFFFFF for x in sink.cpu().tolist()]
    return s[0], s[2] | (s[3] << 32)


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def test_static_scratch_read_matches_pool_scratch_read():
    _need_gpu()
    from demand_paged_kv_gqa_b300 import synth
    from demand_paged_kv_gqa_b300.engine import Engine

    # A 2-layer, 32q/8kv, d=128 bf16 pool with 12 requests and some decode
    # history, so that pages are scattered and pieces are cut between workers.
    w = synth.WORKLOADS["llama8b_32layer"].replace(num_layers=2, batch=12)
    eng = Engine(w, num_pages=2048)
    eng.fill()
    for _ in range(40):
        eng.prepare_inputs()
        eng.step()
    eng.pool.sync()
    slots = torch.tensor(eng.active(), dtype=torch.int32, device="cuda")
    for mode in (0, 1, 2):
        ref = torch.zeros(4, dtype=torch.int32, device="cuda")
        eng.pool.kv_read_ceiling(0, 2, mode, slots, ref)
        eng.pool.sync()
        want = _sink_result(ref)
        assert want[1] > 0
        for _call in range(2):  # two calls in a row share the static array
            got = torch.zeros(4, dtype=torch.int32, device="cuda")
            eng.pool.kv_read_ceiling_static(0, 2, mode, slots, got)
            eng.pool.sync()
            assert _sink_result(got) == want, (mode, _call)


def test_static_scratch_limit_is_refused():
    # a pool with more request slots than the static array holds: n = 1025 is
    # refused by the static limit itself, before anything is launched
    _need_gpu()
    from demand_paged_kv_gqa_b300 import growpage as gpb
    cfg = gpb.make_config(num_layers=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                          page_size=16, num_pages=64, max_requests=1100, max_pages_per_req=4,
                          dtype=gpb.GP_DTYPE_BF16, max_seq_len=128)
    pool = gpb.Pool(cfg)
    n0 = pool.launch_count()
    with pytest.raises(gpb.GrowPageError, match="static scratch limit") as e:
        pool.kv_read_ceiling_static(0, 1, 0, torch.zeros(1025, dtype=torch.int32, device="cuda"),
                                    torch.zeros(4, dtype=torch.int32, device="cuda"))
    assert e.value.code == gpb.GP_ERR_INVALID
    assert pool.launch_count() == n0
    pool.sync()


def test_static_scratch_read_inside_a_step_changes_nothing():
    # The static call made between the two layers of every step: the run stays
    # in step with the CPU oracle (outputs, summaries, decisions, block tables,
    # kept tokens), and its outputs are bit-identical to a run without it.
    _need_gpu()
    from tests import gpu_harness as H
    from demand_paged_kv_gqa_b300 import synth
    w = synth.WORKLOADS["llama8b_1layer"].replace(num_layers=2, prompt_min=100, prompt_max=128,
                                                  budget_pages=8, max_pages_per_req=16)
    with_calls = H.Harness(w, 4, budget_pages=8)
    plain = H.Harness(w, 4, budget_pages=8)
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")

    def read_between(l):
        if l == 0:
            with_calls.pool.kv_read_ceiling_static(0, 2, 0, with_calls.slots_dev, sink)

    for t in range(70):
        with_calls.step(after_layer=read_between)
        plain.step(check=False)
        assert not with_calls.rep.failures, "\n".join(with_calls.rep.failures)
        for a, b in zip(with_calls.outs, plain.outs):
            assert torch.equal(a, b), t
    assert with_calls.rep.boundaries >= 12
    assert _sink_result(sink)[1] > 0
