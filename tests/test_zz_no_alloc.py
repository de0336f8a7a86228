"""The read-ceiling entry point that needs no caller scratch.

gp_kv_read_ceiling_static is for callers that cannot allocate device memory
at the point of the call (a fixed memory arena, an allocator that must not be
entered there): its per-call scratch is a static device array of the
library.  It must read exactly what gp_kv_read_ceiling reads.  This file is
collected last, so a failure here comes after every other test has run.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _sink_result(sink):
    s = [int(x) & 0xFFFFFFFF for x in sink.cpu().tolist()]
    return s[0], s[2] | (s[3] << 32)


def test_static_scratch_read_matches_pool_scratch_read():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from demand_paged_kv_gqa_b300 import growpage as gpb
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
    # beyond the static maximum: a clear error, nothing launched
    with pytest.raises(gpb.GrowPageError, match="static scratch limit|bad read-ceiling"):
        eng.pool.kv_read_ceiling_static(0, 1, 0, torch.zeros(1025, dtype=torch.int32, device="cuda"),
                                        torch.zeros(4, dtype=torch.int32, device="cuda"))
