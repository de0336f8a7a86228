"""Refused calls and flagged steps, injected from the host.

Nothing here faults, traps or hangs the GPU: an exhausted pool is refused by
the host before anything is enqueued, and a bad slot list or a position past
max_seq_len is caught by the plan kernel, which flags the device status word
and drops the whole step before any state changes.  After each refusal the
pool's state is read back and must equal what it was before, and the pool
must go on (after gp_clear_status) as if the refused call had not been made.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests import gpu_harness
    from demand_paged_kv_gqa_b300 import growpage, synth
    return gpu_harness, growpage, synth


def _check(rep):
    assert not rep.failures, "\n".join(rep.failures)


def _snapshot(pool):
    """Everything a step or an admission may change, copied to the host."""
    st = pool.state(tok_pos=True)
    c = st["ctrl"]
    return dict(req=[bytes(m) for m in st["req"]], block=st["block"].copy(),
                free=st["free_stack"].copy(), tok_pos=st["tok_pos"].copy(),
                ctrl=(c.free_top, c.status, c.steps, c.boundaries, c.grows, c.compacts),
                summary=pool.region("summary").cpu().numpy().copy(),
                staging=pool.region("staging").float().cpu().numpy().copy(),
                kv=pool.region("kv").float().cpu().numpy().copy())


def _same(a, b):
    for k in a:
        if isinstance(a[k], np.ndarray):
            assert np.array_equal(a[k], b[k]), k
        else:
            assert a[k] == b[k], k


def _tensors(w, n, length, seed=0):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(w.num_layers, length, w.num_kv_heads, w.head_dim, generator=g)
    v = torch.randn(w.num_layers, length, w.num_kv_heads, w.head_dim, generator=g)
    return k.to(w.torch_dtype).cuda(), v.to(w.torch_dtype).cuda()


def test_admission_without_pages_is_refused(env):
    H, gp, synth = env
    w = synth.WORKLOADS["tiny"].replace(prefix_len=64)
    cfg = gp.config_for(w, max_requests=4, num_pages=6, max_prefixes=2)
    pool = gp.Pool(cfg)
    k, v = _tensors(w, 1, 64)
    pool.add_request(0, k, v, 4)
    before = _snapshot(pool)
    with pytest.raises(gp.GrowPageError) as e:
        pool.add_request(1, k[:, :32].contiguous(), v[:, :32].contiguous(), 4)
    assert e.value.code == gp.GP_ERR_NO_PAGES
    with pytest.raises(gp.GrowPageError) as e:
        pool.add_prefix(k[:, :48].contiguous(), v[:, :48].contiguous())
    assert e.value.code == gp.GP_ERR_NO_PAGES
    pool.sync()
    _same(before, _snapshot(pool))
    # the two pages left are still there for a request that fits
    pool.add_request(1, k[:, :32].contiguous(), v[:, :32].contiguous(), 2)
    assert pool.stats().free_top == 0
    m, bt = pool.request(1)
    assert m.active == 1 and bt == [4, 5]


def test_bad_slot_lists_drop_the_step(env):
    # descending, repeated and out-of-range slot lists: the step is dropped
    # on the device, gp_sync reports "bad-slot-list", the state is unchanged,
    # and after gp_clear_status the trajectory goes on in step with the oracle
    H, gp, synth = env
    w = synth.WORKLOADS["tiny"].replace(batch=2, prompt_min=40, prompt_max=60)
    h = H.Harness(w, 2)
    _check(h.run(20))
    before = _snapshot(h.pool)
    q = torch.zeros(2, w.num_q_heads, w.head_dim, device="cuda")
    kv = torch.zeros(2, w.num_kv_heads, w.head_dim, device="cuda")
    out = torch.zeros_like(q)
    for bad in ([1, 0], [0, 0], [0, 7]):
        slots = torch.tensor(bad, dtype=torch.int32, device="cuda")
        for l in range(w.num_layers):
            h.pool.decode_step(l, slots, q, kv, kv, out)
        h.pool.boundary(slots)
        with pytest.raises(gp.GrowPageError, match="bad-slot-list") as e:
            h.pool.sync()
        assert e.value.code == gp.GP_ERR_DEVICE
        st, info = h.pool.clear_status()
        assert st & 0x1
        h.pool.sync()
        _same(before, _snapshot(h.pool))
    rep = h.run(60)
    _check(rep)
    assert rep.boundaries >= 6


def test_inactive_slot_and_position_range(env):
    # an inactive slot in the list, then a request that reaches max_seq_len:
    # both drop their step with the matching status bits
    H, gp, synth = env
    w = synth.WORKLOADS["tiny"]
    cfg = gp.config_for(w, max_requests=4, num_pages=32, max_seq_len=70)
    pool = gp.Pool(cfg)
    k, v = _tensors(w, 1, 64)
    pool.add_request(0, k, v, 4)
    pool.add_request(2, k[:, :40].contiguous(), v[:, :40].contiguous(), 4)
    q = torch.randn(2, w.num_q_heads, w.head_dim, device="cuda")
    kv = torch.randn(2, w.num_kv_heads, w.head_dim, device="cuda")
    out = torch.zeros_like(q)

    def step(slot_list):
        slots = torch.tensor(slot_list, dtype=torch.int32, device="cuda")
        pool.decode_step(0, slots, q[: len(slot_list)], kv[: len(slot_list)],
                         kv[: len(slot_list)], out[: len(slot_list)])
        pool.boundary(slots)

    pool.sync()
    before = _snapshot(pool)
    step([0, 1])                     # slot 1 holds no request
    with pytest.raises(gp.GrowPageError, match="bad-slot-list"):
        pool.sync()
    st, info = pool.clear_status()
    assert st == 0x1 and info == 1
    _same(before, _snapshot(pool))
    for t in range(6):               # positions 64 .. 69: the last ones the table holds
        step([0, 2])
    pool.sync()
    assert pool.request(0)[0].pos == 70
    before = _snapshot(pool)
    step([0, 2])                     # slot 0 would need position 70
    with pytest.raises(gp.GrowPageError, match="position-beyond-max_seq_len"):
        pool.sync()
    st, info = pool.clear_status()
    assert st & 0x20 and st & 0x1
    _same(before, _snapshot(pool))
    step([2])                        # the other request still decodes
    pool.sync()
    assert pool.request(2)[0].pos == 47
