"""CUDA path vs the oracle on the larger workloads.

* Continuous batching with shared, refcounted prefixes (the 36-layer
  Qwen3-shaped workload's features at reduced size): requests join and leave
  mid-run, slots are reused, prefixes are released; every request and every
  block table is compared.
* The three large workloads at their full sizes and in the launch
  configuration bench.py times (32-layer stack with a 40 GB pool and 64
  requests; 36-layer stack with shared 2048-token prefixes and 128 request
  slots; 256 requests all at a boundary in the same step with a 120 GB pool):
  two sampled requests are simulated by the oracle and compared step by step.
"""
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


def _cb_workload(synth):
    # Qwen3-8B-shaped heads (32q/8kv, d=128, bf16, RoPE 1e6), 2 layers,
    # 64-token prefixes shared by groups of 4, prompt = the prefix only,
    # 2-page initial budget, short lognormal outputs.
    return synth.WORKLOADS["qwen3_8b_36layer_cb"].replace(
        num_layers=2, prefix_len=64, prefix_group=4, budget_pages=2, out_median=120,
        out_min=70, out_max=220, max_pages_per_req=64, top_p=0.9)


@pytest.mark.parametrize("full_kv", [False, True])
def test_continuous_batching_with_shared_prefixes(env, full_kv):
    H, gp, synth = env
    w = _cb_workload(synth)
    mode = gp.GP_MODE_FULL_KV if full_kv else gp.GP_MODE_GROWPAGE
    sc = H.Scenario(w, max_requests=8, num_pages=400, mode=mode, max_prefixes=16,
                    max_seq_len=64 + 256 + 16)
    remaining = {}
    next_rid = 0
    users = {}

    def admit(slot, prefix):
        nonlocal next_rid
        remaining[slot] = sc.admit(slot, next_rid, prefix=prefix)
        users[prefix] = users.get(prefix, 0) + 1
        next_rid += 1

    sc.add_prefix(0)
    for s in range(4):
        admit(s, 0)
    sc.release_prefix(0)            # the creator lets go; requests keep it alive
    prefix_of = {s: 0 for s in range(4)}
    next_prefix = 1
    for t in range(260):
        if t == 30:                 # a second group arrives
            sc.add_prefix(next_prefix)
            for s in range(4, 8):
                admit(s, next_prefix)
                prefix_of[s] = next_prefix
            sc.release_prefix(next_prefix)
            next_prefix += 1
        sc.step()
        if sc.rep.failures:
            break
        for s in list(remaining):
            remaining[s] -= 1
            if remaining[s] == 0:   # leaves; its slot is reused by a new group
                sc.free(s)
                del remaining[s]
                users[prefix_of[s]] -= 1
                if t < 200:
                    if next_prefix not in sc.gpid:
                        sc.add_prefix(next_prefix)
                    admit(s, next_prefix)
                    prefix_of[s] = next_prefix
                    if users[next_prefix] == 2:
                        sc.release_prefix(next_prefix)
                        next_prefix += 1
        sc.ora.check_invariants()
    _check(sc.rep)
    assert sc.rep.boundaries > 20
    if full_kv:
        assert sc.rep.compacts == 0
    else:
        assert sc.rep.compacts > 0


def _run_sampled(sc, steps):
    try:
        for _ in range(steps):
            sc.step()
            if sc.rep.failures:
                break
        _check(sc.rep)
    finally:
        torch.cuda.synchronize()


def test_llama8b_32layer_full_size_sampled(env):
    # 32 layers, batch 64, 40 GB pool (19073 pages), the bench's launch shape.
    H, gp, synth = env
    w = synth.WORKLOADS["llama8b_32layer"]
    sc = H.Scenario(w, max_requests=w.batch, num_pages=w.num_pages, compare_all=False,
                    gen_device="cuda", oracle_pages=256)
    lens = synth.draw_lengths(w, w.batch)
    # the two requests with the longest prompts reach their first boundary soonest
    sampled = sorted(range(w.batch), key=lambda r: -lens[r][0])[:2]
    for rid in range(w.batch):
        sc.admit(rid, rid, compare=rid in sampled)
    need = 1024 - max(lens[r][0] for r in sampled)
    _run_sampled(sc, min(need + 70, 200))
    assert sc.rep.boundaries >= 3
    del sc
    torch.cuda.empty_cache()


def test_qwen3_36layer_full_size_sampled(env):
    # 36 layers, 128 request slots, 40 GB pool (16954 pages), 2048-token
    # prefixes shared by groups of 8; initial budget cut to 4 pages so that
    # the sampled requests reach boundaries within the window.
    H, gp, synth = env
    w = synth.WORKLOADS["qwen3_8b_36layer_cb"].replace(budget_pages=4)
    sc = H.Scenario(w, max_requests=w.batch, num_pages=w.num_pages, compare_all=False,
                    gen_device="cuda", oracle_pages=512, max_prefixes=8)
    sc.add_prefix(0, compare=True)
    sc.add_prefix(1, compare=False)
    for rid in range(16):
        sc.admit(rid, rid, compare=rid in (0, 5), prefix=rid // 8)
    _run_sampled(sc, 100)
    assert sc.rep.boundaries >= 4
    del sc
    torch.cuda.empty_cache()


def test_stress_burst_full_size_sampled(env):
    # 256 requests, prompts of exactly the initial budget: all at a boundary
    # on the first step and every 16th after it; 120 GB pool (57220 pages).
    H, gp, synth = env
    w = synth.WORKLOADS["stress_burst"]
    sc = H.Scenario(w, max_requests=w.batch, num_pages=w.num_pages, compare_all=False,
                    gen_device="cuda", oracle_pages=256)
    for rid in range(w.batch):
        sc.admit(rid, rid, compare=rid in (3, 200))
    _run_sampled(sc, 34)
    assert sc.rep.boundaries == 2 * 3
    st = sc.pool.stats()
    assert st.boundaries == 256 * 3
    del sc
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode_name", ["GROWPAGE", "FULL_KV"])
def test_graph_replay_equals_eager_steps(env, mode_name):
    # Steps replayed as one captured CUDA graph each end bit-identical to the
    # same steps launched call by call: outputs, request metadata, block
    # tables, token positions, summaries (one Llama-3-8B-shaped layer, 16
    # requests, boundaries, grows, compactions and refills on the way).
    import numpy as np
    from demand_paged_kv_gqa_b300.engine import Engine
    H, gp, synth = env
    mode = getattr(gp, "GP_MODE_" + mode_name)
    w = synth.WORKLOADS["llama8b_1layer"].replace(decode_steps=300, num_pages=2048)
    runs = []
    for graph in (False, True):
        eng = Engine(w, mode=mode, use_graph=graph)
        eng.fill()
        for _ in range(400):
            eng.prepare_inputs()
            eng.step()
        eng.pool.sync()
        runs.append(eng)
    a, b = runs
    assert b.graph_launches > 0 and b.finished == a.finished > 0
    assert torch.equal(a.out, b.out)
    sa, sb = a.pool.state(tok_pos=True), b.pool.state(tok_pos=True)
    assert [bytes(m) for m in sa["req"]] == [bytes(m) for m in sb["req"]]
    for key in ("block", "free_stack", "tok_pos"):
        assert np.array_equal(sa[key], sb[key]), key
    assert torch.equal(a.pool.region("summary"), b.pool.region("summary"))
    assert sa["ctrl"].boundaries == sb["ctrl"].boundaries > 0


def test_llama8b_32layer_every_request_matches_dense_attention(env):
    # Full size, the bench's launch shape (64 requests, 32 layers, 40 GB pool,
    # the weighted worker split cutting almost every (request, head) between
    # workers): at one step, every request's output in two layers is checked
    # against dense softmax attention in fp64 over the resident tokens the pool
    # held at the start of the step plus the step's own token (rotated with the
    # oracle's RoPE, rounded once to bf16).  This covers the requests the
    # sampled comparison does not simulate.
    import numpy as np
    from demand_paged_kv_gqa_b300.engine import Engine
    from oracle import numerics as nm
    H, gp, synth = env
    w = synth.WORKLOADS["llama8b_32layer"]
    eng = Engine(w)
    eng.fill()
    for _ in range(300):
        eng.prepare_inputs()
        eng.step()
    eng.prepare_inputs()
    act = eng.active()
    assert len(act) == w.batch
    st = eng.pool.state()
    layers = (5, 31)
    P, hk, hq, d, G = w.page_size, w.num_kv_heads, w.num_q_heads, w.head_dim, w.group
    kv = eng.pool.region("kv")
    metas = {s: st["req"][s] for s in act}
    pages = sorted({int(p) for s in act
                    for p in st["block"][s, : metas[s].n_pre_pages + metas[s].n_pages]})
    pidx = torch.tensor(pages, dtype=torch.long, device="cuda")
    where = {p: k for k, p in enumerate(pages)}
    snap = np.stack([kv[:, l].index_select(0, pidx).float().cpu().numpy() for l in layers],
                    axis=1)                                 # [pg][2][Hk][2][P][d]
    q = eng.q[list(layers)].float().cpu().numpy()          # [2][n][Hq][d]
    kn = eng.k[list(layers)].float().cpu().numpy()
    vn = eng.v[list(layers)].float().cpu().numpy()
    eng.step()
    eng.pool.sync()
    out = eng.out[list(layers)].float().cpu().numpy()
    rope = nm.RopeTable(w.rope_theta, d)
    worst = 0.0
    for i, s in enumerate(act):
        m = metas[s]
        R = m.n_pre_pages * P + m.seq_priv
        bt = st["block"][s]
        rows = [(where[int(bt[j // P])], j % P) for j in range(R)]
        pi = np.array([r[0] for r in rows])
        si = np.array([r[1] for r in rows])
        for li in range(len(layers)):
            K = snap[pi, li, :, 0, si].astype(np.float64)  # [R][Hk][d]
            V = snap[pi, li, :, 1, si].astype(np.float64)
            kt = nm.round_bf16(nm.rope_apply(kn[li, i].astype(np.float64), rope, m.pos))
            vt = vn[li, i].astype(np.float64)
            qr = nm.rope_apply(q[li, i].astype(np.float64), rope, m.pos).reshape(hk, G, d)
            sc = np.einsum("gqd,rgd->gqr", qr, K) / np.sqrt(d)
            st_ = np.einsum("gqd,gd->gq", qr, kt)[:, :, None] / np.sqrt(d)
            allsc = np.concatenate([sc, st_], axis=2)
            pr = np.exp(allsc - allsc.max(axis=2, keepdims=True))
            pr /= pr.sum(axis=2, keepdims=True)
            ref = np.einsum("gqr,rgd->gqd", pr[:, :, :-1], V) + pr[:, :, -1:] * vt[:, None, :]
            ref = ref.reshape(hq, d)
            err = np.max(np.abs(out[li, i] - ref)) / np.max(np.abs(ref))
            worst = max(worst, float(err))
    assert worst < 2e-2, worst
    del eng
    torch.cuda.empty_cache()
