"""CUDA path vs the CPU oracle, step by step, on the seeded workloads.

Marked ``gpu``: these call the C-ABI library on a B300.  Sizes are the
workloads' own where the oracle finishes in seconds to a minute; longer
trajectories are cut to a window that still spans many boundaries.
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


def test_tiny_growpage_full_trajectory(env):
    # 1 request, 1 layer, 2 kv heads x 2 q heads, d=64, fp32, page 16,
    # prompt 64 = initial budget: boundaries at step 1 and every 16 steps.
    H, gp, synth = env
    h = H.Harness(synth.WORKLOADS["tiny"], 1)
    rep = h.run(256)
    _check(rep)
    assert rep.boundaries == 16
    assert rep.max_out_err < 1e-4


def test_tiny_full_kv(env):
    H, gp, synth = env
    h = H.Harness(synth.WORKLOADS["tiny"], 1, mode=gp.GP_MODE_FULL_KV)
    rep = h.run(256)
    _check(rep)
    assert rep.compacts == 0 and rep.grows == rep.boundaries == 16


@pytest.mark.parametrize("G", [1, 4])
def test_tiny_variants_gqa_group_and_rope(env, G):
    # G=1 is plain multi-head attention; RoPE on with theta 10000.
    H, gp, synth = env
    w = synth.WORKLOADS["tiny"].replace(num_q_heads=2 * G, rope_theta=10000.0, batch=3)
    h = H.Harness(w, 3)
    rep = h.run(120)
    _check(rep)
    assert rep.boundaries >= 3 * 7


def test_tiny_fp32_d128_several_requests(env):
    H, gp, synth = env
    w = synth.WORKLOADS["tiny"].replace(head_dim=128, num_q_heads=8, num_kv_heads=2,
                                        rope_theta=500000.0, batch=4, prompt_min=20,
                                        prompt_max=64, num_pages=64, num_layers=2)
    h = H.Harness(w, 4)
    rep = h.run(150)
    _check(rep)
    assert rep.boundaries > 10


def test_llama8b_1layer_window(env):
    # One Llama-3-8B-shaped layer (32q / 8kv, d=128, bf16, RoPE 5e5), the 16
    # requests of the workload, first 640 decode steps (dozens of boundaries).
    H, gp, synth = env
    h = H.Harness(synth.WORKLOADS["llama8b_1layer"], 16)
    rep = h.run(640)
    _check(rep)
    assert rep.boundaries > 50
    assert rep.max_out_err < 2e-2


def test_llama8b_1layer_small_budget_compacts(env):
    # Same layer with a budget of 8 pages and Top-p 0.99: many compactions.
    H, gp, synth = env
    w = synth.WORKLOADS["llama8b_1layer"].replace(prompt_min=100, prompt_max=128, top_p=0.99,
                                                  budget_pages=8, max_pages_per_req=12)
    h = H.Harness(w, 6, budget_pages=8)
    rep = h.run(300)
    _check(rep)
    assert rep.compacts > 20


def test_llama8b_1layer_full_kv(env):
    H, gp, synth = env
    w = synth.WORKLOADS["llama8b_1layer"].replace(prompt_min=900, prompt_max=1024)
    h = H.Harness(w, 8, mode=gp.GP_MODE_FULL_KV)
    rep = h.run(200)
    _check(rep)
    assert rep.grows > 8 and rep.compacts == 0


def test_pool_exhaustion_compacts_instead(env):
    # tau < 0: every boundary wants to grow; 6 pages in the pool, 4 taken by
    # the prompt: the first two boundaries grow, the rest compact (denied).
    H, gp, synth = env
    w = synth.WORKLOADS["tiny"].replace(tau=-1.0, num_pages=6)
    h = H.Harness(w, 1)
    rep = h.run(100)
    _check(rep)
    assert rep.grows == 2 and rep.compacts >= 4


@pytest.mark.parametrize("mode_name,rate", [("FIXED", 0.0), ("INVERSE", 0.0), ("RANDOM", 0.3)])
def test_ablation_policies(env, mode_name, rate):
    # the review's ablation policies on the same kernels: fixed budget,
    # inverted signal, frequency-matched random decisions
    H, gp, synth = env
    mode = getattr(gp, "GP_MODE_" + mode_name)
    w = synth.WORKLOADS["llama8b_1layer"].replace(prompt_min=100, prompt_max=128, budget_pages=8,
                                                  max_pages_per_req=20)
    h = H.Harness(w, 6, mode=mode, budget_pages=8, random_grow_rate=rate)
    rep = h.run(260)
    _check(rep)
    assert rep.boundaries > 30
    if mode_name == "FIXED":
        assert rep.grows == 0
    else:
        assert rep.grows > 0 and rep.compacts > 0
    t = H.Harness(synth.WORKLOADS["tiny"], 1, mode=mode, random_grow_rate=rate)
    _check(t.run(200))


def test_review_hyperparameters_page_256(env):
    # the authors' settings: KV block 256 tokens, Top-p 0.99, retention 64
    H, gp, synth = env
    w = synth.WORKLOADS["llama8b_1layer"].replace(page_size=256, top_p=0.99, recent_window=64,
                                                  prompt_min=480, prompt_max=512, budget_pages=2,
                                                  num_pages=64, max_pages_per_req=8)
    h = H.Harness(w, 6, budget_pages=2)
    rep = h.run(300)
    _check(rep)
    assert rep.boundaries >= 12


def test_page_size_not_a_power_of_two(env):
    # 48-token pages: three 16-token blocks per page, block-table and
    # in-page offsets by division rather than shifts, in the attention
    # kernel, its block copies and the compaction moves
    H, gp, synth = env
    w = synth.WORKLOADS["llama8b_1layer"].replace(page_size=48, prompt_min=280, prompt_max=288,
                                                  budget_pages=6, num_pages=200, max_pages_per_req=24)
    h = H.Harness(w, 5, budget_pages=6)
    rep = h.run(160)
    _check(rep)
    assert rep.boundaries >= 10
    assert rep.compacts > 0


def test_shrink_policy(env):
    # the SHRINK ablation: boundaries that do not grow release a page while
    # the kept set still holds the recent window, else compact in place;
    # grows and releases of several requests in the same step exercise the
    # allocator order (block tables are compared exactly)
    H, gp, synth = env
    w = synth.WORKLOADS["llama8b_1layer"].replace(prompt_min=180, prompt_max=192, budget_pages=12,
                                                  max_pages_per_req=20)
    h = H.Harness(w, 6, mode=gp.GP_MODE_SHRINK, budget_pages=12)
    rep = h.run(260)
    _check(rep)
    assert rep.shrinks > 6 and rep.boundaries > 30
    st = h.pool.stats()
    assert st.shrinks == rep.shrinks
    t = H.Harness(synth.WORKLOADS["tiny"], 1, mode=gp.GP_MODE_SHRINK)
    rt = t.run(200)
    _check(rt)
    assert rt.shrinks >= 1


def test_signal_quality_traces_match_oracle(env):
    # the Delta / demand traces the signal-quality analysis reads from the
    # device equal the oracle's, and so do the statistics drawn from them
    H, gp, synth = env
    from demand_paged_kv_gqa_b300 import signal_quality as sq
    w = synth.WORKLOADS["llama8b_1layer"].replace(prompt_min=100, prompt_max=128, budget_pages=8,
                                                  max_pages_per_req=24)
    h = H.Harness(w, 6, budget_pages=8)
    req, wset = h.pool.region("req"), h.pool.region("wset")
    gpu_tr, ora_tr = {}, {}
    for _ in range(300):
        res = h.step()
        _check(h.rep)
        meta = req[: h.n].cpu()
        ws = wset[: h.n].sum(dim=(1, 2)).cpu()
        for s, rec in res["records"].items():
            delta = (int(meta[s, 9]) << 32) | (int(meta[s, 8]) & 0xFFFFFFFF)
            gpu_tr.setdefault(s, []).append((delta, int(ws[s, 0])))
            ora_tr.setdefault(s, []).append((int(rec.delta), int(rec.w_short.sum())))
    g, o = sq.statistics(gpu_tr), sq.statistics(ora_tr)
    assert g["pairs"] == o["pairs"] > 30
    if h.rep.w_in_band == 0:
        assert gpu_tr == ora_tr
    assert abs(g["spearman_rho"] - o["spearman_rho"]) < 0.05


@pytest.mark.parametrize("over", [dict(top_p=1.0), dict(top_p=0.05), dict(recent_window=0),
                                  dict(recent_window=10000)],
                         ids=["top_p_1", "top_p_0.05", "window_0", "window_covers_all"])
def test_degenerate_settings(env, over):
    # Top-p at the whole mass and at a sliver of it; no recent window; a
    # window wider than the kept set (the C - P most recent tokens are kept)
    H, gp, synth = env
    h = H.Harness(synth.WORKLOADS["tiny"].replace(**over), 1)
    rep = h.run(200)
    _check(rep)
    assert rep.boundaries >= 12
    w = synth.WORKLOADS["llama8b_1layer"].replace(prompt_min=100, prompt_max=128, budget_pages=8,
                                                  max_pages_per_req=16, **over)
    hb = H.Harness(w, 4, budget_pages=8)
    rb = hb.run(120)
    _check(rb)
    assert rb.boundaries >= 8


def test_empty_steps_and_call_order(env):
    # a step with no requests changes nothing; calls out of order are
    # refused with GP_ERR_INVALID and leave the pool usable
    H, gp, synth = env
    h = H.Harness(synth.WORKLOADS["tiny"], 1)
    rep = h.run(20)
    _check(rep)
    w = h.w
    none = torch.zeros(0, dtype=torch.int32, device="cuda")
    qe = torch.zeros(0, w.num_q_heads, w.head_dim, dtype=w.torch_dtype, device="cuda")
    ke = torch.zeros(0, w.num_kv_heads, w.head_dim, dtype=w.torch_dtype, device="cuda")
    for _ in range(3):
        for l in range(w.num_layers):
            h.pool.decode_step(l, none, qe, ke, ke, qe)
        h.pool.boundary(none)
    with pytest.raises(gp.GrowPageError) as e:
        h.pool.boundary(h.slots_dev)        # gp_boundary before the step's layers
    assert e.value.code == gp.GP_ERR_INVALID
    with pytest.raises(gp.GrowPageError):
        h.pool.free(5)                      # not an active slot
    h.pool.sync()
    rep = h.run(60)                         # the trajectory continues in step with the oracle
    _check(rep)
    assert rep.boundaries >= 4


def test_get_state_matches_per_request_reads(env):
    # one call copies the whole state; it agrees with the per-request and
    # counter reads, and with the oracle's block tables and kept positions
    H, gp, synth = env
    w = synth.WORKLOADS["llama8b_1layer"].replace(prompt_min=100, prompt_max=128, budget_pages=8,
                                                  max_pages_per_req=16)
    h = H.Harness(w, 4, budget_pages=8)
    _check(h.run(60))
    st = h.pool.state(tok_pos=True)
    c = h.pool.stats()
    assert st["ctrl"].boundaries == c.boundaries and st["ctrl"].free_top == c.free_top
    assert len(st["free_stack"]) == c.free_top
    for s in h.slots:
        m, bt = h.pool.request(s)
        assert bytes(st["req"][s]) == bytes(m)
        assert st["block"][s, : len(bt)].tolist() == bt == h.ora.block_table(s)
        pos = H._private_positions(st["tok_pos"], bt[m.n_pre_pages:], m.seq_priv, w.num_layers,
                                   w.num_kv_heads, w.page_size)
        assert np.array_equal(np.sort(pos, axis=-1), h.ora.kept_positions(s))
    owned = {p for s in h.slots for p in h.pool.request(s)[1]}
    assert not owned & set(st["free_stack"].tolist())
    assert len(owned) + c.free_top == h.cfg.num_pages


def test_select_rows_beyond_shared_memory(env):
    # Rows longer than the select kernel stages in shared memory (4096
    # tokens): the working-set counts and the compaction keys read the scores
    # and token positions from global memory.  One Llama-3-8B-shaped layer,
    # 4 requests whose 4480-token prompts fill their 280-page budgets, so the
    # first boundary is on step 1 and then every 16 steps.
    H, gp, synth = env
    w = synth.WORKLOADS["llama8b_1layer"].replace(prompt_min=4480, prompt_max=4480,
                                                  budget_pages=280, max_pages_per_req=320,
                                                  num_pages=1400)
    h = H.Harness(w, 4, budget_pages=280, max_seq_len=4480 + 200)
    rep = h.run(130)
    _check(rep)
    assert rep.boundaries == 4 * 9
    assert rep.grows > 0 and rep.compacts > 0
    assert rep.max_out_err < 2e-2


def test_select_rows_staged_without_first_pass_bins(env):
    # Rows of 2049 .. 4096 tokens are staged in shared memory but leave no
    # room for the first Top-p pass's per-warp bins: that pass takes the
    # digit-group adds.  Two Llama-3-8B-shaped layers, 3 requests whose
    # 3072-token prompts fill their 192-page budgets.
    H, gp, synth = env
    w = synth.WORKLOADS["llama8b_1layer"].replace(num_layers=2, prompt_min=3072, prompt_max=3072,
                                                  budget_pages=192, max_pages_per_req=240,
                                                  num_pages=900)
    h = H.Harness(w, 3, budget_pages=192, max_seq_len=3072 + 120)
    rep = h.run(70)
    _check(rep)
    assert rep.boundaries == 3 * 5
    assert rep.compacts > 0


def test_select_rows_beyond_shared_memory_with_prefix(env):
    # The 36-layer Qwen3-shaped workload's request shape on one layer: a
    # 2048-token shared prefix plus 2304 private tokens (R = 4352 > 4096,
    # C = 2304), three requests sharing the prefix.
    H, gp, synth = env
    w = synth.WORKLOADS["qwen3_8b_36layer_cb"].replace(
        num_layers=1, prompt_min=2304, prompt_max=2304, budget_pages=144, max_pages_per_req=200)
    sc = H.Scenario(w, max_requests=3, num_pages=1200, max_prefixes=2,
                    max_seq_len=2048 + 2304 + 200)
    sc.add_prefix(0)
    for s in range(3):
        sc.admit(s, s, prefix=0, budget_pages=144)
    sc.release_prefix(0)
    for _ in range(110):
        sc.step()
        if sc.rep.failures:
            break
        sc.ora.check_invariants()
    _check(sc.rep)
    assert sc.rep.boundaries == 3 * 7
    assert sc.rep.compacts > 0


@pytest.mark.parametrize("shape", ["tiny", "llama8b_1layer"])
def test_full_kv_stops_at_the_page_cap(env, shape):
    # Full KV with a cap on a request's private pages: once a request holds
    # max_pages_per_req pages its boundaries cannot grow, and drop the step's
    # token (starved), as a boundary with no free page does.  Starvation is
    # counted, not raised: the pool's status word stays clear.
    H, gp, synth = env
    if shape == "tiny":
        w = synth.WORKLOADS["tiny"].replace(max_pages_per_req=6)
        n, budget, steps = 1, None, 120
    else:
        w = synth.WORKLOADS["llama8b_1layer"].replace(prompt_min=100, prompt_max=128,
                                                      budget_pages=8, max_pages_per_req=10)
        n, budget, steps = 4, 8, 120
    h = H.Harness(w, n, mode=gp.GP_MODE_FULL_KV, budget_pages=budget)
    rep = h.run(steps)
    _check(rep)
    st = h.pool.stats()
    assert st.starved > 0 and st.status == 0
    assert st.starved + st.grows == st.boundaries == rep.boundaries
    for s in h.slots:
        m, _ = h.pool.request(s)
        assert m.n_pages == w.max_pages_per_req and m.n_starved > 0


@pytest.mark.parametrize("mode_name", ["GROWPAGE", "FULL_KV"])
def test_async_boundary_work(env, mode_name):
    # gp_boundary_async: the requests at a boundary get their boundary work
    # on a second stream and sit out the next step.  Checked step by step
    # against the oracle (which simply leaves them out of that step); then a
    # twin pool replays the same steps with no host sync between them, so the
    # second stream really runs beside the next step, and must end
    # bit-identical: every output of every step, block tables, token
    # positions, the free stack and the summaries.
    H, gp, synth = env
    mode = getattr(gp, "GP_MODE_" + mode_name)
    w = synth.WORKLOADS["llama8b_1layer"].replace(num_layers=2, prompt_min=60, prompt_max=128,
                                                  budget_pages=8, max_pages_per_req=16)
    side = torch.cuda.Stream()
    sc = H.Scenario(w, max_requests=6, num_pages=200, mode=mode, side=side, record=True)
    for s in range(6):
        sc.admit(s, s, budget_pages=8)
    out_of_step = set()
    for _ in range(150):
        bnd = sc.step(exclude=out_of_step)
        if sc.rep.failures:
            break
        out_of_step = bnd
        sc.ora.check_invariants()
    _check(sc.rep)
    assert sc.rep.boundaries > 30
    twin = gp.Pool(sc.cfg)
    for s in range(6):
        pl, T = synth.draw_lengths(w, 1, s)[0]
        k, v = synth.RequestStream(w, s, T).prompt(pl)
        twin.add_request(s, k.cuda().contiguous(), v.cuda().contiguous(), 8)
    side2 = torch.cuda.Stream()
    outs = []
    for slots, q, k, v, _ in sc.trace:
        sd = torch.tensor(slots, dtype=torch.int32, device="cuda")
        step_out = []
        for l in range(w.num_layers):
            if not slots:
                twin.decode_step(l, sd, None, None, None, None)
                continue
            o = torch.empty(len(slots), w.num_q_heads, w.head_dim, dtype=w.torch_dtype, device="cuda")
            twin.decode_step(l, sd, q[:, l].contiguous(), k[:, l].contiguous(),
                             v[:, l].contiguous(), o)
            step_out.append(o)
        twin.boundary_async(sd, side2)
        outs.append(step_out)
    twin.sync()
    for (_, _, _, _, ref), got in zip(sc.trace, outs):
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    a, b = sc.pool.state(tok_pos=True), twin.state(tok_pos=True)
    assert [bytes(m) for m in a["req"]] == [bytes(m) for m in b["req"]]
    for key in ("block", "free_stack", "tok_pos"):
        assert np.array_equal(a[key], b[key]), key
    assert torch.equal(sc.pool.region("summary"), twin.region("summary"))


@pytest.mark.parametrize("mode_name", ["GROWPAGE", "SHRINK"])
def test_twelve_layers(env, mode_name):
    # a deeper stack than the other full comparisons: 12 layers, 4 requests,
    # every step, request, layer and head against the oracle
    H, gp, synth = env
    mode = getattr(gp, "GP_MODE_" + mode_name)
    w = synth.WORKLOADS["llama8b_1layer"].replace(num_layers=12, prompt_min=100, prompt_max=128,
                                                  budget_pages=8, max_pages_per_req=16)
    h = H.Harness(w, 4, mode=mode, budget_pages=8)
    rep = h.run(80)
    _check(rep)
    assert rep.boundaries >= 12


def test_key_rotation_bits_equal_fp64_definition(env):
    # The staged key of a step and the stored prompt keys are rotated to
    # their positions and rounded once to bf16, bit for bit as the fp64
    # expression of the oracle gives them.  The kernels evaluate it in fp32
    # with a certified error bound and fall back to fp64 where the bound
    # cannot decide the rounding: the inputs mix ordinary keys, pairs with
    # heavy cancellation (x·c close to y·s), tiny, huge and zero keys (the
    # fallback), at positions up to 60k.
    H, gp, synth = env
    from oracle import numerics as nm
    L, hq, hk, d, P = 1, 32, 8, 128, 16
    theta = 500000.0
    cfg = gp.make_config(num_layers=L, num_q_heads=hq, num_kv_heads=hk, head_dim=d, page_size=P,
                         num_pages=8192, max_requests=16, max_pages_per_req=4096,
                         dtype=torch.bfloat16, max_seq_len=65536, rope_theta=theta,
                         top_p=0.9, recent_window=64)
    pool = gp.Pool(cfg)
    rng = np.random.default_rng(20261203)
    table = nm.RopeTable(theta, d)
    prompt_lens = [1, 2, 17, 100, 333, 1000, 4097, 9000, 30000, 60000, 5, 64]
    n = len(prompt_lens)
    dev = torch.device("cuda")

    def bf16(x):
        return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)

    prompts = []
    for s, pl in enumerate(prompt_lens):
        k = bf16(rng.standard_normal((L, pl, hk, d)) * 2.0)
        v = bf16(rng.standard_normal((L, pl, hk, d)))
        pool.add_request(s, k.to(dev), v.to(dev), budget_pages=(pl + P - 1) // P + 1)
        prompts.append(k)
    pos = [pool.request(s)[0].pos for s in range(n)]
    h2 = d // 2
    knew = rng.standard_normal((n, hk, d)).astype(np.float64)
    knew[1] *= 1e-25                     # tiny: the fp64 fallback
    knew[2] *= 1e25                      # huge
    knew[3, :4] = 0.0                    # zero rows, signed zeros
    knew[3, 4:6] = -0.0
    knew[3, 6, ::2] = -0.0
    knew[4, :, ::3] *= 1e-30             # mixed inside a row
    for s in (5, 6, 7, 8, 9):            # x·c - y·s much smaller than |x| + |y|
        c, sn = table(pos[s])
        x = nm.round_bf16(knew[s, :, :h2])
        ok = np.abs(sn) > 1e-3
        y = nm.round_bf16(x * c / np.where(ok, sn, 1.0))
        knew[s, :, :h2] = x
        knew[s, :, h2:] = np.where(ok, y, knew[s, :, h2:])
    kd = bf16(knew).to(dev)
    q = bf16(rng.standard_normal((n, hq, d))).to(dev)
    v = bf16(rng.standard_normal((n, hk, d))).to(dev)
    out = torch.empty(n, hq, d, dtype=torch.bfloat16, device=dev)
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    pool.decode_step(0, slots, q, kd, v, out)
    pool.sync()
    got = pool.region("staging")[:n, 0, :, 0].float().cpu().double().numpy()
    kin = kd.float().cpu().double().numpy()
    for s in range(n):
        want = nm.round_bf16(nm.rope_apply(kin[s], table, pos[s]))
        bad = np.argwhere(got[s] != want)
        assert bad.size == 0, f"slot {s} position {pos[s]}: staged key differs at {bad[:4].tolist()}"
    # the prompt keys in the pages (admission), token t at position t
    kv = pool.region("kv")
    for s, pl in enumerate(prompt_lens):
        m, bt = pool.request(s)
        pages = torch.as_tensor(bt[m.n_pre_pages: m.n_pre_pages + (pl + P - 1) // P], dtype=torch.long)
        rows = kv.index_select(0, pages.to(dev))[:, 0, :, 0].float().cpu().double().numpy()
        stored = rows.transpose(0, 2, 1, 3).reshape(-1, hk, d)[:pl]         # [token][head][d]
        kp = prompts[s][0].float().double().numpy()
        for t in sorted({0, min(1, pl - 1), pl // 2, pl - 1}):
            want = nm.round_bf16(nm.rope_apply(kp[t], table, t))
            assert np.array_equal(stored[t], want), f"slot {s}: prompt key {t} differs"
