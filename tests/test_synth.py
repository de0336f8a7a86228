"""The seeded input generator (no GPU): determinism and the recipe."""
import math

import numpy as np
import torch

from demand_paged_kv_gqa_b300 import synth


def test_request_stream_is_deterministic_per_request():
    w = synth.WORKLOADS["tiny"]
    a, b, c = (synth.RequestStream(w, r, 64) for r in (3, 3, 4))
    for _ in range(5):
        qa, ka, va = a.next_step()
        qb, kb, vb = b.next_step()
        qc, _, _ = c.next_step()
        assert torch.equal(qa, qb) and torch.equal(ka, kb) and torch.equal(va, vb)
        assert not torch.equal(qa, qc)


def test_planted_keys_follow_the_walk():
    # at the planted steps floor(j T / 8) the new key is sqrt(d) times the
    # unit walk direction, which the queries of its group share
    w = synth.WORKLOADS["tiny"]
    T = 100
    st = synth.RequestStream(w, 0, T)
    planted = sorted({(j * T) // 8 for j in range(8)})
    assert planted == sorted(st.planted)
    d = w.head_dim
    for t in range(T):
        q, k, _ = st.next_step()
        if t in planted:
            assert torch.allclose(k.norm(dim=-1), torch.full(k.shape[:-1], math.sqrt(d)), rtol=1e-5)
            # the group's queries point the same way (their noise is smaller)
            qg = q.view(w.num_layers, w.num_kv_heads, w.group, d).mean(dim=2)
            cos = torch.nn.functional.cosine_similarity(qg, k, dim=-1)
            assert float(cos.min()) > 0.8


def test_batch_stream_plants_at_the_same_steps():
    w = synth.WORKLOADS["tiny"]
    Ts = [100, 37, 8, 256]
    bs = synth.BatchStream(w, len(Ts), Ts, device="cpu", seed=0)
    d = w.head_dim
    hot = {i: [] for i in range(len(Ts))}
    for t in range(260):
        q, k, _ = bs.next_step()
        u = bs.walk / bs.walk.norm(dim=-1, keepdim=True)
        for i in range(len(Ts)):
            if torch.allclose(k[i], math.sqrt(d) * u[i], atol=1e-5):
                hot[i].append(t)
    for i, T in enumerate(Ts):
        assert hot[i] == sorted({(j * T) // 8 for j in range(8)})


def test_lengths_within_the_workload_ranges():
    w = synth.WORKLOADS["llama8b_32layer"]
    lens = synth.draw_lengths(w, 200)
    assert lens == synth.draw_lengths(w, 200)
    pl = np.array([a for a, _ in lens])
    T = np.array([b for _, b in lens])
    assert pl.min() >= w.prompt_min and pl.max() <= w.prompt_max
    assert T.min() >= w.out_min and T.max() <= w.out_max
    # lognormal around the median
    assert 0.6 * w.out_median < np.median(T) < 1.6 * w.out_median


def test_demand_phases_switch_noise_scale():
    w = synth.WORKLOADS["llama8b_32layer"]
    st = synth.RequestStream(w, 5, 4096)
    s0 = st.sigma_q()
    st.t = w.phase_len
    s1 = st.sigma_q()
    assert {s0, s1} == {w.sigma_q, w.sigma_q * w.diffuse_factor}
