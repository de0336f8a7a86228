"""CPU oracle for the GrowPage decode path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct fp64 restatement of what the decode path
computes, used to check the CUDA path.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm
may import it.  The product path (the C-ABI library and its binding) never
imports, links or executes anything here, and nothing here imports the
product path: the two share no code.  The only thing both consume is the
seeded input generator ``demand_paged_kv_gqa_b300.synth``, which holds no
arithmetic of the method; the oracle itself does not import it either.

Source of the method: the web pages titled "GrowPage: On-Demand KV Budgeting
for Efficient LLM Reasoning Serving" -- the paper's abstract, and the
evolve.pub AI review (sections "Summary" and "Frequently asked questions").
Those pages give the method in prose only; every convention they leave open
is a reading stated in the docstring of the function that takes it.

Parity status of each function (what pins it, see tests/test_oracle_pins.py):

* ``numerics.rope_*``       pinned: complex-exponential form, relative-position
                            identity, norm preservation.
* ``numerics.round_bf16``   pinned: exact rational rounding (fractions) and
                            torch's fp32->bf16 cast.
* ``numerics.ema_fold``     pinned: fp64 closed form of the recurrence; beta=0.
* ``policy.topp_count``     pinned: brute force over all subsets; uniform and
                            one-hot closed forms.
* ``policy.drop_set``       pinned: brute-force ranking with Python tuples.
* ``pool.OraclePool``       pinned: dense softmax attention (torch SDPA) with
                            compaction off; GQA G=1 equals MHA; pool
                            invariants; hand-built grow / compact cases.
* boundary wiring: ``OraclePool._summary_scores``, ``policy.private_importance``
  and ``policy.delta_range``, pinned in tests/test_oracle_boundary_pins.py:
  the summary scores against a recomputation with complex-rotation RoPE and
  closed-form EMAs; the importance normalisation by a case where
  normalising over private tokens only keeps another set; the near-tie
  exemption by enumerating every working-set size inside its band.  Each
  pin is shown to fail on its plausible mistake.
* decision statistics vs the paper's measured grow ratios: parity unpinned
  (the pages print no worked example or intermediate values).
"""
