#!/usr/bin/env python
"""Decode throughput of the GrowPage hot path on one B300 (or N replicas).

Default workload: a 32-layer Llama-3-8B-shaped attention stack (32 q heads,
8 kv heads, d=128, bf16 K/V/q, fp32 summaries), batch 64 kept full from a
seeded request stream (prompts 128-1024 tokens, lognormal output lengths,
median 4096, clipped to 1k-16k, demand phases every 512 steps), page 16,
a 40 GB page pool, initial budget 64 pages, Top-p 0.9, recent window 64.

One step = one decode step of the whole path: for every layer the fused
paged-attention + summary kernel, then the boundary kernels (working sets,
grow / compact, compaction moves, commit).  The same kernels are timed
again in full-KV mode (every boundary grows, nothing is compacted; the host
preempts when the pool is full).

Timing: CUDA events on the pool's stream around each step's launches; the
next step's inputs are drawn on the device between steps, outside the
events.  The pool (tens of GB) is far larger than L2.  The attention
kernel's average launch time comes from events around layers 1..L-1 of
each timed step.  Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import contextlib
import gc
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

# DRAM bytes (read + write) per attention launch over its algorithmic K/V
# bytes, from one ncu capture of attn_mma_kernel on the same heads and
# requests with 4 layers and a 1.5 GB pool (two launches: 1.033 and 1.031).
# The bench's launches are too large to capture, so the traffic it reports
# is this ratio times its own algorithmic bytes per launch.
TRAFFIC_RATIO = 1.032
TRAFFIC_SOURCE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of attn_mma_kernel on a "
                  "4-layer, 1.5 GB-pool case (ratio 1.032 to its algorithmic bytes), scaled to "
                  "this launch's algorithmic bytes")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b_32layer")
    ap.add_argument("--preroll", type=int, default=1024,
                    help="untimed decode steps before warm-up (boundaries need history)")
    ap.add_argument("--no-full-kv", action="store_true")
    ap.add_argument("--no-policies", action="store_true",
                    help="skip the ablation policies (fixed, inverse, random, shrink)")
    ap.add_argument("--e2e-steps", type=int, default=48)
    ap.add_argument("--e2e-chunk", type=int, default=8,
                    help="largest group of layers per host<->device copy in the e2e measurement")
    ap.add_argument("--e2e-ramp", type=int, default=0,
                    help="1: copy groups grow 1, 2, 4, .. up to --e2e-chunk for the inputs and "
                         "shrink back to 1 for the outputs; 0: equal groups")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (small profiling cases)")
    ap.add_argument("--pool-gb", type=float, default=0.0,
                    help="override the page-pool size in GB (small profiling cases)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch size (small profiling cases)")
    ap.add_argument("--late-preroll", type=int, default=4096,
                    help="second timed window of the default workload after this many decode "
                         "steps, where full KV has grown (0: none)")
    ap.add_argument("--late-steps", type=int, default=128)
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads (1-layer, continuous batching, burst)")
    ap.add_argument("--workloads", default="llama8b_1layer,qwen3_8b_36layer_cb,stress_burst")
    ap.add_argument("--cb-preroll", type=int, default=2560,
                    help="continuous-batching workload: decode steps before its window "
                         "(arrivals fill the 128 slots by about step 1600)")
    ap.add_argument("--cb-steps", type=int, default=128)
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay of the one-layer workload")
    ap.add_argument("--no-async", action="store_true",
                    help="skip the asynchronous boundary measurement")
    ap.add_argument("--burst-steps", type=int, default=1024,
                    help="burst workload: timed steps from its first step (a burst every 16)")
    return ap.parse_args()


def workload_for(args):
    """The named workload, with the profiling overrides applied."""
    from demand_paged_kv_gqa_b300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.layers:
        w = w.replace(num_layers=args.layers)
    if args.batch:
        w = w.replace(batch=args.batch)
    if args.layers or args.pool_gb:
        gb = args.pool_gb or (w.num_pages * 2 * w.num_kv_heads * w.page_size * w.head_dim
                              * w.elem_bytes * synth.WORKLOADS[args.workload].num_layers / 1e9)
        page = w.num_layers * w.num_kv_heads * 2 * w.page_size * w.head_dim * w.elem_bytes
        w = w.replace(num_pages=int(gb * 1e9 // page))
    return w


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = []
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        smax = 0.0
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = max(smax, float(r[2]))
            except ValueError:
                continue
            for nm, val in zip(names, r[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(nm)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def reduce_over_ranks(t_ms, tokens, device):
    """Max over ranks of the timed milliseconds and sum of the tokens.

    Replicas share nothing on the data path (requests are independent); this
    host-side reduction of the timing is the only cross-rank step."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(t_ms), float(tokens)
    tt = torch.tensor([float(t_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    nn = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(nn)
    return float(tt.item()), float(nn.item())


# ------------------------------------------------------------ byte counts

def attention_bytes(w, tok, req_steps, btok):
    """Algorithmic HBM bytes of the attention kernel for one layer.

    tok: resident tokens summed over the requests (and steps) covered;
    req_steps: request-steps covered; btok: resident tokens of requests at a
    boundary (their summary scores are written).
    """
    eb = w.elem_bytes
    hk, hq, d, P = w.num_kv_heads, w.num_q_heads, w.head_dim, w.page_size
    kv = tok * hk * 2 * d * eb                       # K and V of resident tokens
    per_req = (2 * hq * d * eb                       # q read, out written
               + 2 * hk * d * eb                     # new k, v read
               + 2 * hk * d * eb                     # staged token written
               + 2 * 2 * hk * d * 4)                 # both summaries read + written
    bt = tok / P * 4                                 # block-table entries
    logits = btok * 2 * hk * 4                       # summary scores written
    return kv + req_steps * per_req + bt + logits


# ------------------------------------------------------------ our arm

def _load_peaks():
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = json.load(open(pk)) if os.path.exists(pk) else {}
    if "hbm_gbs" in peaks:
        return float(peaks["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


@contextlib.contextmanager
def no_gc():
    """Python's garbage collector off inside a timed region (collected just
    before): a collection pause while the host is issuing a step's launches
    would leave the GPU idle inside that step's events."""
    gc.collect()
    gc.disable()
    try:
        yield
    finally:
        gc.enable()


def time_window(eng, steps, w, sample_clocks=False, local=0, layer_events=True):
    """Time `steps` decode steps of an engine with CUDA events on its stream.

    Events per step: before the step, after layer 0, after the last layer,
    after the boundary call.  The layer-call time is taken over layers
    1..L-1 (for a 1-layer stack: the whole step before the boundary call,
    plan kernel included).  With layer_events False (a step replayed as one
    CUDA graph) only the step's ends are timed.  Returns the window's counters
    and times.
    """
    stream = eng.pool.stream
    L = w.num_layers
    torch.cuda.synchronize()
    st0 = eng.pool.stats()
    launches0 = eng.pool.launch_count() + eng.graph_launches
    tok0 = eng.tokens_timed
    pre0 = eng.preempted
    evs, nbs = [], []
    req_steps = 0
    clk = ClockSampler(local) if sample_clocks else None
    if clk:
        clk.start()
    # the whole window, input draws between steps included (compares the
    # synchronous and asynchronous boundary paths on equal terms)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with no_gc():
        w0.record(stream)
        for _ in range(steps):
            eng.prepare_inputs()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

            def before():
                e[0].record(stream)

            def after_layer(l):
                if l == 0:
                    e[1].record(stream)
                if l == L - 1:
                    e[2].record(stream)

            def after():
                e[3].record(stream)

            n = eng.step(timed=True, before_step=before, after_step=after,
                         after_layer=after_layer if layer_events else None)
            if n:
                req_steps += n
                evs.append(e)
                nbs.append(eng.last_boundaries)
        if eng.side is not None:
            stream.wait_stream(eng.side)
        w1.record(stream)
        torch.cuda.synchronize()
    clocks = clk.stop() if clk else None
    st1 = eng.pool.stats()
    step_t = [e[0].elapsed_time(e[3]) for e in evs]
    bnd_t = [e[2].elapsed_time(e[3]) for e in evs] if layer_events else [0.0] * len(evs)
    if not layer_events:
        attn_ms, n_attn = 0.0, 0
    elif L > 1:
        attn_ms = sum(e[1].elapsed_time(e[2]) for e in evs)
        n_attn = (L - 1) * len(evs)
    else:
        attn_ms = sum(e[0].elapsed_time(e[2]) for e in evs)
        n_attn = len(evs)
    step_ms = sum(step_t)
    dtok = st1.tokens_attended - st0.tokens_attended
    dbtok = st1.boundary_tokens - st0.boundary_tokens
    nsteps = max(1, len(evs))
    per_layer_bytes = attention_bytes(w, dtok, req_steps, dbtok)   # one layer, all steps
    res = dict(steps=len(evs), step_ms=step_ms, attn_ms=attn_ms, tokens=eng.tokens_timed - tok0,
               clocks=clocks, launches=eng.pool.launch_count() + eng.graph_launches - launches0,
               dtok=dtok,
               dbtok=dbtok, req_steps=req_steps,
               boundaries=st1.boundaries - st0.boundaries, grows=st1.grows - st0.grows,
               compacts=st1.compacts - st0.compacts, denied=st1.denied - st0.denied,
               shrinks=st1.shrinks - st0.shrinks, starved=st1.starved - st0.starved,
               moved=st1.moved_tokens - st0.moved_tokens, preempted=eng.preempted - pre0,
               free_pages=st1.free_top, num_pages=eng.num_pages,
               attn_launch_ms=attn_ms / n_attn if n_attn else float("nan"),
               attn_bytes_per_launch=per_layer_bytes / nsteps,
               attn_gbs=(per_layer_bytes * n_attn / nsteps / (attn_ms * 1e-3) / 1e9) if attn_ms else 0.0,
               step_bytes=per_layer_bytes * L / nsteps,
               step_gbs=per_layer_bytes * L / (step_ms * 1e-3) / 1e9 if step_ms else 0.0,
               window_ms=w0.elapsed_time(w1))
    # steps with boundaries against steps without (the boundary burst)
    bt = [(t, b) for t, b, nb in zip(step_t, bnd_t, nbs) if nb > 0]
    qt = [t for t, nb in zip(step_t, nbs) if nb == 0]
    res["boundary_steps"] = len(bt)
    res["boundary_step_ms"] = sum(t for t, _ in bt) / len(bt) if bt else None
    res["boundary_call_ms"] = sum(b for _, b in bt) / len(bt) if bt else None
    res["plain_step_ms"] = sum(qt) / len(qt) if qt else None
    res["mean_boundaries_per_boundary_step"] = (sum(nb for nb in nbs if nb) / len(bt)) if bt else 0
    return res


def summarize(r, ws, hbm_peak):
    """The per-mode object of the JSON line from a timed window."""
    o = {"value": round(r["tokens"] / (r["step_ms"] * 1e-3) * ws, 1) if r["step_ms"] else 0.0,
         "unit": "tokens/s",
         "ms_per_step": round(r["step_ms"] / max(1, r["steps"]), 4),
         "layer_call_gbs": round(r["attn_gbs"], 1),
         "layer_call_frac": round(r["attn_gbs"] / hbm_peak, 4),
         "step_gbs": round(r["step_gbs"], 1),
         "mean_batch": round(r["req_steps"] / max(1, r["steps"]), 1),
         "window_value": round(r["tokens"] / (r["window_ms"] * 1e-3) * ws, 1),
         "mean_resident_tokens": round(r["dtok"] / max(1, r["req_steps"]), 1)}
    o.update({k: int(r[k]) for k in ("steps", "tokens", "boundaries", "grows", "compacts",
                                     "denied", "starved", "shrinks", "preempted")})
    if r["boundary_steps"]:
        o["boundary_steps"] = {
            "count": r["boundary_steps"],
            "mean_requests_at_boundary": round(r["mean_boundaries_per_boundary_step"], 1),
            "step_ms": round(r["boundary_step_ms"], 4),
            "boundary_call_ms": round(r["boundary_call_ms"], 4),
            "plain_step_ms": round(r["plain_step_ms"], 4) if r["plain_step_ms"] else None}
    return o


def run_ours(args, ws, rank, local):
    from demand_paged_kv_gqa_b300 import growpage as gpb
    from demand_paged_kv_gqa_b300 import synth
    from demand_paged_kv_gqa_b300.engine import Engine

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workload_for(args)
    hbm_peak, peak_src = _load_peaks()

    def run_engine(wl, mode, label, windows, rate=0.0, extras=False, async_boundary=False,
                   graph=False):
        """One engine; windows = [(decode steps before the window, timed steps)].
        The warm-up steps come right before the first window."""
        eng = Engine(wl, mode=mode, device=dev, seed_offset=rank, random_grow_rate=rate,
                     async_boundary=async_boundary, use_graph=graph)
        eng.fill()
        out = []
        for k, (start, steps) in enumerate(windows):
            target = start + (args.warmup if k == 0 else 0)
            while eng.clock < target:
                eng.prepare_inputs()
                eng.step()
            if k == 0 and ws > 1:
                torch.distributed.barrier()
            r = time_window(eng, steps, wl, sample_clocks=(k == 0), local=local,
                            layer_events=not graph)
            r["label"], r["start"] = label, eng.clock - steps
            if k == 0 and extras:
                r["ceilings"] = measure_ceilings(eng, wl)
                r["e2e"] = (measure_e2e(eng, wl, args.e2e_steps, args.e2e_chunk, bool(args.e2e_ramp))
                            if args.e2e_steps else None)
            out.append(r)
        eng.pool.sync()
        del eng
        torch.cuda.empty_cache()
        return out

    def measure_ceilings(eng, wl):
        """Read-only streaming of the same resident K/V through the same grid:
        paged (the attention kernel's access pattern), sequential TMA, and
        sequential plain loads; GB/s of bytes moved."""
        act = eng.active()
        if eng.cfg.dtype != gpb.GP_DTYPE_BF16 or eng.cfg.head_dim != 128 or not act:
            return None
        slots = torch.tensor(act, dtype=torch.int32, device=dev)
        sink = torch.zeros(4, dtype=torch.int32, device=dev)
        stream = eng.pool.stream
        L = wl.num_layers
        out = {}
        for mode, name in ((0, "paged_tma"), (1, "seq_tma"), (2, "seq_ldg")):
            eng.pool.kv_read_ceiling(0, L, mode, slots, sink)      # warm
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            eng.pool.kv_read_ceiling(0, L, mode, slots, sink)
            e1.record(stream)
            torch.cuda.synchronize()
            s = sink.cpu().tolist()
            nbytes = (s[2] & 0xffffffff) + ((s[3] & 0xffffffff) << 32)
            out[name + "_gbs"] = round(nbytes * L / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
        out["bytes_per_launch"] = nbytes
        return out

    def groups(L, chunk, ramp):
        """Layer groups [(first, end)]: equal groups of `chunk`, or with
        `ramp` sizes 1, 2, 4, .. up to `chunk` and then `chunk`."""
        out, c, size = [], 0, (1 if ramp else chunk)
        while c < L:
            out.append((c, min(c + size, L)))
            c += size
            size = min(2 * size, chunk)
        return out

    def measure_e2e(eng, wl, k, chunk=8, ramp=True):
        """Same metric through the C-ABI with each step's q, k, v copied from
        pinned host memory and its outputs copied back to pinned host memory,
        all copies inside the events.  The copies run on a second stream in
        groups of layers: a group's inputs are copied ahead, the compute
        stream waits once per group, and a group's outputs go back while the
        next group computes (what a serving loop over the per-layer call
        does; waiting before every layer would break the programmatic
        chaining of the layer kernels).  With `ramp`, the input groups start
        small (the first layer waits only for its own inputs) and the output
        groups end small (little is left to copy after the last layer)."""
        stream = eng.pool.stream
        copy = torch.cuda.Stream(device=dev)
        L = wl.num_layers
        chunks = groups(L, chunk, ramp)
        out_chunks = [(L - b, L - a) for a, b in reversed(groups(L, chunk, ramp))]
        hq_ = torch.empty_like(eng.q, device="cpu").pin_memory()
        hk_ = torch.empty_like(eng.k, device="cpu").pin_memory()
        hv_ = torch.empty_like(eng.v, device="cpu").pin_memory()
        ho_ = torch.empty_like(eng.out, device="cpu").pin_memory()
        ms = 0.0
        toks = 0
        warm = 3  # untimed: the copy stream's and pinned buffers' first use
        with no_gc():
            for it in range(k + warm):
                eng.prepare_inputs()
                hq_.copy_(eng.q); hk_.copy_(eng.k); hv_.copy_(eng.v)
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                in_ready = {c0: torch.cuda.Event() for c0, _ in chunks}
                out_ready = {c1 - 1: torch.cuda.Event() for _, c1 in out_chunks}

                def before():
                    e0.record(stream)
                    copy.wait_event(e0)
                    with torch.cuda.stream(copy):
                        for c0, c1 in chunks:
                            eng.q[c0:c1].copy_(hq_[c0:c1], non_blocking=True)
                            eng.k[c0:c1].copy_(hk_[c0:c1], non_blocking=True)
                            eng.v[c0:c1].copy_(hv_[c0:c1], non_blocking=True)
                            in_ready[c0].record(copy)

                def before_layer(l):
                    if l in in_ready:
                        stream.wait_event(in_ready[l])

                def after_layer(l):
                    if l in out_ready:
                        c0 = max(c for c, _ in out_chunks if c <= l)
                        out_ready[l].record(stream)
                        copy.wait_event(out_ready[l])
                        with torch.cuda.stream(copy):
                            ho_[c0:l + 1].copy_(eng.out[c0:l + 1], non_blocking=True)

                def after():
                    done = torch.cuda.Event()
                    done.record(copy)
                    stream.wait_event(done)
                    e1.record(stream)

                n = eng.step(before_step=before, after_step=after, before_layer=before_layer,
                             after_layer=after_layer)
                torch.cuda.synchronize()
                if it >= warm:
                    ms += e0.elapsed_time(e1)
                    toks += n
        h2d = hq_.nbytes + hk_.nbytes + hv_.nbytes
        d2h = ho_.nbytes
        return dict(value=toks / (ms * 1e-3), h2d=h2d, d2h=d2h)

    windows = [(args.preroll, args.steps)]
    if args.late_preroll and args.late_preroll > args.preroll + args.warmup + args.steps:
        windows.append((args.late_preroll, args.late_steps))
    gp_runs = run_engine(w, gpb.GP_MODE_GROWPAGE, "growpage", windows, extras=True)
    gp_res = gp_runs[0]
    fk_runs = None if args.no_full_kv else run_engine(w, gpb.GP_MODE_FULL_KV, "full_kv", windows)
    # the review's ablation policies on the same kernels and workload; RANDOM
    # grows at GrowPage's measured grow frequency
    pol_res = {}
    if not args.no_policies:
        rate = gp_res["grows"] / max(1, gp_res["boundaries"])
        for name, mode, r in (("fixed", gpb.GP_MODE_FIXED, 0.0),
                              ("inverse", gpb.GP_MODE_INVERSE, 0.0),
                              ("random", gpb.GP_MODE_RANDOM, rate),
                              ("shrink", gpb.GP_MODE_SHRINK, 0.0)):
            pol_res[name] = run_engine(w, mode, name, windows[:1], rate=r)[0]
            pol_res[name]["rate"] = r
    # the boundary work on a second stream (gp_boundary_async), requests at a
    # boundary sitting out one step: the default workload and the burst
    async_res = {}
    if not args.no_async:
        async_res[w.name] = run_engine(w, gpb.GP_MODE_GROWPAGE, "async", windows[:1],
                                       async_boundary=True)[0]
    # the other workloads, each GrowPage against full KV on the same kernels
    other = {}
    if not args.no_workloads:
        plan = {"llama8b_1layer": (args.preroll, args.steps),
                "qwen3_8b_36layer_cb": (args.cb_preroll, args.cb_steps),
                "stress_burst": (0, args.burst_steps)}
        for name in [x for x in args.workloads.split(",") if x]:
            wl = synth.WORKLOADS[name]
            start, steps = plan.get(name, (args.preroll, args.steps))
            other[name] = {"growpage": run_engine(wl, gpb.GP_MODE_GROWPAGE, "growpage",
                                                  [(start, steps)])[0],
                           "full_kv": run_engine(wl, gpb.GP_MODE_FULL_KV, "full_kv",
                                                 [(start, steps)])[0]}
            if name == "llama8b_1layer" and not args.no_graph:
                # a one-layer step is too short to hide the host's launches:
                # the same steps replayed as one CUDA graph each
                for key, mode in (("growpage_graph", gpb.GP_MODE_GROWPAGE),
                                  ("full_kv_graph", gpb.GP_MODE_FULL_KV)):
                    try:
                        other[name][key] = run_engine(wl, mode, key, [(start, steps)], graph=True)[0]
                    except Exception as ex:  # capture refused: report it, keep the rest
                        other[name][key + "_error"] = str(ex)[:200]
            if name == "stress_burst" and not args.no_async:
                async_res[name] = run_engine(wl, gpb.GP_MODE_GROWPAGE, "async", [(start, steps)],
                                             async_boundary=True)[0]

    # max over ranks of the time, sum of tokens
    t_ms, tokens = reduce_over_ranks(gp_res["step_ms"], gp_res["tokens"], dev)
    if rank != 0:
        return None
    value = tokens / (t_ms * 1e-3)
    a_gbs = gp_res["attn_gbs"]
    mma_path = w.dtype == "bf16" and w.head_dim == 128  # attn_mma_kernel runs
    line = {
        "metric": "decode tokens/s per B300 (GrowPage vs full-KV); % of HBM roofline",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded walk queries, planted keys, N(0,1) keys/values)",
        "config": {
            "workload": f"{w.name}: {w.num_layers} layers, {w.num_q_heads}q/{w.num_kv_heads}kv, "
                        f"d={w.head_dim}, {w.dtype}, batch {w.batch}, page {w.page_size}, "
                        f"pool {gp_res['num_pages']} pages, budget {w.budget_pages} pages, "
                        f"top_p {w.top_p}, window {w.recent_window}",
            "mode": "growpage",
            "preroll_steps": args.preroll,
            "l2": "inputs larger than L2 (page pool of tens of GB)",
            "timing": "CUDA events around each step's launches; inputs drawn between steps",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": ("attn_mma_kernel + combine_kernel" if mma_path else "attn_kernel")
                      + " (one gp_decode_step layer call: paged GQA decode + summaries)",
            "achieved": round(a_gbs, 1),
            "peak": hbm_peak,
            "peak_source": peak_src,
            "unit": "GB/s",
            "frac": round(a_gbs / hbm_peak, 4),
            "traffic": (round(TRAFFIC_RATIO * gp_res["attn_bytes_per_launch"])
                        if mma_path else None),
            "traffic_source": TRAFFIC_SOURCE if mma_path else None,
            "bytes_per_launch": round(gp_res["attn_bytes_per_launch"]),
            "launch_ms": round(gp_res["attn_launch_ms"], 5),
        },
        "step_roofline": {
            "achieved": round(gp_res["step_gbs"], 1), "unit": "GB/s",
            "frac": round(gp_res["step_gbs"] / hbm_peak, 4),
            "frac_of_8tbs": round(gp_res["step_gbs"] / 8000.0, 4),
        },
        "read_ceilings": gp_res.get("ceilings"),
        "gpu_launches": int(gp_res["launches"]),
        "clocks": gp_res["clocks"],
        "growpage": summarize(gp_res, ws, hbm_peak),
    }
    line["growpage"]["moved"] = int(gp_res["moved"])
    if gp_res.get("e2e"):
        e = gp_res["e2e"]
        line["e2e"] = {"value": round(e["value"] * ws, 1), "unit": "tokens/s",
                       "h2d_bytes_per_step": int(e["h2d"]), "d2h_bytes_per_step": int(e["d2h"])}
    if fk_runs:
        line["full_kv"] = summarize(fk_runs[0], ws, hbm_peak)
        line["growpage_vs_full_kv"] = round(line["growpage"]["value"] / max(1e-9, line["full_kv"]["value"]), 4)
    if len(gp_runs) > 1:
        late = {"start_step": int(gp_runs[1]["start"]), "growpage": summarize(gp_runs[1], ws, hbm_peak)}
        if fk_runs:
            late["full_kv"] = summarize(fk_runs[1], ws, hbm_peak)
            late["growpage_vs_full_kv"] = round(late["growpage"]["value"] /
                                                max(1e-9, late["full_kv"]["value"]), 4)
        line["late_window"] = late
    if pol_res:
        line["policies"] = {}
        for name, r in pol_res.items():
            o = summarize(r, ws, hbm_peak)
            if name == "random":
                o["random_grow_rate"] = round(r["rate"], 4)
            line["policies"][name] = o
    if async_res:
        line["async_boundary"] = {}
        for name, r in async_res.items():
            sync_r = gp_res if name == w.name else other[name]["growpage"]
            o = {"growpage_async": summarize(r, ws, hbm_peak),
                 "growpage_sync_window_value": summarize(sync_r, ws, hbm_peak)["window_value"]}
            o["async_over_sync"] = round(o["growpage_async"]["window_value"] /
                                         max(1e-9, o["growpage_sync_window_value"]), 4)
            line["async_boundary"][name] = o
    if other:
        line["workloads"] = {}
        for name, rr in other.items():
            wl = synth.WORKLOADS[name]
            o = {"config": f"{wl.num_layers} layers, {wl.num_q_heads}q/{wl.num_kv_heads}kv, "
                           f"d={wl.head_dim}, {wl.dtype}, batch {wl.batch}, page {wl.page_size}, "
                           f"pool {rr['growpage']['num_pages']} pages, budget {wl.budget_pages} pages"
                           + (f", prefix {wl.prefix_len} per {wl.prefix_group} requests, Poisson "
                              f"{wl.arrival_rate}/s on {wl.step_seconds * 1000:.0f} ms steps, "
                              f"{wl.total_requests} requests" if wl.prefix_len else ""),
                 "window_start_step": int(rr["growpage"]["start"]),
                 "growpage": summarize(rr["growpage"], ws, hbm_peak),
                 "full_kv": summarize(rr["full_kv"], ws, hbm_peak)}
            o["growpage_vs_full_kv"] = round(o["growpage"]["value"] / max(1e-9, o["full_kv"]["value"]), 4)
            for key in ("growpage_graph", "full_kv_graph"):
                if key in rr:
                    o[key] = summarize(rr[key], ws, hbm_peak)
                    o[key]["gpu_launches"] = int(rr[key]["launches"])
                elif key + "_error" in rr:
                    o[key] = {"unavailable": rr[key + "_error"]}
            if "growpage_graph" in rr and "full_kv_graph" in rr:
                o["graph_growpage_vs_full_kv"] = round(o["growpage_graph"]["value"] /
                                                       max(1e-9, o["full_kv_graph"]["value"]), 4)
            line["workloads"][name] = o
    return line


# ------------------------------------------------------------ oracle arm

class OracleRunner:
    """The CPU oracle on one request of the workload (all layers), one thread.

    The request is admitted with a full initial budget (prompt = budget) so
    that its first step is a boundary, and every page-size-th step after
    it; `run` continues the same trajectory.
    """

    def __init__(self, w):
        from demand_paged_kv_gqa_b300 import synth
        from oracle.pool import OracleConfig, OraclePool
        try:
            from threadpoolctl import threadpool_limits
            self._lim = threadpool_limits(1)
        except Exception:
            self._lim = None
        torch.set_num_threads(1)
        self.w = w
        pl = w.budget_pages * w.page_size
        self.st = synth.RequestStream(w, 0, 1 << 20)
        k, v = self.st.prompt(pl)
        self.pool = OraclePool(OracleConfig.from_workload(w, num_pages=4 * w.budget_pages + 64,
                                                          max_pages_per_req=4 * w.budget_pages))
        self.pool.add_request(0, k.double().numpy(), v.double().numpy(), w.budget_pages)
        self.steps = 0

    def run(self, seconds, max_steps=None):
        """Decode steps until `seconds` have passed (at least one); returns
        (steps, seconds)."""
        n, t0 = 0, time.time()
        while True:
            q, kk, vv = self.st.next_step()
            self.pool.step([0], q[None].double().numpy(), kk[None].double().numpy(),
                           vv[None].double().numpy())
            n += 1
            el = time.time() - t0
            if el >= seconds or (max_steps and n >= max_steps):
                break
        self.steps += n
        return n, el


def oracle_sample(w, seconds, max_steps=None):
    """Tokens/s of the oracle over one bounded run: (tokens/s, steps, s, threads)."""
    r = OracleRunner(w)
    n, el = r.run(seconds, max_steps)
    return n / el, n, el, 1


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    w = workload_for(args)
    per_step = max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    runner = OracleRunner(w)
    for _ in range(args.warmup):          # warm-up: single decode steps, untimed
        runner.run(0.0, max_steps=1)
    steps, secs = 0, 0.0
    for _ in range(args.steps):           # each timed step: a bounded slice of the trajectory
        s, e = runner.run(per_step)
        steps += s
        secs += e
    value = steps / secs
    sample = (f"one request of {w.name} ({w.num_layers} layers, prompt = budget "
              f"{w.budget_pages * w.page_size} tokens, a boundary every {w.page_size} steps), "
              f"one continuous trajectory: {args.warmup} warm-up steps, then {steps} oracle "
              f"decode steps over {args.steps} samples")
    return {
        "impl": "reference",
        "metric": "decode tokens/s per B300 (GrowPage vs full-KV); % of HBM roofline",
        "value": round(value, 4), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1000 * secs / max(1, steps), 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "mode": "growpage"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    ws, rank, local = dist_info()
    if ws > 1:
        backend = "gloo" if args.impl == "reference" else "nccl"
        torch.distributed.init_process_group(backend)
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
    else:
        line = run_ours(args, ws, rank, local)
        if line is not None and not args.no_cpu_baseline and ws == 1:  # N = 1 only
            w = workload_for(args)
            v, s, e, cores = oracle_sample(w, args.cpu_seconds)
            line["cpu_baseline"] = {
                "value": round(v, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "sample": f"one request of {w.name}, all {w.num_layers} layers, {s} decode steps "
                          f"({e:.1f} s), prompt = initial budget so boundaries occur"}
    if line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
