"""Seeded synthetic workloads for the GrowPage decode path.

This module only draws random numbers and arranges them into the tensors a
decode step consumes (prompt keys/values, per-step queries, keys and values).
It holds none of the method's arithmetic: no RoPE, no summaries, no softmax,
no page bookkeeping. Both the CUDA path (through the binding) and the CPU
oracle are fed from these same tensors.

Recipe (shared by every workload; the sizes are in ``WORKLOADS``):

* Per (request, layer, kv head) a slow Gaussian random walk
  ``w_0 ~ N(0, I)``, ``w_t = w_{t-1} + walk_step * N(0, I)`` and its direction
  ``u_t = w_t / |w_t|``.  With RoPE on, the walk is confined to the slowest
  rotating quarter of the rotary pairs (the last d/8 indices of each half of
  the head), so that an alignment between a query and a key survives the
  rotation by their relative position; without RoPE it spans all d dims.
* Query of q head h (kv head g = h // G) at decode step t:
  ``q = sqrt(d) * u_t + sigma_q * N(0, I)``.  ``sigma_q`` is 0.5, or 1.5 in the
  "diffuse" demand phase of workloads that switch phases.
* New key and value of a decode step ~ N(0, I), except that at the planted
  steps ``s_j = j * T // n_planted`` (T = the request's decode length) the new
  key of every (layer, kv head) is ``sqrt(d) * u_t`` (a hot key).
* Prompt keys/values ~ N(0, I).
* All tensors are produced in fp32 and then cast once to the storage dtype.

Determinism: every request owns a ``torch.Generator`` seeded from
``(workload seed, request id)``, so a request's stream does not depend on
which other requests share its batch.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    dtype: str                 # "f32" or "bf16": storage dtype of K/V/q/out
    rope_theta: float          # 0.0 means no rotary embedding
    top_p: float
    recent_window: int
    beta_s: float = 0.9
    beta_l: float = 0.999
    tau: float = 0.0
    batch: int = 1             # concurrent requests
    prompt_min: int = 64
    prompt_max: int = 64
    budget_pages: int = 4      # initial private pages per request
    num_pages: int = 32        # physical pages in the pool
    decode_steps: int = 256    # fixed decode length (when out_median == 0)
    out_median: int = 0        # lognormal output lengths when > 0
    out_sigma: float = 0.0
    out_min: int = 0
    out_max: int = 0
    sigma_q: float = 0.5
    diffuse_factor: float = 1.0
    phase_len: int = 0         # 0: no demand phases
    walk_step: float = 0.05
    n_planted: int = 8
    prefix_len: int = 0        # shared prefix tokens (0: none)
    prefix_group: int = 0      # consecutive requests sharing one prefix
    arrival_rate: float = 0.0  # Poisson arrivals per second (continuous batching)
    step_seconds: float = 0.0  # virtual clock per decode step
    total_requests: int = 0
    max_pages_per_req: int = 0
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


GiB = 1 << 30


def _pages_for(bytes_total: float, w_layers: int, hk: int, d: int, p: int, eb: int) -> int:
    page_bytes = w_layers * hk * 2 * p * d * eb
    return int(bytes_total // page_bytes)


# The five workloads.  Names describe them; sizes follow the benchmark's configs.
WORKLOADS = {
    # 1 request, 1 layer, 2 kv heads x 2 q heads each, d=64, fp32, no RoPE.
    "tiny": Workload(
        name="tiny", num_layers=1, num_q_heads=4, num_kv_heads=2, head_dim=64,
        page_size=16, dtype="f32", rope_theta=0.0, top_p=0.9, recent_window=16,
        batch=1, prompt_min=64, prompt_max=64, budget_pages=4, num_pages=32,
        decode_steps=256, max_pages_per_req=32, seed=0),
    # One Llama-3-8B-shaped attention layer, batch 16.
    "llama8b_1layer": Workload(
        name="llama8b_1layer", num_layers=1, num_q_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, dtype="bf16", rope_theta=500000.0,
        top_p=0.9, recent_window=64, batch=16, prompt_min=128, prompt_max=1024,
        budget_pages=64, num_pages=4096, decode_steps=2048,
        max_pages_per_req=256, seed=1),
    # 32-layer Llama-3-8B-shaped attention stack, batch 64, demand phases.
    "llama8b_32layer": Workload(
        name="llama8b_32layer", num_layers=32, num_q_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, dtype="bf16", rope_theta=500000.0,
        top_p=0.9, recent_window=64, batch=64, prompt_min=128, prompt_max=1024,
        budget_pages=64,
        num_pages=_pages_for(40e9, 32, 8, 128, 16, 2),
        out_median=4096, out_sigma=math.log(2.0), out_min=1024, out_max=16384,
        sigma_q=0.5, diffuse_factor=3.0, phase_len=512,
        max_pages_per_req=1088, seed=2),
    # 36-layer Qwen3-8B-shaped stack, continuous batching, shared prefixes.
    "qwen3_8b_36layer_cb": Workload(
        name="qwen3_8b_36layer_cb", num_layers=36, num_q_heads=32,
        num_kv_heads=8, head_dim=128, page_size=16, dtype="bf16",
        rope_theta=1000000.0, top_p=0.9, recent_window=64, batch=128,
        prompt_min=0, prompt_max=0, budget_pages=64,
        num_pages=_pages_for(40e9, 36, 8, 128, 16, 2),
        out_median=8192, out_sigma=math.log(2.0), out_min=2048, out_max=32768,
        prefix_len=2048, prefix_group=8, arrival_rate=4.0, step_seconds=0.02,
        total_requests=512, max_pages_per_req=1024, seed=3),
    # Boundary-burst stress: every request at a boundary in the same step.
    "stress_burst": Workload(
        name="stress_burst", num_layers=32, num_q_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, dtype="bf16", rope_theta=500000.0,
        top_p=0.9, recent_window=64, batch=256, prompt_min=1024,
        prompt_max=1024, budget_pages=64,
        num_pages=_pages_for(120e9, 32, 8, 128, 16, 2),
        decode_steps=32768, max_pages_per_req=512, seed=4),
}


def walk_mask(w: Workload) -> torch.Tensor:
    """Boolean [d] mask of the dims the walk (and the hot keys) live in."""
    d = w.head_dim
    m = torch.zeros(d, dtype=torch.bool)
    if w.rope_theta == 0.0:
        m[:] = True
    else:
        h = d // 2
        q = max(1, h // 4)
        m[h - q:h] = True
        m[d - q:d] = True
    return m


def request_seed(w: Workload, rid: int) -> int:
    return (w.seed * 1_000_003 + rid * 7919 + 12345) & 0x7FFFFFFFFFFF


def draw_lengths(w: Workload, n: int, rid0: int = 0):
    """(prompt_len, decode_len) for requests rid0 .. rid0+n-1."""
    out = []
    for rid in range(rid0, rid0 + n):
        g = torch.Generator().manual_seed(request_seed(w, rid) ^ 0x5A5A)
        if w.prompt_max > w.prompt_min:
            pl = int(torch.randint(w.prompt_min, w.prompt_max + 1, (1,), generator=g))
        else:
            pl = w.prompt_min
        if w.out_median > 0:
            z = float(torch.randn(1, generator=g))
            t = int(round(w.out_median * math.exp(w.out_sigma * z)))
            t = min(max(t, w.out_min), w.out_max)
        else:
            t = w.decode_steps
        out.append((pl, t))
    return out


class RequestStream:
    """Per-request seeded generator of prompt and decode-step tensors."""

    def __init__(self, w: Workload, rid: int, decode_len: int, device="cpu"):
        self.w = w
        self.rid = rid
        self.T = decode_len
        self.device = torch.device(device)
        self.gen = torch.Generator(device=self.device)
        self.gen.manual_seed(request_seed(w, rid))
        L, hk, d = w.num_layers, w.num_kv_heads, w.head_dim
        self.mask = walk_mask(w).to(self.device).float()
        self.walk = self._randn(L, hk, d) * self.mask
        self.t = 0  # decode steps drawn so far
        if w.phase_len > 0:
            self.phase0 = int(torch.randint(0, 2, (1,), generator=self.gen,
                                            device=self.device).item())
        else:
            self.phase0 = 0
        n_pl = max(1, w.n_planted)
        self.planted = {(j * self.T) // n_pl for j in range(n_pl)} if w.n_planted > 0 else set()

    def _randn(self, *shape):
        return torch.randn(*shape, generator=self.gen, device=self.device,
                           dtype=torch.float32)

    def prompt(self, length: int):
        """Pre-RoPE prompt keys and values, each [L][length][Hk][d]."""
        w = self.w
        k = self._randn(w.num_layers, length, w.num_kv_heads, w.head_dim)
        v = self._randn(w.num_layers, length, w.num_kv_heads, w.head_dim)
        return k.to(w.torch_dtype), v.to(w.torch_dtype)

    def sigma_q(self) -> float:
        w = self.w
        if w.phase_len <= 0:
            return w.sigma_q
        phase = (self.phase0 + self.t // w.phase_len) % 2
        return w.sigma_q * (w.diffuse_factor if phase == 1 else 1.0)

    def next_step(self):
        """q [L][Hq][d], k [L][Hk][d], v [L][Hk][d] of the next decode step."""
        w = self.w
        L, hk, hq, d = w.num_layers, w.num_kv_heads, w.num_q_heads, w.head_dim
        if self.t > 0:
            self.walk = self.walk + w.walk_step * self._randn(L, hk, d) * self.mask
        u = self.walk / self.walk.norm(dim=-1, keepdim=True)
        sd = math.sqrt(d)
        sig = self.sigma_q()
        q = sd * u.repeat_interleave(w.group, dim=1) + sig * self._randn(L, hq, d)
        k = self._randn(L, hk, d)
        v = self._randn(L, hk, d)
        if self.t in self.planted:
            k = sd * u
        self.t += 1
        dt = w.torch_dtype
        return q.to(dt), k.to(dt), v.to(dt)


def prefix_tensors(w: Workload, prefix_index: int, device="cpu"):
    """Pre-RoPE keys/values of shared prefix number ``prefix_index``."""
    g = torch.Generator(device=torch.device(device))
    g.manual_seed((w.seed * 65_537 + prefix_index * 104_729 + 99) & 0x7FFFFFFFFFFF)
    shape = (w.num_layers, w.prefix_len, w.num_kv_heads, w.head_dim)
    k = torch.randn(*shape, generator=g, device=device)
    v = torch.randn(*shape, generator=g, device=device)
    return k.to(w.torch_dtype), v.to(w.torch_dtype)


def poisson_arrivals(w: Workload, n: int):
    """Arrival step of each of n requests (virtual clock of step_seconds)."""
    g = torch.Generator().manual_seed(w.seed * 31 + 7)
    gaps = torch.empty(n, dtype=torch.float64).exponential_(1.0, generator=g) / w.arrival_rate
    t = torch.cumsum(gaps, 0)
    return [int(x // w.step_seconds) for x in t.tolist()]


class BatchStream:
    """Device-side batched generator with the same recipe, for timing runs.

    Draws the inputs of a whole batch at once on one device.  It does not
    reproduce ``RequestStream`` bit for bit (a different draw order); it is
    used where only the distribution matters.
    """

    def __init__(self, w: Workload, n: int, decode_lens, device="cuda", seed=0):
        self.w = w
        self.n = n
        self.device = torch.device(device)
        self.gen = torch.Generator(device=self.device)
        self.gen.manual_seed(w.seed * 7 + seed + 1)
        L, hk, d = w.num_layers, w.num_kv_heads, w.head_dim
        self.mask = walk_mask(w).to(self.device).float()
        self.walk = self._randn(n, L, hk, d) * self.mask
        self.t = torch.zeros(n, dtype=torch.long, device=self.device)
        self.T = torch.as_tensor(list(decode_lens), device=self.device)
        if w.phase_len > 0:
            self.phase0 = torch.randint(0, 2, (n,), generator=self.gen, device=self.device)
        else:
            self.phase0 = torch.zeros(n, dtype=torch.long, device=self.device)

    def _randn(self, *shape):
        return torch.randn(*shape, generator=self.gen, device=self.device,
                           dtype=torch.float32)

    def reset_request(self, i: int, decode_len: int):
        L, hk, d = self.w.num_layers, self.w.num_kv_heads, self.w.head_dim
        self.walk[i] = self._randn(L, hk, d) * self.mask
        self.t[i] = 0
        self.T[i] = decode_len

    def next_step(self):
        """q [n][L][Hq][d], k/v [n][L][Hk][d] in the storage dtype."""
        w = self.w
        n, L, hk, hq, d = self.n, w.num_layers, w.num_kv_heads, w.num_q_heads, w.head_dim
        step = (self.t > 0).float().view(n, 1, 1, 1)
        self.walk = self.walk + step * w.walk_step * self._randn(n, L, hk, d) * self.mask
        u = self.walk / self.walk.norm(dim=-1, keepdim=True)
        sd = math.sqrt(d)
        if w.phase_len > 0:
            phase = (self.phase0 + self.t // w.phase_len) % 2
            sig = w.sigma_q * torch.where(phase == 1, w.diffuse_factor, 1.0)
        else:
            sig = torch.full((n,), w.sigma_q, device=self.device)
        q = sd * u.repeat_interleave(w.group, dim=2) + sig.view(n, 1, 1, 1) * self._randn(n, L, hq, d)
        k = self._randn(n, L, hk, d)
        v = self._randn(n, L, hk, d)
        # planted steps floor(j T / n_planted), j < n_planted, as in RequestStream:
        # t is one iff j = ceil(t n / T) is below n and floor(j T / n) == t
        npl = w.n_planted
        if npl > 0:
            j = (self.t * npl + self.T - 1) // self.T
            hot = (j < npl) & (j * self.T < (self.t + 1) * npl)
            k = torch.where(hot.view(n, 1, 1, 1), sd * u, k)
        self.t += 1
        dt = w.torch_dtype
        return q.to(dt), k.to(dt), v.to(dt)
