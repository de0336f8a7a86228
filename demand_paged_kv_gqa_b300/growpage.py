"""Python binding of libgrowpage.so (include/growpage.h).

Argument marshalling only: every step of the decode path runs in the
library's CUDA kernels.  torch provides device memory (the pool buffer the
library lays out, the per-step tensors) and the stream.  If the compiled
library is missing, importing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# GROWPAGE_LIB may name another build of the same library (e.g. a variant
# compiled with different tile constants); the default is the in-tree build.
LIB_PATH = os.environ.get("GROWPAGE_LIB") or os.path.join(_HERE, "libgrowpage.so")

GP_OK, GP_ERR_INVALID, GP_ERR_NO_PAGES, GP_ERR_CUDA, GP_ERR_DEVICE = 0, 1, 2, 3, 4
GP_DTYPE_F32, GP_DTYPE_BF16 = 0, 1
GP_MODE_GROWPAGE, GP_MODE_FULL_KV, GP_MODE_FIXED, GP_MODE_INVERSE, GP_MODE_RANDOM = 0, 1, 2, 3, 4
GP_MODE_SHRINK = 5
DEC_NONE, DEC_GROW, DEC_COMPACT, DEC_COMPACT_DENIED, DEC_STARVED, DEC_SHRINK = 0, 1, 2, 3, 4, 5


class gp_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "num_q_heads", "num_kv_heads", "head_dim", "page_size",
        "num_pages", "max_requests", "max_pages_per_req", "max_prefixes",
        "max_prefix_len", "max_seq_len", "dtype", "mode", "recent_window")] + [
        ("beta_s", ctypes.c_float), ("beta_l", ctypes.c_float),
        ("top_p", ctypes.c_float), ("tau", ctypes.c_float),
        ("rope_theta", ctypes.c_double), ("flags", ctypes.c_int32),
        ("random_grow_rate", ctypes.c_float)]


class gp_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "kv", "tok_pos", "block", "req", "summary", "staging", "logits", "wset",
        "free_stack", "ctrl", "prefix", "prefix_pages", "rope", "scratch", "total",
        "page_bytes")] + [(n, ctypes.c_int32) for n in (
        "block_width", "logit_width", "max_prefix_pages", "num_workers")]


class gp_req_meta(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "active", "prefix_id", "n_pre_pages", "n_pages", "seq_priv", "pos",
        "steps", "last_decision")] + [("delta", ctypes.c_int64)] + [
        (n, ctypes.c_int32) for n in ("n_boundaries", "n_grows", "n_compacts",
                                      "n_denied", "n_starved", "n_shrinks")]


class gp_ctrl(ctypes.Structure):
    _fields_ = [("free_top", ctypes.c_int32), ("status", ctypes.c_uint32),
                ("status_info", ctypes.c_int32), ("plan_n", ctypes.c_int32)] + [
        (n, ctypes.c_int64) for n in (
            "steps", "tokens_attended", "boundary_tokens", "boundaries", "grows",
            "compacts", "denied", "starved", "moved_tokens", "shrinks")] + [
        ("reserved", ctypes.c_int64 * 3)]


class gp_state_view(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("req", "block", "ctrl", "wset", "tok_pos",
                                               "free_stack")]


assert ctypes.sizeof(gp_req_meta) == 64


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m demand_paged_kv_gqa_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sigs = {
        "gp_pool_bytes": (ctypes.c_int, [ctypes.POINTER(gp_config), ctypes.POINTER(SZ)]),
        "gp_create_pool": (ctypes.c_int, [ctypes.POINTER(gp_config), P, SZ, P, ctypes.POINTER(P)]),
        "gp_destroy_pool": (ctypes.c_int, [P]),
        "gp_set_stream": (ctypes.c_int, [P, P]),
        "gp_get_layout": (ctypes.c_int, [P, ctypes.POINTER(gp_layout)]),
        "gp_add_prefix": (ctypes.c_int, [P, P, P, I32, ctypes.POINTER(I32)]),
        "gp_release_prefix": (ctypes.c_int, [P, I32]),
        "gp_add_request": (ctypes.c_int, [P, I32, P, P, I32, I32, I32]),
        "gp_decode_step": (ctypes.c_int, [P, I32, I32, P, P, P, P, P]),
        "gp_boundary": (ctypes.c_int, [P, I32, P]),
        "gp_boundary_async": (ctypes.c_int, [P, I32, P, P]),
        "gp_free": (ctypes.c_int, [P, I32]),
        "gp_sync": (ctypes.c_int, [P]),
        "gp_clear_status": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_uint32),
                                           ctypes.POINTER(I32)]),
        "gp_get_stats": (ctypes.c_int, [P, ctypes.POINTER(gp_ctrl)]),
        "gp_get_request": (ctypes.c_int, [P, I32, ctypes.POINTER(gp_req_meta),
                                          ctypes.POINTER(I32), I32]),
        "gp_get_state": (ctypes.c_int, [P, ctypes.POINTER(gp_state_view)]),
        "gp_kv_read_ceiling": (ctypes.c_int, [P, I32, I32, I32, I32, P, P]),
        "gp_kv_read_ceiling_static": (ctypes.c_int, [P, I32, I32, I32, I32, P, P]),
        "gp_last_error": (ctypes.c_char_p, [P]),
        "gp_launch_count": (I64, [P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class GrowPageError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"growpage error {code}: {msg}")
        self.code = code


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return GP_DTYPE_F32
    if dt == torch.bfloat16:
        return GP_DTYPE_BF16
    raise ValueError(dt)


def make_config(*, num_layers, num_q_heads, num_kv_heads, head_dim, page_size,
                num_pages, max_requests, max_pages_per_req, dtype, max_seq_len,
                max_prefixes=0, max_prefix_len=0, mode=GP_MODE_GROWPAGE,
                recent_window=64, beta_s=0.9, beta_l=0.999, top_p=0.9, tau=0.0,
                rope_theta=0.0, random_grow_rate=0.0) -> gp_config:
    c = gp_config()
    c.num_layers, c.num_q_heads, c.num_kv_heads = num_layers, num_q_heads, num_kv_heads
    c.head_dim, c.page_size, c.num_pages = head_dim, page_size, num_pages
    c.max_requests, c.max_pages_per_req = max_requests, max_pages_per_req
    c.max_prefixes, c.max_prefix_len, c.max_seq_len = max_prefixes, max_prefix_len, max_seq_len
    c.dtype = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    c.mode, c.recent_window = mode, recent_window
    c.beta_s, c.beta_l, c.top_p, c.tau = beta_s, beta_l, top_p, tau
    c.rope_theta, c.flags = rope_theta, 0
    c.random_grow_rate = random_grow_rate
    return c


def pool_bytes(cfg: gp_config) -> int:
    n = ctypes.c_size_t(0)
    rc = lib.gp_pool_bytes(ctypes.byref(cfg), ctypes.byref(n))
    if rc != GP_OK:
        raise GrowPageError(rc, "unsupported configuration")
    return n.value


class Pool:
    """Owns the device buffer (a torch tensor) and the library handle."""

    def __init__(self, cfg: gp_config, device="cuda", stream: Optional[torch.cuda.Stream] = None):
        self.cfg = cfg
        self.device = torch.device(device)
        self.nbytes = pool_bytes(cfg)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=self.device)
        self.stream = stream or torch.cuda.current_stream(self.device)
        h = ctypes.c_void_p()
        rc = lib.gp_create_pool(ctypes.byref(cfg), _ptr(self.buf), self.nbytes,
                                ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(h))
        if rc != GP_OK:
            raise GrowPageError(rc, "gp_create_pool failed")
        self.h = h
        lay = gp_layout()
        self._check(lib.gp_get_layout(self.h, ctypes.byref(lay)))
        self.layout = lay
        self.storage_dtype = torch.float32 if cfg.dtype == GP_DTYPE_F32 else torch.bfloat16

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            lib.gp_destroy_pool(h)
            self.h = None

    def _check(self, rc):
        if rc != GP_OK:
            raise GrowPageError(rc, lib.gp_last_error(self.h).decode())

    # ---- the calls of the decode path (+ administration) ----
    def add_prefix(self, k: torch.Tensor, v: torch.Tensor) -> int:
        pid = ctypes.c_int32(-1)
        self._check(lib.gp_add_prefix(self.h, _ptr(k), _ptr(v), k.shape[1], ctypes.byref(pid)))
        return pid.value

    def release_prefix(self, pid: int):
        self._check(lib.gp_release_prefix(self.h, pid))

    def add_request(self, slot: int, k: Optional[torch.Tensor], v: Optional[torch.Tensor],
                    budget_pages: int, prefix_id: int = -1):
        n = 0 if k is None else k.shape[1]
        self._check(lib.gp_add_request(self.h, slot, _ptr(k) if n else None,
                                       _ptr(v) if n else None, n, budget_pages, prefix_id))

    def decode_step(self, layer: int, slots: torch.Tensor, q, k, v, out):
        self._check(lib.gp_decode_step(self.h, layer, slots.numel(), _ptr(slots), _ptr(q),
                                       _ptr(k), _ptr(v), _ptr(out)))

    def boundary(self, slots: torch.Tensor):
        self._check(lib.gp_boundary(self.h, slots.numel(), _ptr(slots)))

    def boundary_async(self, slots: torch.Tensor, side: torch.cuda.Stream):
        """gp_boundary_async: the boundary requests' work on `side`; they sit
        out the next step."""
        self._check(lib.gp_boundary_async(self.h, slots.numel(), _ptr(slots),
                                          ctypes.c_void_p(side.cuda_stream)))

    def free(self, slot: int):
        self._check(lib.gp_free(self.h, slot))

    def sync(self):
        self._check(lib.gp_sync(self.h))

    def set_stream(self, stream: torch.cuda.Stream):
        """Enqueue later calls on `stream` (gp_set_stream)."""
        self._check(lib.gp_set_stream(self.h, ctypes.c_void_p(stream.cuda_stream)))
        self.stream = stream

    def clear_status(self):
        """Read and clear the device status word: (GP_ST_* bits, info)."""
        st, info = ctypes.c_uint32(0), ctypes.c_int32(0)
        self._check(lib.gp_clear_status(self.h, ctypes.byref(st), ctypes.byref(info)))
        return st.value, info.value

    def stats(self) -> gp_ctrl:
        s = gp_ctrl()
        self._check(lib.gp_get_stats(self.h, ctypes.byref(s)))
        return s

    def request(self, slot: int):
        m = gp_req_meta()
        w = self.layout.block_width
        bt = (ctypes.c_int32 * w)()
        self._check(lib.gp_get_request(self.h, slot, ctypes.byref(m), bt, w))
        return m, list(bt)[: m.n_pre_pages + m.n_pages]

    def state(self, tok_pos: bool = False) -> dict:
        """The pool's state on the host (gp_get_state): request metadata, block
        tables, counters, working-set sizes, the free stack and, if asked,
        every slot's token position."""
        import numpy as np
        c, lay = self.cfg, self.layout
        R = c.max_requests
        req = (gp_req_meta * R)()
        ctrl = gp_ctrl()
        block = np.zeros((R, lay.block_width), np.int32)
        wset = np.zeros((R, c.num_layers, c.num_kv_heads, 2), np.int32)
        free = np.zeros(c.num_pages, np.int32)
        pos = (np.zeros((c.num_pages, c.num_layers, c.num_kv_heads, c.page_size), np.int32)
               if tok_pos else None)
        v = gp_state_view(ctypes.cast(req, ctypes.c_void_p), block.ctypes.data,
                          ctypes.addressof(ctrl), wset.ctypes.data,
                          pos.ctypes.data if pos is not None else None, free.ctypes.data)
        self._check(lib.gp_get_state(self.h, ctypes.byref(v)))
        out = {"req": list(req), "block": block, "ctrl": ctrl, "wset": wset,
               "free_stack": free[: ctrl.free_top]}
        if pos is not None:
            out["tok_pos"] = pos
        return out

    def kv_read_ceiling(self, layer0: int, count: int, mode: int, slots: torch.Tensor,
                        sink: torch.Tensor):
        """Read-only streaming of layers' resident K/V (a bandwidth ceiling)."""
        self._check(lib.gp_kv_read_ceiling(self.h, layer0, count, mode, slots.numel(),
                                           _ptr(slots), _ptr(sink)))

    def kv_read_ceiling_static(self, layer0: int, count: int, mode: int, slots: torch.Tensor,
                               sink: torch.Tensor):
        """The same read, with its scratch in the library's static device array."""
        self._check(lib.gp_kv_read_ceiling_static(self.h, layer0, count, mode, slots.numel(),
                                                  _ptr(slots), _ptr(sink)))

    def launch_count(self) -> int:
        return int(lib.gp_launch_count(self.h))

    # ---- views of the caller-owned buffer (documented layout) ----
    def _view(self, off, count, dtype, shape):
        es = torch.empty((), dtype=dtype).element_size()
        return self.buf[off: off + count * es].view(dtype).view(*shape)

    def region(self, name: str) -> torch.Tensor:
        c, l = self.cfg, self.layout
        L, hk, d, P = c.num_layers, c.num_kv_heads, c.head_dim, c.page_size
        R = c.max_requests
        sd = self.storage_dtype
        if name == "kv":
            return self._view(l.kv, c.num_pages * L * hk * 2 * P * d, sd, (c.num_pages, L, hk, 2, P, d))
        if name == "tok_pos":
            return self._view(l.tok_pos, c.num_pages * L * hk * P, torch.int32, (c.num_pages, L, hk, P))
        if name == "block":
            return self._view(l.block, R * l.block_width, torch.int32, (R, l.block_width))
        if name == "summary":
            return self._view(l.summary, R * L * hk * 2 * d, torch.float32, (R, L, hk, 2, d))
        if name == "staging":
            return self._view(l.staging, R * L * hk * 2 * d, sd, (R, L, hk, 2, d))
        if name == "logits":
            return self._view(l.logits, R * L * hk * 2 * l.logit_width, torch.float32,
                              (R, L, hk, 2, l.logit_width))
        if name == "wset":
            return self._view(l.wset, R * L * hk * 2, torch.int32, (R, L, hk, 2))
        if name == "req":  # gp_req_meta as 16 int32 words per slot (delta: words 8-9)
            return self._view(l.req, R * 16, torch.int32, (R, 16))
        if name == "free_stack":
            return self._view(l.free_stack, c.num_pages, torch.int32, (c.num_pages,))
        raise KeyError(name)


def config_for(w, mode=GP_MODE_GROWPAGE, max_requests=None, num_pages=None,
               max_seq_len=None, max_prefixes=None, random_grow_rate=0.0,
               max_pages_per_req=None) -> gp_config:
    """gp_config for a synth.Workload."""
    max_out = max(w.decode_steps, w.out_max)
    seq = max_seq_len or (w.prefix_len + w.prompt_max + max_out + 16)
    if max_prefixes is None:
        max_prefixes = 0
        if w.prefix_len:
            grp = max(1, w.prefix_group)
            max_prefixes = (w.batch + grp - 1) // grp + 1
    return make_config(
        num_layers=w.num_layers, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
        head_dim=w.head_dim, page_size=w.page_size,
        num_pages=num_pages or w.num_pages, max_requests=max_requests or w.batch,
        max_pages_per_req=max_pages_per_req or w.max_pages_per_req,
        dtype=GP_DTYPE_F32 if w.dtype == "f32" else GP_DTYPE_BF16, max_seq_len=seq,
        max_prefixes=max_prefixes, max_prefix_len=w.prefix_len, mode=mode,
        recent_window=w.recent_window, beta_s=w.beta_s, beta_l=w.beta_l, top_p=w.top_p,
        tau=w.tau, rope_theta=w.rope_theta, random_grow_rate=random_grow_rate)
