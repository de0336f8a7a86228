"""Scalar conventions of the oracle: RoPE, storage rounding, EMA summaries.

Test infrastructure only (see the package docstring).

Source: "GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning
Serving", evolve.pub review, Summary: two exponentially smoothed query
summaries with beta = 0.9 (short) and 0.999 (long), maintained pre-RoPE.
The FAQ section ("Is GrowPage's code available?") repeats beta_S = 0.9 and
beta_L = 0.999.
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------- RoPE ----

def rope_inv_freq(theta: float, d: int) -> list:
    """inv_freq_i = theta^(-2i/d), i < d/2, via the C library's pow().

    Reading: rotate-half RoPE (pairs (i, i + d/2)), the Llama / Qwen
    convention; the pages do not name a variant.
    """
    return [math.pow(theta, -(2.0 * i) / d) for i in range(d // 2)]


def rope_cos_sin(theta: float, d: int, pos: int):
    """fp64 cos / sin of pos * inv_freq_i (C library cos() and sin())."""
    inv = rope_inv_freq(theta, d)
    c = np.array([math.cos(float(pos) * f) for f in inv], dtype=np.float64)
    s = np.array([math.sin(float(pos) * f) for f in inv], dtype=np.float64)
    return c, s


class RopeTable:
    """Cache of fp64 (cos, sin) rows by position."""

    def __init__(self, theta: float, d: int):
        self.theta = float(theta)
        self.d = d
        self.rows = {}

    def __call__(self, pos: int):
        r = self.rows.get(pos)
        if r is None:
            r = rope_cos_sin(self.theta, self.d, pos)
            self.rows[pos] = r
        return r


def rope_apply(x: np.ndarray, table: RopeTable, pos: int) -> np.ndarray:
    """Rotate the last axis of x (fp64) to position pos.

    Each product and each sum is one fp64 operation (no fused multiply-add):
      y[i]       = x[i] * c_i - x[i + d/2] * s_i
      y[i + d/2] = x[i + d/2] * c_i + x[i] * s_i
    theta == 0 means no rotary embedding (identity).
    """
    x = np.asarray(x, dtype=np.float64)
    if table.theta == 0.0:
        return x.copy()
    c, s = table(pos)
    h = x.shape[-1] // 2
    a, b = x[..., :h], x[..., h:]
    y = np.empty_like(x)
    y[..., :h] = (a * c) - (b * s)
    y[..., h:] = (b * c) + (a * s)
    return y


# ------------------------------------------------------ storage rounding ----

def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values once, to nearest-even, onto the bfloat16 grid.

    bfloat16: 8 significant bits, exponent range of fp32 (normal numbers
    down to 2^-126, subnormal spacing 2^-133).  Returns the rounded values as
    fp64.  frexp / ldexp / rint are exact operations here.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = np.isfinite(x) & (x != 0.0)
    xm = x[nz]
    _, e = np.frexp(xm)                   # |x| = m * 2^e, 0.5 <= m < 1
    q = np.maximum(e - 8, -133)           # spacing of the bf16 grid at x
    r = np.ldexp(np.rint(np.ldexp(xm, -q)), q)
    big = np.abs(r) > float.fromhex("0x1.fep127")
    r[big] = np.copysign(np.inf, r[big])
    out[nz] = r
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


def round_f32(x: np.ndarray) -> np.ndarray:
    """Round fp64 values once, to nearest-even, to fp32 (returned as fp64)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    return round_bf16(x) if dtype == "bf16" else round_f32(x)


# ------------------------------------------------------------ summaries ----

def group_mean_f32(qg: np.ndarray) -> np.ndarray:
    """Mean of the G query heads of one kv head, in fp32.

    qg: [..., G, d].  Summed in head order, then divided by G (both fp32,
    one rounding each).  Reading: one summary per kv head, taken over the
    mean of its query heads.
    """
    qg = np.asarray(qg, dtype=np.float32)
    acc = qg[..., 0, :].copy()
    for h in range(1, qg.shape[-2]):
        acc = (acc + qg[..., h, :]).astype(np.float32)
    return (acc / np.float32(qg.shape[-2])).astype(np.float32)


def ema_fold(s: np.ndarray, qbar: np.ndarray, beta: float) -> np.ndarray:
    """One fp32 EMA step: s <- fl(fl(b * s) + fl(a * qbar)), a = fl(1 - b).

    b is beta rounded to fp32.  Reading: the first fold of a request sets
    s = qbar (no bias correction); the caller handles that case.
    """
    b = np.float32(beta)
    a = np.float32(np.float32(1.0) - b)
    s = np.asarray(s, dtype=np.float32)
    qbar = np.asarray(qbar, dtype=np.float32)
    return ((b * s).astype(np.float32) + (a * qbar).astype(np.float32)).astype(np.float32)
