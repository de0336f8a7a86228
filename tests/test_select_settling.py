"""The boundary selects' radix passes, restated on the host, against their definitions.

The boundary select kernel counts each summary's Top-p working set ("GrowPage:
On-Demand KV Budgeting for Efficient LLM Reasoning Serving", evolve.pub review,
section "Summary": Top-p attention working sets of the two query summaries) on
fixed-point masses: every weight e_j in [0, 1] (fp32) becomes round(e_j * 2^40),
the threshold is ceil(top_p * total), and W is the smallest count of the largest
weights whose mass reaches it.  The kernel finds W by a most-significant-first
radix select over the fp32 bit patterns, 8 bits a pass, and settles a summary
as soon as the digit it picks holds a single element.

This file restates those steps in exact integer arithmetic and checks, on rows
chosen to settle at every pass, to tie at the threshold and to hold zeros, that
(1) the select with settling gives the same W as the select that always runs
all four passes, and (2) both equal the definition computed by sorting.  The
compaction select is restated the same way at the end of the file.  The GPU
parity tests compare the kernels themselves with the fp64 oracle.
"""
from fractions import Fraction
from math import ceil

import numpy as np
import pytest

FIX = 2 ** 40


def mass_q(e32: np.ndarray) -> np.ndarray:
    """round(e * 2^40), ties to even; exact, since e * 2^40 is exact in fp64."""
    return np.rint(e32.astype(np.float64) * FIX).astype(np.int64)


def threshold(top_p: np.float32, total: int) -> int:
    """ceil(top_p * total) for the fp32 value top_p, exactly."""
    return ceil(Fraction(float(top_p)) * total)


def topp_by_sorting(e32: np.ndarray, top_p: np.float32) -> int:
    """Smallest k whose k largest weights carry at least the threshold mass."""
    mq = mass_q(e32)
    thr = threshold(top_p, int(mq.sum()))
    if thr <= 0:
        return 1
    cs = np.cumsum(np.sort(mq)[::-1])
    return int(np.searchsorted(cs, thr, side="left")) + 1


def topp_radix(e32: np.ndarray, top_p: np.float32, settle: bool):
    """The kernel's select: four 8-bit passes from the top byte of the fp32
    bit pattern.  Each pass histograms (count, mass) over the digits of the
    elements that match the prefix picked so far, and picks, from the top
    digit down, the first digit at which the mass above it plus its own
    reaches the mass still needed.  With `settle`, a picked digit holding one
    element ends the select: W = (elements above it) + 1.  Returns (W, the
    pass that settled it or None)."""
    bits = e32.view(np.uint32).astype(np.int64)
    mq = mass_q(e32)
    thr = threshold(top_p, int(mq.sum()))
    prefix, pmask = 0, 0
    mass_above, cnt_above = 0, 0
    for p in range(4):
        shift = 24 - 8 * p
        inb = (bits & pmask) == prefix
        dig = (bits[inb] >> shift) & 255
        cnt = np.bincount(dig, minlength=256)
        mass = np.zeros(256, dtype=np.int64)
        np.add.at(mass, dig, mq[inb])
        need = thr - mass_above
        acc_m, acc_c, pick = 0, 0, None
        for d in range(255, -1, -1):
            if acc_m < need <= acc_m + int(mass[d]):
                pick = d
                break
            acc_m += int(mass[d])
            acc_c += int(cnt[d])
        if pick is None:        # nothing reaches the mass still needed
            pick, acc_m, acc_c = 0, 0, 0
        prefix |= pick << shift
        pmask |= 255 << shift
        mass_above += acc_m
        cnt_above += acc_c
        if settle and cnt[pick] == 1:
            return cnt_above + 1, p
    qstar = int(mass_q(np.array([prefix], dtype=np.uint32).view(np.float32))[0])
    rest = max(thr - mass_above, 0)
    k = -(-rest // qstar) if qstar else 1
    return cnt_above + (k if k else 1), None


def _rows(rng):
    """Rows of fp32 weights in [0, 1] with the largest equal to 1, as the
    kernel forms them (e_j = exp(u_j - max))."""
    out = []
    for n in (1, 2, 3, 17, 255, 1000, 1320, 4096):
        u = rng.standard_normal(n) * rng.choice([0.5, 2.0, 6.0])
        out.append(np.exp(u - u.max()).astype(np.float32))
    # ties: weights drawn from a few values, so the threshold falls inside a
    # run of equal weights
    for n in (8, 100, 2000):
        vals = np.array([1.0, 0.5, 0.25, 0.125, 3e-3], dtype=np.float32)
        out.append(rng.choice(vals, n).astype(np.float32))
    # one dominant weight (settles in the first pass), and weights that share
    # their top one, two and three bytes with the threshold element
    out.append(np.concatenate([[1.0], np.full(500, 1e-9)]).astype(np.float32))
    base = np.float32(0.375).view(np.uint32)
    for keep in (8, 16, 24):
        lo = rng.integers(0, 1 << (32 - keep), 64, dtype=np.uint64).astype(np.uint32)
        same = ((base >> (32 - keep)) << (32 - keep)) | (lo & ((1 << (32 - keep)) - 1))
        out.append(np.concatenate([[np.float32(1.0)], same.view(np.float32)]).astype(np.float32))
    # zeros and subnormals next to normal weights
    z = np.zeros(300, dtype=np.float32)
    z[:5] = [1.0, 0.3, 1e-40, 0.0, 2e-38]
    out.append(z)
    return out


TOP_PS = [np.float32(x) for x in (1.0, 0.99, 0.9, 0.5, 0.05, 1e-6)]


def test_settling_matches_full_passes_and_the_definition():
    rng = np.random.default_rng(20261203)
    passes = []
    for e in _rows(rng):
        for tp in TOP_PS:
            want = topp_by_sorting(e, tp)
            full, _ = topp_radix(e, tp, settle=False)
            fast, at = topp_radix(e, tp, settle=True)
            assert full == want, (len(e), float(tp), full, want)
            assert fast == want, (len(e), float(tp), fast, want)
            passes.append(at)
    # the rule is exercised: rows settle before the last pass, and some rows
    # (ties at the threshold) run all four passes without settling
    assert sum(1 for a in passes if a is not None and a < 3) > len(passes) // 4
    assert any(a is None for a in passes)


@pytest.mark.parametrize("p", [0, 1, 2, 3])
def test_settling_at_each_pass(p):
    # weights 1.0, a, b where a and b share their first p bytes and differ at
    # byte p (a the larger); the threshold falls inside a's mass, so W = 2 and
    # a is alone in its digit first at pass p.  For p = 0 the set needs 1.0
    # only, alone in its top byte.
    if p == 0:
        e = np.array([1.0, 1e-3], dtype=np.float32)
        tp = np.float32(0.5)
        want = 1
    else:
        base = 0x3F400000  # 0.75
        shift = 24 - 8 * p
        clear = base & ~(0xFF << shift)
        a = np.uint32(clear | (0x20 << shift)).view(np.float32)
        b = np.uint32(clear | (0x10 << shift)).view(np.float32)
        e = np.array([1.0, a, b], dtype=np.float32)
        mq = mass_q(e).astype(np.float64)
        tp = np.float32((mq[0] + mq[1] / 2) / mq.sum())
        want = 2
    w, at = topp_radix(e, tp, settle=True)
    assert (w, at) == (want, p)
    assert topp_by_sorting(e, tp) == want
    assert topp_radix(e, tp, settle=False)[0] == want


def test_single_weight_and_all_zero_rows():
    one = np.array([1.0], dtype=np.float32)
    zeros = np.zeros(7, dtype=np.float32)
    for tp in TOP_PS:
        assert topp_radix(one, tp, settle=True)[0] == topp_by_sorting(one, tp) == 1
        assert topp_radix(zeros, tp, settle=True)[0] == 1
        assert topp_radix(zeros, tp, settle=False)[0] == 1


# ---- the compaction select ------------------------------------------------
#
# The compaction plan drops the k lowest candidates by the 64-bit key
# (importance bits << 32 | position), importance = max(p_S, p_L) of a private
# token older than the recent window ("GrowPage: On-Demand KV Budgeting for
# Efficient LLM Reasoning Serving", evolve.pub review, section "Summary":
# compaction ranks history by the maximum of both importance scores).  The
# kernel finds a threshold key with exactly k candidates at or below it by an
# 8-bit radix select from the top byte, and stops as soon as the digit it
# picks is taken whole (the threshold is then that prefix with all lower bits
# set).  Keys are distinct: they end with the token position.


def kth_smallest_radix(keys, k):
    """The kernel's select over candidate keys (Python ints < 2^64)."""
    prefix, pmask, below = 0, 0, 0
    for p in range(8):
        shift = 56 - 8 * p
        cnt = [0] * 256
        for x in keys:
            if x & pmask == prefix:
                cnt[(x >> shift) & 255] += 1
        acc, pick = below, None
        for d in range(256):
            if acc + cnt[d] >= k:
                pick = d
                break
            acc += cnt[d]
        if pick is None:            # fewer than k candidates: the scan ends on 255
            pick, acc = 255, acc - cnt[255]
        prefix |= pick << shift
        pmask |= 255 << shift
        below = acc
        if acc + cnt[pick] == k:    # the picked digit is taken whole
            return prefix | ((1 << shift) - 1)
    return prefix


def _compaction_keys(rng, n, ties):
    imp = rng.random(n).astype(np.float32)
    if ties:                        # few distinct importances: ties broken by position
        imp = rng.choice(imp[:4], n)
    bits = imp.view(np.uint32).astype(np.uint64)
    pos = rng.permutation(1 << 20)[:n].astype(np.uint64)
    return [int(b) << 32 | int(q) for b, q in zip(bits, pos)]


@pytest.mark.parametrize("n,k,ties", [(16, 16, False), (40, 16, False), (1000, 16, False),
                                      (1000, 16, True), (3000, 32, True), (17, 1, False),
                                      (256, 255, True)])
def test_compaction_select_takes_exactly_the_k_lowest(n, k, ties):
    rng = np.random.default_rng(n * 7 + k + ties)
    keys = _compaction_keys(rng, n, ties)
    thr = kth_smallest_radix(keys, k)
    chosen = sorted(x for x in keys if x <= thr)
    assert chosen == sorted(keys)[:k]


def test_compaction_select_stops_early_on_a_whole_digit():
    # the k lowest keys share a top byte that no other key has: the select
    # stops after the first pass with every lower bit of the threshold set
    low = [(0x10 << 56) | i for i in range(16)]
    high = [(0x20 << 56) | i for i in range(100)]
    thr = kth_smallest_radix(low + high, 16)
    assert thr == (0x10 << 56) | ((1 << 56) - 1)
    assert sorted(x for x in low + high if x <= thr) == low
