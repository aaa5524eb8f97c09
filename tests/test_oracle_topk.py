"""Pins of the oracle's exact top-k, 256-bin histogram and EMA threshold (CPU only).

Top-k is pinned by brute force over all subsets (the defining property of the
exact top-k with ties to the lower index), by numpy's stable argsort (a
textbook routine), and by the degenerate cases.  The histogram is pinned by
hand-computed bins and by monotonicity; the EMA by its closed forms.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _is_topk(scores, subset):
    """The defining property: every chosen token beats every other token, where a
    tie goes to the lower index."""
    S = set(subset)
    for s in S:
        for t in range(len(scores)):
            if t in S:
                continue
            if not (scores[s] > scores[t] or (scores[s] == scores[t] and s < t)):
                return False
    return True


def test_brute_force_small(orc):
    rng = np.random.default_rng(0)
    for trial in range(60):
        n = int(rng.integers(1, 10))
        k = int(rng.integers(1, 12))
        scores = rng.integers(0, 4, n).astype(np.float32)        # many ties
        idx, kth = orc.topk(scores, k)
        take = min(k, n)
        chosen = [i for i in idx if i >= 0]
        assert len(chosen) == take and all(i == -1 for i in idx[take:])
        assert chosen == sorted(chosen)
        winners = [c for c in itertools.combinations(range(n), take) if _is_topk(scores, c)]
        assert winners == [tuple(chosen)]
        assert kth == min(scores[i] for i in chosen)


def test_matches_stable_argsort(orc):
    rng = np.random.default_rng(1)
    for n, k in [(1000, 37), (5000, 2048), (4096, 4096), (300, 1000)]:
        s = np.round(rng.standard_normal(n) * 8).astype(np.float32)
        idx, kth = orc.topk(s, k)
        order = np.argsort(-s, kind="stable")[:min(k, n)]
        assert np.array_equal(idx[:min(k, n)], np.sort(order))
        assert kth == s[order[-1]]


def test_all_equal_and_k_ge_n(orc):
    idx, kth = orc.topk(np.full(100, 3.5, np.float32), 10)
    assert list(idx) == list(range(10)) and kth == 3.5
    idx, kth = orc.topk(np.array([5, 1, 3], np.float32), 5)
    assert list(idx) == [0, 1, 2, -1, -1] and kth == 1.0
    idx, kth = orc.topk(np.zeros(0, np.float32), 4)
    assert list(idx) == [-1] * 4 and kth == -math.inf


def test_signed_zero_ties_and_nan(orc):
    s = np.array([-0.0, 0.0, -1.0, -0.0], np.float32)
    idx, kth = orc.topk(s, 2)
    assert list(idx) == [0, 1] and kth == 0.0 and math.copysign(1, kth) > 0
    with pytest.raises(orc.OracleError):
        orc.topk(np.array([1.0, np.nan], np.float32), 1)


def test_golden_topk():
    # hand-worked: tests/golden/topk_ties.json
    import oracle
    with open(os.path.join(GOLDEN, "topk_ties.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        idx, kth = oracle.topk(np.array(case["scores"], np.float32), case["k"])
        assert list(idx) == case["idx"], case
        assert kth == case["kth"]


def test_order_key(orc):
    assert orc.order_key(1.0) == 0xBF800000
    assert orc.order_key(-1.0) == 0x407FFFFF
    assert orc.order_key(0.0) == 0x80000000
    assert orc.order_key(-0.0) == 0x80000000
    assert orc.order_key(np.inf) == 0xFF800000
    assert orc.order_key(-np.inf) == 0x007FFFFF
    xs = np.sort(np.random.default_rng(2).standard_normal(2000).astype(np.float32))
    keys = [orc.order_key(float(x)) for x in xs]
    assert keys == sorted(keys)


def test_hist256_hand_bins(orc):
    # bin = top 8 bits of the order key of (score - shift)
    h = orc.hist256(np.array([1.0, -1.0, 0.0, 5.0, 2.0, 3.0], np.float32), 0.0)
    assert h[0xBF] == 1           # 1.0: exponent 127 -> 0x3F8..., key 0xBF8...
    assert h[0x40] == 1           # -1.0
    assert h[0x80] == 1           # 0.0
    assert h[0xC0] == 3           # 2.0, 3.0 and 5.0 share exponent-pair bin 0x40|0x80
    assert h.sum() == 6
    h = orc.hist256(np.array([5.0, 4.0, 3.0], np.float32), 4.0)
    assert h[0xBF] == 1 and h[0x80] == 1 and h[0x40] == 1
    # no prediction yet (theta = +inf): unshifted
    assert np.array_equal(orc.hist256(np.array([1.0], np.float32), np.inf),
                          orc.hist256(np.array([1.0], np.float32), 0.0))


def test_hist256_monotone_and_total(orc):
    rng = np.random.default_rng(3)
    s = np.sort(rng.standard_normal(5000).astype(np.float32) * 50 + 100)
    theta = np.float32(130.0)
    h = orc.hist256(s, theta)
    assert h.sum() == s.size
    bins = np.array([orc.order_key(float(np.float32(x - theta))) >> 24 for x in s])
    assert np.all(np.diff(bins) >= 0)                             # monotone in the score
    assert np.array_equal(np.bincount(bins, minlength=256), h)


def test_ema_closed_forms(orc):
    # constant k-th score: the prediction equals it from the second step on
    th = np.inf
    for t in range(6):
        th = orc.ema(th, 12.5, 0.5)
        assert th == 12.5
    # after a jump to 0 the prediction halves each step: theta_t = 12.5 * 2^-t
    for t in range(1, 12):
        th = orc.ema(th, 0.0, 0.5)
        assert th == 12.5 * 2.0 ** -t
    # general alpha: alpha*x + (1-alpha)*th, each operation rounded in fp32
    a = np.float32(0.3)
    got = orc.ema(np.float32(7.0), np.float32(3.0), a)
    want = np.float32(np.float32(a * np.float32(3.0)) + np.float32(np.float32(np.float32(1) - a) * np.float32(7.0)))
    assert got == want
    assert orc.ema(5.0, -np.inf, 0.5) == 5.0                      # empty request keeps theta
