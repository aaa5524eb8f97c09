"""Pins of the oracle's fp64 indexer score (CPU only).

I[s] = sum_h w[h] * ReLU(q[h] . k[s]) over dequantised E4M3 values.  Each check
below is a special case whose value follows from the definition without the
oracle: exact integer arithmetic, one head (a plain dot product), a zero
query, sign flips that the ReLU must cut, and exact power-of-two scaling.
"""
import numpy as np
import pytest

H, D = 64, 128


def _codes_for_ints(orc, vals):
    """E4M3 codes of small integers (exactly representable)."""
    tab = orc.e4m3_table()
    lut = {}
    for c in range(256):
        v = tab[c]
        if not np.isnan(v) and float(v).is_integer() and (v not in lut or c < 128):
            lut[v] = c
    return np.vectorize(lambda v: lut[float(v)])(vals).astype(np.uint8)


def test_integer_exact_construction(orc):
    rng = np.random.default_rng(0)
    n = 40
    qi = rng.integers(-4, 5, (H, D))
    ki = rng.integers(-4, 5, (n, D))
    q8 = _codes_for_ints(orc, qi)
    k8 = _codes_for_ints(orc, ki)
    qs = (2.0 ** rng.integers(-3, 3, H)).astype(np.float32)
    ks = (2.0 ** rng.integers(-2, 2, n)).astype(np.float32)
    w = (rng.integers(0, 9, H) / 8.0).astype(np.float32)          # dyadic weights
    got, _ = orc.scores(q8, qs, w, k8, ks)
    dots = ki.astype(np.int64) @ qi.astype(np.int64).T              # [n, H] exact integers
    # every term is a dyadic rational; summing them in fp64 is exact here
    want = (np.maximum(dots, 0) * (qs.astype(np.float64) * w)[None, :]).sum(1) * ks
    assert np.array_equal(got, want)


def test_one_head_is_a_dot_product(orc):
    rng = np.random.default_rng(1)
    n = 64
    q8 = rng.integers(0, 256, (1, D)).astype(np.uint8)
    q8[(q8 & 0x7F) == 0x7F] = 0x38                                  # no NaN codes
    k8 = rng.integers(0, 256, (n, D)).astype(np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x30
    tab = orc.e4m3_table()
    qs = np.array([0.25], np.float32)
    ks = rng.uniform(0.5, 2.0, n).astype(np.float32)
    got, ab = orc.scores(q8, qs, np.array([1.0], np.float32), k8, ks)
    qv = tab[q8[0]] * 0.25
    for s in range(n):
        dot = float(np.dot(qv, tab[k8[s]] * float(ks[s])))
        assert got[s] == pytest.approx(max(dot, 0.0), rel=1e-12, abs=1e-12)
        assert ab[s] == pytest.approx(float(np.abs(qv * tab[k8[s]] * float(ks[s])).sum()), rel=1e-12)


def test_zero_query_scores_zero(orc):
    rng = np.random.default_rng(2)
    k8 = rng.integers(0, 0x7E, (32, D)).astype(np.uint8)
    got, ab = orc.scores(np.zeros((H, D), np.uint8), np.ones(H, np.float32),
                         np.ones(H, np.float32), k8, np.ones(32, np.float32))
    assert np.all(got == 0.0) and np.all(ab == 0.0)


def test_relu_cuts_negative_heads(orc):
    # head h sees k = +q for even h (positive dot) and the negation for odd h
    rng = np.random.default_rng(3)
    base = _codes_for_ints(orc, rng.integers(1, 4, D))
    q8 = np.tile(base, (H, 1))
    q8[1::2] ^= 0x80                                               # odd heads: -q
    k8 = base[None, :].copy()
    w = np.ones(H, np.float32)
    got, _ = orc.scores(q8, np.ones(H, np.float32), w, k8, np.ones(1, np.float32))
    tab = orc.e4m3_table()
    per_head = float((tab[base] ** 2).sum())
    assert got[0] == per_head * (H // 2)                            # only the even heads count
    # one-hot weight on an odd head gives exactly zero
    w1 = np.zeros(H, np.float32)
    w1[5] = 1.0
    got1, _ = orc.scores(q8, np.ones(H, np.float32), w1, k8, np.ones(1, np.float32))
    assert got1[0] == 0.0
    w1[:] = 0
    w1[4] = 1.0
    got2, _ = orc.scores(q8, np.ones(H, np.float32), w1, k8, np.ones(1, np.float32))
    assert got2[0] == per_head


def test_scales_are_exact_factors(orc):
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, H, D)).astype(np.float32)
    w = rng.uniform(0, 1, (1, H)).astype(np.float32)
    q8, qs, _ = orc.quantize_q(q, w)
    k8 = rng.integers(0, 0x7E, (16, D)).astype(np.uint8) | (rng.integers(0, 2, (16, D)) << 7).astype(np.uint8)
    ks = rng.uniform(0.1, 1.0, 16).astype(np.float32)
    a, _ = orc.scores(q8[0], qs[0], w[0], k8, ks)
    b, _ = orc.scores(q8[0], qs[0], w[0], k8, ks * np.float32(4.0))
    c, _ = orc.scores(q8[0], qs[0] * np.float32(0.5), w[0], k8, ks)
    assert np.array_equal(b, a * 4.0)
    assert np.array_equal(c, a * 0.5)


def test_token_subset_matches_full(orc):
    rng = np.random.default_rng(5)
    k8 = rng.integers(0, 0x7E, (50, D)).astype(np.uint8)
    ks = rng.uniform(0.1, 1.0, 50).astype(np.float32)
    q = rng.standard_normal((1, H, D)).astype(np.float32)
    w = rng.uniform(0, 1, (1, H)).astype(np.float32)
    q8, qs, _ = orc.quantize_q(q, w)
    full, _ = orc.scores(q8[0], qs[0], w[0], k8, ks)
    tok = np.array([49, 0, 7, 7, 31], np.int64)
    sub, _ = orc.scores(q8[0], qs[0], w[0], k8, ks, tok=tok)
    assert np.array_equal(sub, full[tok])
