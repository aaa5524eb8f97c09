"""Pins of the oracle's sparse MLA decode attention (CPU only).

The attention over the selected slots is pinned by closed forms that do not
retype its formula: one valid token gives back its row; equal scores give the
plain mean of the rows; two tokens with a score gap g weigh their rows by the
logistic of g; large scores stay finite; the order of the slots does not
matter; no valid slot gives zeros and -inf.
"""
import math

import numpy as np
import pytest

H, D, DV = 4, 576, 512


def bf16_bits(x):
    """bf16 bit patterns of float32 values that bf16 holds exactly."""
    b = (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32), np.asarray(x, np.float32))
    return b


def bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def random_rows(rng, n):
    # small dyadic values: exact in bf16
    return bf16_bits(rng.integers(-64, 65, (n, D)) / 16.0)


def test_bf16_decode(orc):
    assert orc.bf16_value(0x3F80) == 1.0 and orc.bf16_value(0xC020) == -2.5
    assert orc.bf16_value(0x0000) == 0.0 and orc.bf16_value(0x3E80) == 0.25
    assert math.isinf(orc.bf16_value(0x7F80))


def test_one_valid_token_returns_its_row(orc):
    rng = np.random.default_rng(0)
    kv = random_rows(rng, 10)
    q = random_rows(rng, H)
    slots = np.array([-1, 7, -1, -1], np.int32)
    out, lse, _ = orc.mla_decode(q, kv, slots, 0.125)
    assert np.array_equal(out, np.broadcast_to(bf16_values(kv[7, :DV]), (H, DV)))
    s = 0.125 * (bf16_values(q) @ bf16_values(kv[7]))
    assert np.allclose(lse, s, rtol=0, atol=1e-12)


def test_zero_query_gives_the_mean(orc):
    rng = np.random.default_rng(1)
    kv = random_rows(rng, 20)
    q = np.zeros((H, D), np.uint16)
    slots = np.array([3, 9, 11, -1, 17], np.int32)
    out, lse, _ = orc.mla_decode(q, kv, slots, 1.0)
    want = bf16_values(kv[[3, 9, 11, 17], :DV]).mean(0)
    assert np.allclose(out, np.broadcast_to(want, (H, DV)), rtol=0, atol=1e-12)
    assert np.allclose(lse, math.log(4), rtol=0, atol=1e-12)


@pytest.mark.parametrize("gap", [0.0, 1.5, -3.0, 40.0])
def test_two_tokens_logistic_weights(orc, gap):
    # q has one nonzero dimension (5); the two rows hold -gap/2 and +gap/2 there
    rng = np.random.default_rng(2)
    kv = random_rows(rng, 4).copy()
    kv[:, 5] = bf16_bits([0.0, 0.0, 0.0, 0.0])
    kv[2, 5] = bf16_bits([gap / 2.0])[0]
    kv[1, 5] = bf16_bits([-gap / 2.0])[0]
    q = np.zeros((H, D), np.uint16)
    q[:, 5] = bf16_bits([1.0])[0]
    out, lse, _ = orc.mla_decode(q, kv, np.array([1, 2], np.int32), 1.0)
    p2 = 1.0 / (1.0 + math.exp(-gap))
    want = (1 - p2) * bf16_values(kv[1, :DV]) + p2 * bf16_values(kv[2, :DV])
    assert np.allclose(out, np.broadcast_to(want, (H, DV)), rtol=0, atol=1e-12)
    assert np.allclose(lse, -gap / 2 + math.log1p(math.exp(gap)) if gap < 30 else gap / 2, rtol=0, atol=1e-9)


def test_large_scores_stay_finite(orc):
    rng = np.random.default_rng(3)
    kv = random_rows(rng, 6)
    q = bf16_bits(np.full((H, D), 2.0))
    out, lse, mass = orc.mla_decode(q, kv, np.arange(6, dtype=np.int32), 50.0)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse)) and np.all(np.isfinite(mass))
    # the best-scoring token dominates: its row within the other tokens' share
    s = bf16_values(kv).sum(1)
    best = int(np.argmax(s))
    assert np.allclose(out[0], bf16_values(kv[best, :DV]), atol=1e-6)


def test_slot_order_does_not_matter(orc):
    rng = np.random.default_rng(4)
    kv = random_rows(rng, 50)
    q = random_rows(rng, H)
    slots = rng.permutation(50)[:20].astype(np.int32)
    a = orc.mla_decode(q, kv, slots, 0.05)
    b = orc.mla_decode(q, kv, slots[::-1].copy(), 0.05)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-12, atol=1e-12)
    assert np.all(a[2] >= np.abs(a[0]) - 1e-12)           # mass bounds the output


def test_no_valid_slot(orc):
    kv = np.zeros((3, D), np.uint16)
    q = np.zeros((H, D), np.uint16)
    out, lse, _ = orc.mla_decode(q, kv, np.array([-1, -1], np.int32), 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    with pytest.raises(orc.OracleError):
        orc.mla_decode(q, kv, np.array([3], np.int32), 1.0)   # slot beyond the rows
