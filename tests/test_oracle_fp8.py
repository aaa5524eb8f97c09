"""Pins of the oracle's E4M3 codec and query quantisation (CPU only).

The E4M3 format is fixed by the OCP 8-bit floating point specification; the
checks below pin the oracle to values that follow from that definition by
hand, and to torch's own float8_e4m3fn conversion (an independent library
routine) on the in-range values where the two definitions coincide.
"""
import math

import numpy as np
import pytest
import torch


def test_decode_table_hand_values(orc):
    # sign / exponent (bias 7) / mantissa, worked by hand from the definition
    assert orc.e4m3_decode(0x00) == 0.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9          # smallest subnormal: 1/8 * 2^-6
    assert orc.e4m3_decode(0x07) == 7 / 8 * 2.0 ** -6  # largest subnormal
    assert orc.e4m3_decode(0x08) == 2.0 ** -6          # smallest normal
    assert orc.e4m3_decode(0x38) == 1.0                # e=7 -> 2^0
    assert orc.e4m3_decode(0x3C) == 1.5
    assert orc.e4m3_decode(0x7E) == 448.0              # largest finite: 1.75 * 2^8
    assert math.isnan(orc.e4m3_decode(0x7F))
    assert math.isnan(orc.e4m3_decode(0xFF))
    assert orc.e4m3_decode(0xB8) == -1.0
    v = orc.e4m3_decode(0x80)
    assert v == 0.0 and math.copysign(1.0, v) < 0


def test_decode_table_matches_torch(orc):
    tab = orc.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(tab))
    assert np.array_equal(tab[~nan], ref[~nan])
    assert nan.sum() == 2


@pytest.mark.parametrize("x,code", [
    (1.0, 0x38), (448.0, 0x7E), (2.0 ** -9, 0x01),
    (2.0 ** -10, 0x00),            # half the smallest subnormal: tie -> even code 0
    (3 * 2.0 ** -10, 0x02),        # halfway between codes 1 and 2 -> even code 2
    (1.0625, 0x38),                # halfway between 1.0 (0x38) and 1.125 (0x39) -> 0x38
    (1.1875, 0x3A),                # halfway between 1.125 (0x39) and 1.25 (0x3A) -> 0x3A
    (1.06, 0x38), (1.07, 0x39),
    (464.0, 0x7E), (1e6, 0x7E),    # saturating
    (-1.0, 0xB8), (-0.0, 0x80), (-1e-30, 0x80),
    (240.0, 0x77), (232.0, 0x76),  # 232 is halfway between 224 (0x76) and 240 (0x77) -> even
])
def test_encode_hand_values(orc, x, code):
    assert orc.e4m3_encode(np.array([x], np.float32))[0] == code


def test_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(1)
    # every bit pattern of a few binades across the format's range, plus random values
    parts = []
    for e in range(-12, 9):
        m = np.arange(0, 1 << 23, 97, dtype=np.uint32)
        bits = (np.uint32(e + 127) << np.uint32(23)) | m
        parts.append(bits.view(np.float32))
    parts.append(rng.uniform(-448, 448, 200_000).astype(np.float32))
    x = np.concatenate(parts)
    x = np.concatenate([x, -x])
    x = x[np.abs(x) <= 448]
    got = orc.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_encode_is_nearest_brute_force(orc):
    # nearest value by exhaustive search over all finite codes, ties -> even code
    tab = orc.e4m3_table()
    finite = [c for c in range(256) if not math.isnan(tab[c])]
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.uniform(-450, 450, 3000), rng.uniform(-0.02, 0.02, 3000)]).astype(np.float32)
    got = orc.e4m3_encode(xs)
    for x, g in zip(xs.astype(np.float64), got):
        a = min(abs(x), 448.0)
        best = min(finite, key=lambda c: (abs(abs(tab[c]) - a), c & 1, c))
        sign = 0x80 if math.copysign(1.0, x) < 0 else 0
        assert g == ((best & 0x7F) | sign), (x, g, best)


def test_q_scale_closed_forms(orc):
    # scale = smallest power of two p with amax <= 448 p
    cases = [(448.0, 1.0), (448.00006, 2.0), (1.0, 2.0 ** -8), (1.75, 2.0 ** -8),
             (1.7500001, 2.0 ** -7), (0.0, 1.0), (3.0, 2.0 ** -7), (1e-40, 2.0 ** -126),
             (896.0, 2.0), (896.0001, 4.0)]
    for amax, want in cases:
        q = np.zeros((1, 1, 128), np.float32)
        q[0, 0, 5] = np.float32(amax)
        q[0, 0, 6] = -np.float32(amax) / 2
        q8, qs, wf = orc.quantize_q(q, np.array([[0.75]], np.float32))
        assert qs[0, 0] == np.float32(want), (amax, qs[0, 0], want)
        assert wf[0, 0] == np.float32(0.75 * want)
        if want > 2.0 ** -126:  # unclamped: the largest element keeps 3 mantissa bits
            assert abs(orc.e4m3_decode(q8[0, 0, 5]) * want - np.float32(amax)) <= np.float32(amax) / 16


def test_quantize_is_encode_of_exact_division(orc):
    rng = np.random.default_rng(3)
    q = rng.standard_normal((3, 64, 128)).astype(np.float32) * np.float32(7.5)
    w = rng.uniform(0, 1, (3, 64)).astype(np.float32)
    q8, qs, wf = orc.quantize_q(q, w)
    for b in range(3):
        for h in range(64):
            s = qs[b, h]
            m, e = math.frexp(float(s))
            assert m == 0.5                                   # a power of two
            amax = np.abs(q[b, h]).max()
            assert amax <= 448 * s and amax > 448 * s / 2     # the smallest such
            ref = orc.e4m3_encode((q[b, h].astype(np.float64) / s).astype(np.float32))
            assert np.array_equal(q8[b, h], ref)
            # no code saturates, and the largest element lands in the top binade
            assert np.abs(q8[b, h].view(np.int8) & 0x7F).max() >= 0x70


def test_quantize_rejects_nan(orc):
    q = np.zeros((1, 64, 128), np.float32)
    q[0, 3, 3] = np.nan
    with pytest.raises(orc.OracleError):
        orc.quantize_q(q, np.ones((1, 64), np.float32))
    q[0, 3, 3] = np.inf
    with pytest.raises(orc.OracleError):
        orc.quantize_q(q, np.ones((1, 64), np.float32))
