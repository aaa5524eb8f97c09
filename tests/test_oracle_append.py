"""Pins of the oracle's append step (one new token per request): key codes
checked against E4M3 byte values fixed by the OCP FP8 specification, the
per-token scale, the lowest-free-slot insert, a full region and a full cache."""
import numpy as np
import pytest

D, RB = 128, 32          # key dims; a short KV row (bytes) for the pins


def _state(regions, C, B):
    off = np.concatenate([[0], np.cumsum(regions)]).astype(np.int64)
    n = int(off[-1])
    return dict(off=off, k8=np.zeros((n, D), np.uint8), ks=np.zeros(n, np.float32),
                host=np.zeros((n, RB), np.uint8), t2s=np.full(n, -1, np.int32),
                s2t=np.full(B * C, -1, np.int32), dev=np.zeros((B * C, RB), np.uint8))


def _append(orc, st, end, k, kv, C):
    return orc.append_tokens(st["off"], end, k, kv, st["k8"], st["ks"], st["host"], C, st["t2s"], st["s2t"],
                             st["dev"])


def test_key_codes_are_the_spec_bytes(orc):
    # amax = 448 gives scale 1; OCP E4M3: 448 = 0x7E, 224 = 0x76, 1 = 0x38, 0.5 = 0x30, 0 = 0x00,
    # the sign bit is 0x80
    st = _state([4], 32, 1)
    end = np.array([0], np.int64)
    k = np.zeros((1, D), np.float32)
    k[0, :5] = [448.0, -224.0, 1.0, 0.5, 0.0]
    kv = np.arange(RB, dtype=np.uint8)[None]
    full = _append(orc, st, end, k, kv, 32)
    assert full.tolist() == [0] and end.tolist() == [1]
    assert st["ks"][0] == np.float32(1.0)
    assert st["k8"][0, :5].tolist() == [0x7E, 0xF6, 0x38, 0x30, 0x00]
    assert not st["k8"][0, 5:].any()
    assert np.array_equal(st["host"][0], kv[0])


def test_scale_is_amax_over_448(orc):
    # amax 896: scale exactly 2, codes of 448 and 224; a tenth of it is not a power of two:
    # 89.6 / 448 = 0.2 in fp32, and 89.6 / 0.2 rounds to 448 in fp32
    st = _state([3], 32, 1)
    end = np.array([0], np.int64)
    k = np.zeros((2, D), np.float32)[:1]
    k[0, :2] = [896.0, -448.0]
    _append(orc, st, end, k, np.zeros((1, RB), np.uint8), 32)
    assert st["ks"][0] == np.float32(2.0) and st["k8"][0, :2].tolist() == [0x7E, 0xF6]
    k2 = np.zeros((1, D), np.float32)
    k2[0, 7] = np.float32(89.6)
    _append(orc, st, end, k2, np.zeros((1, RB), np.uint8), 32)
    assert st["ks"][1] == np.float32(89.6) / np.float32(448.0)
    assert st["k8"][1, 7] == 0x7E and not np.delete(st["k8"][1], 7).any()


def test_zero_key_has_zero_scale(orc):
    st = _state([2], 32, 1)
    end = np.array([0], np.int64)
    _append(orc, st, end, np.zeros((1, D), np.float32), np.ones((1, RB), np.uint8), 32)
    assert st["ks"][0] == 0.0 and not st["k8"][0].any()


def test_lowest_free_slot_and_full_cache(orc):
    C = 32
    st = _state([5, 5], C, 2)
    end = np.array([2, 7], np.int64)
    # request 0: slots 0, 1 and 3 taken -> the new token gets slot 2
    st["s2t"][[0, 1, 3]] = [0, 1, 4]
    st["t2s"][[0, 1, 4]] = [0, 1, 3]
    # request 1: every slot taken -> host only
    st["s2t"][C:2 * C] = 0
    kv = np.stack([np.full(RB, 7, np.uint8), np.full(RB, 9, np.uint8)])
    full = _append(orc, st, end, np.ones((2, D), np.float32), kv, C)
    assert full.tolist() == [0, 0] and end.tolist() == [3, 8]
    assert st["t2s"][2] == 2 and st["s2t"][2] == 2 and (st["dev"][2] == 7).all()
    assert st["t2s"][7] == -1 and (st["host"][7] == 9).all()
    assert not st["dev"][C:].any()


def test_full_region_changes_nothing(orc):
    st = _state([2, 3], 32, 2)
    end = np.array([2, 3], np.int64)          # request 0 full, request 1 has room
    before = {k: v.copy() for k, v in st.items()}
    full = _append(orc, st, end, np.ones((2, D), np.float32), np.full((2, RB), 5, np.uint8), 32)
    assert full.tolist() == [1, 0] and end.tolist() == [2, 4]
    assert np.array_equal(st["host"][:2], before["host"][:2]) and (st["host"][3] == 5).all()
    assert st["s2t"][32] == 1 and st["t2s"][3] == 0


def test_nonfinite_key_is_refused(orc):
    st = _state([2], 32, 1)
    end = np.array([0], np.int64)
    k = np.zeros((1, D), np.float32)
    k[0, 3] = np.inf
    with pytest.raises(Exception):
        _append(orc, st, end, k, np.zeros((1, RB), np.uint8), 32)
    assert end.tolist() == [0]
