"""Pins of the oracle's GPU-cache step, early fetch, recall and prefill rows (CPU only).

The cache step is pinned by a hand-worked walkthrough (tests/golden), by the
invariants the explainer page states (the selected set is resident after the
step, the two tables are inverses, nothing is written back) and by its
special cases (disjoint selections miss entirely and reuse the lowest slots;
identical selections move nothing).
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_walkthrough(orc):
    with open(os.path.join(GOLDEN, "cache_walkthrough.json")) as f:
        g = json.load(f)
    t2s = np.full(g["N"], -1, np.int32)
    s2t = np.full(g["C"], -1, np.int32)
    for st in g["steps"]:
        et = None
        if "early" in st:
            e = st["early"]
            et, es = orc.early_fetch(np.array(e["scores"], np.float32), e["theta"], e["cap"], t2s, s2t)
            assert list(et) == e["early_tok"] and list(es) == e["early_slot"], st["why"]
        sel_slot, mt, ms, nf = orc.cache_step(np.array(st["sel"], np.int32), t2s, s2t, early_tok=et,
                                              hold_early=st.get("hold_early", False))
        assert list(sel_slot) == st["sel_slot"], st["why"]
        assert list(mt) == st["miss_tok"] and list(ms) == st["miss_slot"], st["why"]
        assert nf == st["nfreed"], st["why"]
        assert list(t2s) == st["tok2slot"] and list(s2t) == st["slot2tok"], st["why"]


def _check_invariants(t2s, s2t, sel):
    sel = [s for s in sel if s >= 0]
    res = {s for s in range(t2s.size) if t2s[s] >= 0}
    assert res == set(sel)                                   # resident == selected
    for s in res:
        assert s2t[t2s[s]] == s                              # tables are inverses
    for j in range(s2t.size):
        if s2t[j] >= 0:
            assert t2s[s2t[j]] == j


def test_random_sequences_invariants(orc):
    rng = np.random.default_rng(0)
    for trial in range(20):
        n = int(rng.integers(20, 200))
        k = int(rng.integers(1, 20))
        C = int(rng.integers(k, 3 * k + 2))
        t2s = np.full(n, -1, np.int32)
        s2t = np.full(C, -1, np.int32)
        host = rng.integers(0, 256, (n, 32)).astype(np.uint8)
        host0 = host.copy()
        dev = np.zeros((C, 32), np.uint8)

        for step in range(12):
            if rng.random() < 0.5 and step:
                e_scores = rng.standard_normal(n).astype(np.float32)
                cap = int(rng.integers(-1, C + 1))
                et, es = orc.early_fetch(e_scores, 0.5, cap, t2s, s2t)
                assert list(et) == sorted(et) and list(es) == sorted(es)
                orc.recall(host, et, es, dev)
            sel = np.sort(rng.choice(n, min(k, n), replace=False)).astype(np.int32)
            res_before = {s for s in range(n) if t2s[s] >= 0}
            sel_slot, mt, ms, nf = orc.cache_step(sel, t2s, s2t)
            orc.recall(host, mt, ms, dev)
            _check_invariants(t2s, s2t, sel)
            assert set(mt) == set(sel) - res_before               # misses = selected \ resident
            assert nf == len(res_before - set(sel))
            assert list(mt) == sorted(mt)
            for s, j in zip(sel, sel_slot):
                assert t2s[s] == j
                assert np.array_equal(dev[j], host[s])           # cached bytes == host bytes
            assert np.array_equal(host, host0)                   # no write-back



def test_disjoint_with_c_equal_k(orc):
    n, k = 64, 8
    t2s = np.full(n, -1, np.int32)
    s2t = np.full(k, -1, np.int32)
    for step in range(n // k):
        sel = np.arange(step * k, (step + 1) * k, dtype=np.int32)
        sel_slot, mt, ms, nf = orc.cache_step(sel, t2s, s2t)
        assert list(mt) == list(sel) and list(ms) == list(range(k))
        assert nf == (k if step else 0)


def test_capacity_error_leaves_state(orc):
    t2s = np.full(10, -1, np.int32)
    s2t = np.full(2, -1, np.int32)
    with pytest.raises(orc.OracleError):
        orc.cache_step(np.array([1, 2, 3], np.int32), t2s, s2t)
    assert np.all(t2s == -1) and np.all(s2t == -1)


def test_held_early_slots_count_against_capacity(orc):
    """Held-slot variant: selected tokens plus the held slots of unselected early tokens must fit
    in C; the early cap C - k of a decode step guarantees it (the early set leaves room for k
    misses).  Under the contract reading the same step fits: the miss reuses a freed early slot."""
    t2s = np.full(10, -1, np.int32)
    s2t = np.full(3, -1, np.int32)
    et, es = orc.early_fetch(np.array([0, 0, 0, 0, 0, 0, 0, 2.0, 2.0, 0], np.float32), 1.0, -1, t2s, s2t)
    assert list(et) == [7, 8] and list(es) == [0, 1]
    before = (t2s.copy(), s2t.copy())
    with pytest.raises(orc.OracleError):                     # 2 selected + 2 held > 3
        orc.cache_step(np.array([1, 2], np.int32), t2s, s2t, early_tok=et, hold_early=True)
    assert np.array_equal(t2s, before[0]) and np.array_equal(s2t, before[1])
    t2s_c, s2t_c = t2s.copy(), s2t.copy()
    sel_slot, mt, ms, nf = orc.cache_step(np.array([2, 7], np.int32), t2s, s2t, early_tok=et, hold_early=True)
    assert list(sel_slot) == [2, 0] and list(mt) == [2] and list(ms) == [2] and nf == 1
    assert list(s2t) == [7, -1, 2]                           # slot 1 (held for 8) is free again
    # contract reading: 8 is freed at once and the miss 2 takes the lowest free slot, 1
    sel_slot, mt, ms, nf = orc.cache_step(np.array([2, 7], np.int32), t2s_c, s2t_c, early_tok=et)
    assert list(sel_slot) == [1, 0] and list(mt) == [2] and list(ms) == [1] and nf == 1
    assert list(s2t_c) == [7, 2, -1]
    assert [orc.early_cap_for(c, 4096, 2048) for c in (-1, 0, 100, 2048, 5000)] == [2048, 0, 100, 2048, 2048]
    assert orc.early_cap_for(-1, 64, 64) == 0


def test_early_fetch_strict_and_inf(orc):
    t2s = np.full(4, -1, np.int32)
    s2t = np.full(4, -1, np.int32)
    et, _ = orc.early_fetch(np.array([1.0, 2.0, 2.0, 3.0], np.float32), 2.0, -1, t2s, s2t)
    assert list(et) == [3]                                    # 2.0 is not above 2.0
    et, _ = orc.early_fetch(np.array([1e30] * 4, np.float32), np.inf, -1, t2s, s2t)
    assert list(et) == []                                     # no prediction yet
    et, _ = orc.early_fetch(np.array([5.0] * 4, np.float32), 1.0, 0, t2s, s2t)
    assert list(et) == []                                     # cap 0


def test_prefill_rows_causal(orc):
    rng = np.random.default_rng(1)
    R, row0, k = 6, 5, 4
    W = row0 + R + 3
    s = rng.standard_normal((R, W)).astype(np.float32)
    sel, kth, hist, un = orc.prefill_rows(s, row0, k, 0.25)
    for r in range(R):
        p = row0 + r
        idx, kt = orc.topk(s[r, :p + 1], k)
        assert np.array_equal(sel[r], idx) and kth[r] == kt
        assert np.array_equal(hist[r], orc.hist256(s[r, :p + 1], 0.25))
        assert sel[r].max() <= p                                 # causal
    want = np.zeros(row0 + R, np.uint8)
    want[sel[sel >= 0]] = 1
    assert np.array_equal(un, want)
    # rows that see at most k tokens select all of them
    sel, _, _, _ = orc.prefill_rows(s[:, :W], 0, 8, 0.0)
    assert list(sel[2]) == [0, 1, 2, -1, -1, -1, -1, -1]


def test_decode_step_pipeline(orc):
    """The whole-step oracle composes the pinned pieces: its selection equals
    topk of its own scores and every invariant holds."""
    from sparse_attention_kv_echo_gb300 import workloads as wl
    w = wl.scaled(wl.WORKLOADS["tiny"], "tiny2", B=2, lengths=(700, 1300), k=64, C=160, steps=4)
    off = wl.tok_offsets(w.lengths)
    k8, ks = wl.make_keys(w, 0)
    wt = wl.make_weights(w, 0)
    import torch
    host_u8 = wl.make_host_pool(w, 0).view(torch.uint8).numpy().reshape(w.total_tokens, -1)
    qs = wl.QueryStream(w, 0)
    theta = np.full(w.B, np.inf, np.float32)
    t2s = np.full(w.total_tokens, -1, np.int32)
    s2t = np.full(w.B * w.C, -1, np.int32)
    dev = np.zeros((w.B * w.C, host_u8.shape[1]), np.uint8)
    for step in range(w.steps):
        q = qs.next().numpy()
        out = orc.decode_step(off, q, wt.numpy(), k8.numpy(), ks.numpy(), w.k, 0.5, True, -1,
                              theta, w.C, t2s, s2t, host_u8, dev, nthreads=2, want_scores=True)
        for b in range(w.B):
            sc = out["scores"][off[b]:off[b + 1]]
            idx, kth = orc.topk(sc, w.k)
            assert np.array_equal(out["sel_idx"][b], idx) and out["kth"][b] == kth
            t = t2s[off[b]:off[b + 1]]
            st = s2t[b * w.C:(b + 1) * w.C]
            _check_invariants(t, st, idx)
            for s, j in zip(idx, out["sel_slot"][b]):
                assert np.array_equal(dev[b * w.C + j], host_u8[off[b] + s])
        assert np.all(np.isfinite(theta))


def test_cross_layer_early_set_pins(orc):
    # layer l selected {1, 3, 4, 6}; layer l+1 holds token 3 in slot 0 and token 5 in slot 2:
    # the early set is {1, 4, 6} (3 is resident), ascending, on the free slots 1, 3, 4
    n, C = 8, 32
    t2s = np.full(n, -1, np.int32)
    s2t = np.full(C, -1, np.int32)
    t2s[3], s2t[0] = 0, 3
    t2s[5], s2t[2] = 2, 5
    prev = np.array([1, 3, 4, 6, -1, -1], np.int32)
    et, es = orc.early_from_selection(prev, n, -1, t2s, s2t)
    assert et.tolist() == [1, 4, 6] and es.tolist() == [1, 3, 4]
    assert t2s.tolist() == [-1, 1, -1, 0, 3, 2, 4, -1]
    # a cap of 2 takes the two lowest tokens; with 2 free slots only, the free slots bound it
    t2s = np.full(n, -1, np.int32)
    s2t = np.full(C, -1, np.int32)
    et, es = orc.early_from_selection(prev, n, 2, t2s, s2t)
    assert et.tolist() == [1, 3] and es.tolist() == [0, 1]
    t2s = np.full(n, -1, np.int32)
    t2s[7] = 0
    s2t = np.full(C, -1, np.int32)
    s2t[0] = 7
    s2t[1] = 100   # a slot held by a token beyond the request
    with pytest.raises(Exception):
        orc.early_from_selection(prev, n, -1, t2s, s2t)  # inconsistent tables are refused


def test_cross_layer_equals_threshold_fetch_on_indicator_scores(orc):
    # the cross-layer early set is the threshold early fetch whose marked tokens are the previous
    # selection: both take the same tokens and slots on random tables
    rng = np.random.default_rng(4)
    for trial in range(20):
        n, C = 300, 64
        t2s = np.full(n, -1, np.int32)
        s2t = np.full(C, -1, np.int32)
        res = rng.choice(n, 20, replace=False)
        slots = rng.choice(C, 20, replace=False)
        t2s[res], s2t[slots] = slots, res
        prev = np.sort(rng.choice(n, 40, replace=False)).astype(np.int32)
        cap = int(rng.integers(-1, 50))
        ind = np.zeros(n, np.float32)
        ind[prev] = 1.0
        a2s, a_s2t = t2s.copy(), s2t.copy()
        et, es = orc.early_from_selection(np.concatenate([prev, [-1, -1]]), n, cap, t2s, s2t)
        et2, es2 = orc.early_fetch(ind, 0.5, cap, a2s, a_s2t)
        assert np.array_equal(et, et2) and np.array_equal(es, es2)
        assert np.array_equal(t2s, a2s) and np.array_equal(s2t, a_s2t)
