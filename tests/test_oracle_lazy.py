"""Pins of the oracle's lazy-reuse eviction (the cache-step variant in which a freed slot keeps
its token -- a ghost -- until the slot is handed to another token, and a selected ghost is a hit):
hand-worked steps, the early set leaving ghosts out, the reduction to the contract's cache step
when no freed token is ever selected again, and invariants (resident == selected, inverse tables,
every present token's bytes equal its host row) over random step sequences."""
import numpy as np
import pytest


def fresh(n, C):
    return np.full(n, -1, np.int32), np.full(C, -1, np.int32), np.ones(C, np.uint8)


def sel_of(*toks, m=4):
    out = np.full(m, -1, np.int32)
    out[:len(toks)] = toks
    return out


def test_worked_revival(orc):
    t2s, s2t, fr = fresh(16, 8)
    ss, mt, ms, rev = orc.lazy_cache_step(sel_of(0, 1, 2, 3), t2s, s2t, fr)
    assert list(ss) == [0, 1, 2, 3] and list(mt) == [0, 1, 2, 3] and list(ms) == [0, 1, 2, 3] and rev == 0
    # token 0 is not selected: a ghost in slot 0 (slot free, both entries kept)
    ss, mt, ms, rev = orc.lazy_cache_step(sel_of(1, 2, 3), t2s, s2t, fr)
    assert list(ss) == [1, 2, 3, -1] and mt.size == 0 and rev == 0
    assert t2s[0] == 0 and s2t[0] == 0 and fr[0] == 1 and list(fr[1:4]) == [0, 0, 0]
    # selected again while slot 0 still holds it: a hit, no recall
    ss, mt, ms, rev = orc.lazy_cache_step(sel_of(0, 1, 2, 3), t2s, s2t, fr)
    assert list(ss) == [0, 1, 2, 3] and mt.size == 0 and rev == 1 and fr[0] == 0


def test_a_miss_drops_the_ghost_in_its_slot(orc):
    t2s, s2t, fr = fresh(16, 8)
    orc.lazy_cache_step(sel_of(0, 1, 2, 3), t2s, s2t, fr)
    orc.lazy_cache_step(sel_of(1, 2, 3), t2s, s2t, fr)          # 0: ghost in slot 0
    ss, mt, ms, rev = orc.lazy_cache_step(sel_of(1, 2, 3, 7), t2s, s2t, fr)
    assert list(mt) == [7] and list(ms) == [0] and rev == 0     # the lowest free slot is the ghost's
    assert t2s[0] == -1 and t2s[7] == 0 and s2t[0] == 7 and fr[0] == 0


def test_early_set_leaves_ghosts_out(orc):
    n, C = 16, 8
    t2s, s2t, fr = fresh(n, C)
    orc.lazy_cache_step(sel_of(0, 1, 2, 3), t2s, s2t, fr)
    orc.lazy_cache_step(sel_of(1, 2, 3), t2s, s2t, fr)          # 0: ghost in slot 0
    scores = np.zeros(n, np.float32)
    scores[[0, 1, 9, 12]] = 5.0                                  # 0 ghost, 1 resident, 9 and 12 absent
    et, es = orc.lazy_early(scores, 1.0, -1, t2s, s2t, fr)
    assert list(et) == [9, 12] and list(es) == [0, 4]            # the lowest free slots, the ghost's first
    et1, es1 = orc.lazy_early(scores, 1.0, 1, t2s, s2t, fr)      # capped at one
    assert list(et1) == [9] and list(es1) == [0]
    ss, mt, ms, rev = orc.lazy_cache_step(sel_of(1, 2, 3, 9), t2s, s2t, fr, et, es)
    assert list(ss) == [1, 2, 3, 0] and mt.size == 0
    assert t2s[0] == -1                                          # the ghost left with its slot
    assert t2s[12] == 4 and s2t[4] == 12 and fr[4] == 1          # unselected early token: now a ghost


def _stream_without_returns(rng, n, k, steps):
    """Selections in which a token, once dropped, is never selected again."""
    used = set()
    cur = list(rng.choice(n // 4, k, replace=False))
    used.update(cur)
    out = []
    for _ in range(steps):
        keep = [t for t in cur if rng.random() < 0.6]
        pool = [t for t in range(n) if t not in used]
        new = list(rng.choice(pool, k - len(keep), replace=False))
        used.update(new)
        cur = keep + new
        out.append(np.sort(np.array(cur, np.int32)))
    return out


def test_reduces_to_the_contract_when_no_freed_token_returns(orc):
    rng = np.random.default_rng(2)
    n, k, C = 4000, 64, 160
    t2s, s2t = np.full(n, -1, np.int32), np.full(C, -1, np.int32)
    lt2s, ls2t, lfr = fresh(n, C)
    for sel in _stream_without_returns(rng, n, k, 25):
        a = orc.cache_step(sel, t2s, s2t)
        b = orc.lazy_cache_step(sel, lt2s, ls2t, lfr)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
        assert b[3] == 0
        live = np.where((lt2s >= 0) & (lfr[np.maximum(lt2s, 0)] == 0), lt2s, -1)
        assert np.array_equal(live, t2s)                        # the residents are the contract's


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_invariants_and_bytes_over_random_steps(orc, seed):
    """Scores drift around a fixed base, so tokens leave the selection and come back; the early
    set takes the tokens above the previous step's k-th score (at most 10).  After every step the
    resident tokens are the selection, the tables are inverse over the present tokens, ghosts sit
    in free slots, and a byte-level simulation (rows copied for early pairs and misses only)
    finds every present token's row equal to its host row."""
    rng = np.random.default_rng(seed)
    n, k, C, row = 600, 40, 120, 8
    host = rng.integers(0, 256, (n, row), dtype=np.uint8)
    dev = np.zeros((C, row), np.uint8)
    t2s, s2t, fr = fresh(n, C)
    base = rng.random(n).astype(np.float32)
    theta = np.float32(np.inf)
    revived_total = 0
    for step in range(40):
        scores = (base + 0.1 * rng.random(n)).astype(np.float32)
        sel = np.sort(np.argsort(-scores, kind="stable")[:k]).astype(np.int32)
        et, es = orc.lazy_early(scores, theta, 10, t2s, s2t, fr)
        theta = np.sort(scores)[-k]
        dev[es] = host[et]
        ss, mt, ms, rev = orc.lazy_cache_step(sel, t2s, s2t, fr, et, es)
        dev[ms] = host[mt]
        revived_total += rev
        live = {int(t) for t in np.nonzero(t2s >= 0)[0] if fr[t2s[t]] == 0}
        assert live == {int(t) for t in sel}
        assert np.array_equal(ss, t2s[sel])
        present = np.nonzero(t2s >= 0)[0]
        assert np.array_equal(s2t[t2s[present]], present)       # inverse over the present tokens
        assert np.all(s2t[s2t >= 0] >= 0) and np.array_equal(t2s[s2t[s2t >= 0]], np.nonzero(s2t >= 0)[0])
        assert np.array_equal(dev[t2s[present]], host[present])  # ghosts' bytes intact
        assert set(np.nonzero(fr)[0]) == set(range(C)) - {int(t2s[t]) for t in live}
    assert revived_total > 0                                     # the variant's point: hits on ghosts
