"""GPU parity of decode top-k over candidate lists (echo_topk_select_cands) against the
oracle's sort-based top-k: selections, k-th scores and thresholds bit-exact whichever path
a request takes -- its list (hand-built here: exactly k entries, ties at the cut, every
token, shuffled), or all its scores (no list, too few or too many entries, a corrupted
list, a boundary bin larger than shared memory, a request longer than one bitmap window)."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from sparse_attention_kv_echo_gb300 import _lib as L
from sparse_attention_kv_echo_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
dev = "cuda"
NO_CUT = np.uint32(0xFFFFFFFF)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.load(build_if_missing=True)


def order_keys(x):
    """Unsigned keys in the order of the float32 values (-0 counted as +0): input construction."""
    x = np.asarray(x, np.float32) + np.float32(0.0)
    u = x.view(np.uint32)
    return np.where(u & np.uint32(0x80000000), ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def run_select(scores_list, k, lists=None, theta=None, hist=True, cap=L.CAND_CAP):
    """lists[b]: None (no list: cut = none) or (cut_key, keys, idx, cnt) written into the lists."""
    lens = [len(s) for s in scores_list]
    off = wl.tok_offsets(lens)
    flat = np.concatenate([np.asarray(s, np.float32) for s in scores_list]) if sum(lens) else np.zeros(1, np.float32)
    B = len(lens)
    th = np.full(B, np.inf if theta is None else theta, np.float32)
    h = np.stack([orc.hist256(flat[off[b]:off[b + 1]], th[b]) for b in range(B)]).astype(np.uint32)
    cands = L.Cands(B, cap)
    key = np.zeros(B * cap, np.uint32)
    idx = np.zeros(B * cap, np.int32)
    cnt = np.zeros(B, np.int32)
    cut = np.full(B, NO_CUT, np.uint32)
    for b in range(B):
        if lists is None or lists[b] is None:
            continue
        c, kk, ii, nn = lists[b]
        cut[b] = c
        m = min(len(kk), cap)
        key[b * cap:b * cap + m] = kk[:m]
        idx[b * cap:b * cap + m] = ii[:m]
        cnt[b] = nn
    cands.key.copy_(torch.from_numpy(key.view(np.int32)))
    cands.idx.copy_(torch.from_numpy(idx))
    cands.cnt.copy_(torch.from_numpy(cnt))
    cands.cut.copy_(torch.from_numpy(cut.view(np.int32)))
    sc = torch.from_numpy(flat).to(dev)
    tht = torch.from_numpy(th).to(dev)
    ht = torch.from_numpy(h.view(np.int32)).to(dev) if hist else None
    sel = torch.empty((B, k), dtype=torch.int32, device=dev)
    kth = torch.empty(B, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stats = torch.zeros(L.STATS_N, dtype=torch.int32, device=dev)
    L.topk_select_cands(torch.from_numpy(off).to(dev), max(sum(lens), 1), sc, k, ht, tht, 0.5, cands, sel, kth, st,
                        stats=stats)
    torch.cuda.synchronize()
    return dict(sel=sel.cpu().numpy(), kth=kth.cpu().numpy(), theta=tht.cpu().numpy(), status=int(st.item()),
                stats=stats.cpu().numpy(), theta0=th, cut=cands.cut.cpu().numpy().view(np.uint32))


def check_exact(res, scores_list, k):
    for b, s in enumerate(scores_list):
        idx, kt = orc.topk(s, k)
        assert np.array_equal(res["sel"][b], idx), (b, np.nonzero(res["sel"][b] != idx)[0][:5])
        assert res["kth"][b] == np.float32(kt) or (math.isinf(kt) and math.isinf(res["kth"][b])), b
        want = orc.ema(res["theta0"][b], kt, 0.5)
        assert res["theta"][b] == np.float32(want) or (math.isinf(want) and math.isinf(res["theta"][b])), b


def crafted(rng):
    return [
        np.round(rng.standard_normal(5000) * 4).astype(np.float32),   # heavy ties
        np.full(3000, 2.5, np.float32),                               # all equal
        rng.standard_normal(100).astype(np.float32),                  # n < k
        np.zeros(0, np.float32),                                      # empty request
        np.array([-0.0, 0.0, -0.0] * 500, np.float32),                # signed zeros tie
        (rng.standard_normal(70000) * 30 + 140).astype(np.float32),   # boundary bin beyond shared memory
        -np.abs(rng.standard_normal(4097)).astype(np.float32),        # negative scores
        (rng.standard_normal(140000) * 1e4).astype(np.float32),       # long request
        np.full(20000, -3.5, np.float32),                             # equal scores beyond shared memory
    ]


@pytest.mark.parametrize("hist", [True, False])
def test_scan_path_crafted(hist):
    """No lists: every request selects from all its scores."""
    cases = crafted(np.random.default_rng(3))
    res = run_select(cases, 256, hist=hist)
    assert res["status"] == 0
    check_exact(res, cases, 256)
    # the unshifted N(140, 30) bin overflows shared memory: a second round of bins resolves it;
    # 20000 equal scores overflow both rounds and are selected by radix passes over the scores
    assert res["stats"][L.STAT_BOUNDARY_MAX] >= 20000
    assert res["stats"][L.STAT_TOPK_FALLBACK] == 1
    assert res["stats"][L.STAT_CAND_MISS] == 0            # no request had a list


def test_scan_path_with_prediction_and_bad_hist():
    rng = np.random.default_rng(4)
    s = [(rng.standard_normal(40000) * 30 + 140).astype(np.float32) for _ in range(3)]
    k = 2048
    theta = float(np.mean([orc.topk(x, k)[1] for x in s]))
    res = run_select(s, k, theta=theta)
    assert res["status"] == 0
    check_exact(res, s, k)
    assert res["stats"][L.STAT_BOUNDARY_MAX] < 4000       # the shift narrows the boundary bin
    assert res["stats"][L.STAT_TOPK_FALLBACK] == 0
    # the next step's cut leaves at least k tokens at or above it (rank 4k here)
    for b, x in enumerate(s):
        assert res["cut"][b] != NO_CUT
        assert (order_keys(x) >= res["cut"][b]).sum() >= k


def make_list(x, rank, rng, extra=0):
    """The list of the tokens whose key reaches that of rank `rank` (ties included), shuffled."""
    keys = order_keys(x)
    srt = np.sort(keys)[::-1]
    cut = srt[min(rank, x.size) - 1]
    ii = np.nonzero(keys >= cut)[0].astype(np.int32)
    ii = ii[rng.permutation(ii.size)]
    return cut, keys[ii], ii, ii.size + extra


def test_list_path_exact():
    """Lists cut at rank k (ties make them longer), 2k, 4k and at every token; shuffled order."""
    rng = np.random.default_rng(5)
    k = 512
    cases = [
        (rng.standard_normal(30000) * 20).astype(np.float32),
        np.round(rng.standard_normal(20000) * 3).astype(np.float32),    # ties at the k-th score
        np.round(rng.standard_normal(6000)).astype(np.float32),         # few distinct values: long lists
        (rng.standard_normal(9000) * 5 + 3).astype(np.float32),
        np.full(2000, 1.25, np.float32),                                 # every score equal: the list is all
    ]
    lists = [make_list(cases[0], k, rng), make_list(cases[1], 2 * k, rng), make_list(cases[2], k, rng),
             make_list(cases[3], 4 * k, rng), make_list(cases[4], k, rng)]
    assert lists[1][3] > 2 * k and lists[2][3] > k       # the ties lengthen the lists
    res = run_select(cases, k, lists=lists, theta=1.0)
    assert res["status"] == 0
    check_exact(res, cases, k)
    assert res["stats"][L.STAT_CAND_MISS] == 0           # every request selected from its list
    # the next cut: the key of rank 4k when the list holds it
    assert res["cut"][3] == np.sort(order_keys(cases[3]))[::-1][4 * k - 1]


def test_lists_that_cannot_be_used():
    """Too few entries (the k-th score is below the cut), more than the capacity, a corrupted
    entry: those requests select from all their scores, exactly, and are counted."""
    rng = np.random.default_rng(6)
    k = 256
    cases = [(rng.standard_normal(20000) * 10).astype(np.float32) for _ in range(4)]
    short = make_list(cases[0], k // 2, rng)
    over = make_list(cases[1], 3000, rng)
    corrupt = list(make_list(cases[2], 2 * k, rng))
    corrupt[2] = corrupt[2].copy()
    corrupt[2][5] = 20000 + 7                              # a token outside the request
    good = make_list(cases[3], 2 * k, rng)
    res = run_select(cases, k, lists=[short, over, tuple(corrupt), good], cap=2048)
    assert res["status"] == L.ST_BADDATA                  # the corrupted list is reported
    check_exact(res, cases, k)
    assert res["stats"][L.STAT_CAND_MISS] == 3


def test_request_longer_than_one_bitmap_window():
    """600000 tokens (two 2^19-token windows of the ordered write), with and without a list."""
    rng = np.random.default_rng(7)
    k = 2048
    x = (rng.standard_normal(600000) * 50).astype(np.float32)
    y = (rng.standard_normal(600000) * 50).astype(np.float32)
    res = run_select([x, y], k, lists=[None, make_list(y, 3 * k, rng)], theta=float(orc.topk(x, k)[1]))
    assert res["status"] == 0
    check_exact(res, [x, y], k)
    assert res["stats"][L.STAT_CAND_MISS] == 0


def test_decode_layer_without_lists_matches_oracle():
    """The decode step with the previous top-k (8-CTA clusters, no lists) stays exact."""
    from tests._parity import run_decode
    w = wl.scaled(wl.WORKLOADS["batch"], "nolists", B=3, lengths=(20000, 9000, 33000), C=4096)
    run_decode(w, 4, predictor=True, score_sample=512, cands=False)
    run_decode(w, 3, predictor=True, score_sample=512, cands=False, resolved=False)


def test_hot_set_lists_are_used():
    """The hot-set workload's shape (5% of tokens +2 before quantising), 4 requests: after the
    first step most requests select from their lists, and every step stays exact."""
    from tests._parity import run_decode
    w = wl.scaled(wl.WORKLOADS["v32"], "hot4", B=4, lengths=(131072, 65536, 131072, 20000))
    steps = 8
    rep = run_decode(w, steps, predictor=True, score_sample=512, check_every_score_step=False, keys_device="cuda")
    assert rep["cand_miss"] <= (steps - 1) * w.B // 2        # the first step has no lists
    assert rep["fallbacks"] <= w.B                           # only the unshifted first step may overflow
