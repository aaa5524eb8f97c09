"""GPU parity of chunked prefill (echo_prefill_block) against the oracle.

Small prompt, every block, every row: causal scores within the fp64
tolerance (sampled rows), per-row shifted histograms, exact per-row top-k
and k-th scores, the union of a block's selections, the block threshold
EMA, the cache step on the union (tables, slots) and the recalled bytes.
The full-size prompt (102400 tokens in 2048-row blocks, every block) is in
test_gpu_full.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from sparse_attention_kv_echo_gb300 import _lib as L
from sparse_attention_kv_echo_gb300 import workloads as wl
from sparse_attention_kv_echo_gb300.prefill import PrefillRunner
from tests._parity import score_tolerance_ok

pytestmark = pytest.mark.gpu
dev = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.load(build_if_missing=True)


def _check_rows_scores(rows, row0, gs, q, wt, k8, ks, at=None):
    q8, qs, _ = orc.quantize_q(q, wt)
    for r in rows:
        p = row0 + r
        ref, ab = orc.scores(q8[r], qs[r], wt[r], k8, ks, tok=np.arange(p + 1, dtype=np.int64))
        bad, _ = score_tolerance_ok(gs[r if at is None else at[int(r)], :p + 1], ref, ab)
        assert bad.size == 0, (r, bad[:5])


def _run(w, full_rows=True, row_sample=8, blocks=None, keys_device="cpu", same_keys=False):
    k8c, ksc = wl.make_keys(w, 0, device=keys_device)
    if same_keys:  # every token carries the first token's key and scale
        k8c = k8c[:1].expand_as(k8c).contiguous()
        ksc = ksc[:1].expand_as(ksc).contiguous()
    k8, ks = k8c.cpu().numpy(), ksc.cpu().numpy()
    host = wl.make_host_pool(w, 0, device=keys_device, pin=True)
    host_gpu = host.to(dev)
    N = w.total_tokens
    pr = PrefillRunner(k8c.to(dev), ksc.to(dev), w.k, w.C, host, w.prefill_block)
    t2s = np.full(N, -1, np.int32)
    s2t = np.full(w.C, -1, np.int32)
    theta = np.float32(np.inf)
    rng = np.random.default_rng(3)
    nblocks = pr.blocks() if blocks is None else blocks
    for i in range(nblocks):
        q, wt = wl.make_prefill_queries(w, i, device=keys_device)
        row0, R = pr.block(i, q.to(dev), wt.to(dev))
        pr.wait_recall()
        torch.cuda.synchronize()
        assert int(pr.status.item()) == 0, f"status {int(pr.status.item()):#x} at block {i}"
        rows = np.arange(R) if full_rows else np.unique(np.concatenate(
            [rng.choice(R, min(row_sample, R), replace=False), [R - 1]]))
        # the scores of the rows checked (every row, or the sampled ones and the last), as rows of gs
        if full_rows:
            gs = pr.scores[:R].cpu().numpy()
            at = {int(r): int(r) for r in rows}
        else:
            gs = pr.scores[torch.from_numpy(rows).to(dev)].cpu().numpy()
            at = {int(r): j for j, r in enumerate(rows)}
        g_sel = pr.sel_idx[:R].cpu().numpy()
        g_kth = pr.kth[:R].cpu().numpy()
        g_hist = pr.hist[:R].cpu().numpy().view(np.uint32)
        g_list = pr.union_list.cpu().numpy()
        g_cnt = int(pr.union_count.item())
        g_theta = float(pr.theta.item())
        _check_rows_scores(rows[:row_sample] if full_rows else rows, row0, gs, q.cpu().numpy(),
                           wt.cpu().numpy(), k8, ks, at)
        for r in rows:
            p = row0 + r
            idx, kt = orc.topk(gs[at[int(r)], :p + 1], w.k)
            assert np.array_equal(g_sel[r], idx), (i, r)
            assert g_kth[r] == np.float32(kt), (i, r)
            assert np.array_equal(g_hist[r], orc.hist256(gs[at[int(r)], :p + 1], theta)), (i, r)
            assert np.all(g_sel[r][g_sel[r] >= 0] <= p)                     # causal
        # union: exactly the tokens some row selected, ascending, -1 padded
        sel_all = g_sel[g_sel >= 0]
        want_union = np.unique(sel_all)
        if full_rows:
            o_sel, o_kth, _, o_union = orc.prefill_rows(gs, row0, w.k, theta)
            assert np.array_equal(o_sel, g_sel)
            want_union = np.nonzero(o_union)[0].astype(np.int32)
        assert g_cnt == want_union.size
        assert np.array_equal(g_list[:g_cnt], want_union)
        assert np.all(g_list[g_cnt:] == -1)
        # block threshold: EMA of the last row's k-th score
        _, kt_last = orc.topk(gs[at[R - 1], :row0 + R], w.k)
        theta = np.float32(orc.ema(theta, kt_last, 0.5))
        assert g_theta == theta or (math.isinf(g_theta) and math.isinf(theta))
        # cache step on the union
        padded = np.full(pr.W, -1, np.int32)
        padded[:g_cnt] = want_union
        ss, mt, ms, _ = orc.cache_step(padded, t2s, s2t)
        assert np.array_equal(pr.sel_slot.cpu().numpy(), ss), i
        assert np.array_equal(pr.cache.tok2slot.cpu().numpy()[:N], t2s), i
        assert np.array_equal(pr.cache.slot2tok.cpu().numpy(), s2t), i
        tok = torch.from_numpy(want_union).long().to(dev)
        slot = torch.from_numpy(ss[:g_cnt]).long().to(dev)
        assert torch.equal(pr.cache.dev_kv[slot].view(torch.int16), host_gpu[tok].view(torch.int16)), i
    return pr


def test_prefill_small_every_row():
    # 6000-token prompt, 1024-row blocks (the last one ragged: 880 rows), k = 256
    w = wl.scaled(wl.WORKLOADS["prefill"], "pf_small", lengths=(6000,), prefill_block=1024, k=256, C=6016)
    _run(w, full_rows=True)


def test_prefill_rows_fewer_than_k():
    # early rows see fewer than k tokens and select all of them
    w = wl.scaled(wl.WORKLOADS["prefill"], "pf_tiny", lengths=(700,), prefill_block=256, k=300, C=704)
    _run(w, full_rows=True)


def test_prefill_all_keys_equal():
    """Every key the same, so every score of a row ties: each row selects its lowest
    k positions (ties go to the lower index) and the union is [0, k)."""
    w = wl.scaled(wl.WORKLOADS["prefill"], "pf_ties", lengths=(8192,), prefill_block=2048, k=256, C=8192)
    pr = _run(w, full_rows=True, row_sample=4, same_keys=True)
    sel = pr.sel_idx[:2048].cpu().numpy()
    assert np.array_equal(sel[-1], np.arange(256, dtype=np.int32))


def test_prefill_all_keys_equal_past_shared_memory():
    """The same ties in rows longer than 16384 tokens: the boundary bin, then its second-round
    sub-bin, overflow shared memory, and the row is selected by radix passes over its scores
    (sampled rows of every block checked)."""
    w = wl.scaled(wl.WORKLOADS["prefill"], "pf_ties2", lengths=(20000,), prefill_block=4096, k=256, C=20000)
    pr = _run(w, full_rows=False, row_sample=3, same_keys=True)
    sel = pr.sel_idx[:pr.R].cpu().numpy()
    assert np.array_equal(sel[-1], np.arange(256, dtype=np.int32))
    assert int(pr.stats[L.STAT_TOPK_FALLBACK].item()) > 0


