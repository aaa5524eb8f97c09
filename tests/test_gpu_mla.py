"""GPU parity of the sparse MLA decode attention over the selected slots against
the oracle (fp64): ragged selections with padding, a split boundary and a
ragged last tile, an empty request, the full k = 2048 selection."""
import math

import numpy as np
import pytest
import torch

from sparse_attention_kv_echo_gb300 import _lib as L

pytestmark = pytest.mark.gpu
dev = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.load(build_if_missing=True)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _run(B, C, k, valid_frac, seed, scale=1.0 / math.sqrt(192.0), empty=()):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, L.MLA_HEADS, L.MLA_DQK), generator=g).to(torch.bfloat16)
    kv = torch.randn((B * C, L.MLA_DQK), generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    sel = np.full((B, k), -1, np.int32)
    for b in range(B):
        if b in empty:
            continue
        m = max(1, int(k * valid_frac))
        pos = np.sort(rng.choice(k, m, replace=False))
        sel[b, pos] = rng.choice(C, m, replace=False)
    out = torch.empty((B, L.MLA_HEADS, L.MLA_DV), dtype=torch.float32, device=dev)
    lse = torch.empty((B, L.MLA_HEADS), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    L.mla_decode(q.to(dev), torch.from_numpy(sel).to(dev), kv.to(dev), C, scale, out, lse, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return q, kv, sel, out.cpu().numpy(), lse.cpu().numpy(), scale


def _check(q, kv, sel, out, lse, scale, C, orc):
    kvb = _bits(kv)
    qb = _bits(q)
    for b in range(sel.shape[0]):
        ref, ref_lse, mass = orc.mla_decode(qb[b], kvb[b * C:(b + 1) * C], sel[b], scale)
        tol = 5e-3 * mass + 1e-5
        bad = np.abs(out[b] - ref) > tol
        assert not bad.any(), (b, np.argwhere(bad)[:5], out[b][bad][:5], ref[bad][:5])
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse[b]))
        assert np.all(np.abs(lse[b][fin] - ref_lse[fin]) <= 3e-3 * np.maximum(1.0, np.abs(ref_lse[fin])))


def test_one_tile(orc):
    B, C, k = 1, 64, 16            # one split of one tile
    r = _run(B, C, k, 1.0, 3)
    _check(*r, C, orc)


def test_ragged_selection_two_splits(orc):
    B, C, k = 3, 700, 300          # splits of 256 + 44 (a ragged last tile), padding, one empty request
    r = _run(B, C, k, 0.8, 0, empty=(1,))
    _check(*r, C, orc)
    out = r[3]
    assert np.all(out[1] == 0) and np.all(np.isneginf(r[4][1]))


def test_full_selection_batch(orc):
    B, C, k = 2, 4096, 2048        # the decode workload's k and slots
    r = _run(B, C, k, 1.0, 1)
    _check(*r, C, orc)


def test_long_selection_wide_splits(orc):
    # k = 3000: splits of at least 384 tokens (12 tiles), the last one ragged
    B, C, k = 1, 4096, 3000
    r = _run(B, C, k, 0.9, 4)
    _check(*r, C, orc)


def test_odd_split_count(orc):
    # k = 700: a split count that does not divide the 128 heads evenly over the cluster
    B, C, k = 2, 1024, 700
    r = _run(B, C, k, 1.0, 5)
    _check(*r, C, orc)


def test_rejects_oversized_selection():
    q = torch.zeros((1, L.MLA_HEADS, L.MLA_DQK), dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((64, L.MLA_DQK), dtype=torch.bfloat16, device=dev)
    sel = torch.zeros((1, L.MLA_MAX_K + 1), dtype=torch.int32, device=dev)
    out = torch.empty((1, L.MLA_HEADS, L.MLA_DV), dtype=torch.float32, device=dev)
    lse = torch.empty((1, L.MLA_HEADS), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(L.EchoError):
        L.mla_decode(q, sel, kv, 64, 1.0, out, lse, st)


def test_peaked_scores(orc):
    # a large scale makes the softmax nearly one-hot: the running max moves between tiles
    B, C, k = 1, 512, 256
    r = _run(B, C, k, 1.0, 2, scale=0.5)
    _check(*r, C, orc)


@pytest.mark.parametrize("hold_early", [False, True])
def test_attention_in_the_decode_graph(orc, hold_early):
    # the decode step with attention=True, captured in one CUDA graph: each request group's
    # attention runs over its selected slots once its rows are in the cache.  Expected values:
    # the oracle's top-k on the step's fp32 scores, then the oracle attention over those
    # tokens' rows of the host pool (slot placement does not enter)
    from sparse_attention_kv_echo_gb300 import DecodeLayer
    from sparse_attention_kv_echo_gb300 import workloads as wl
    w = wl.scaled(wl.WORKLOADS["batch"], "attn", B=4, lengths=(3000, 5000, 700, 4096), k=512, C=1024)
    off = wl.tok_offsets(w.lengths)
    k8, ks = wl.make_keys(w, 0)
    wt = wl.make_weights(w, 0)
    host = wl.make_host_pool(w, 0, pin=True)
    lay = DecodeLayer(off, k8.to(dev), ks.to(dev), w.k, w.C, host, attention=True, hold_early=hold_early,
                      device=dev)
    assert len(lay.groups) == 2
    qs = wl.QueryStream(w, 0)
    g = torch.Generator().manual_seed(9)
    mq = [torch.randn((w.B, L.MLA_HEADS, L.MLA_DQK), generator=g).to(torch.bfloat16) for _ in range(3)]
    qq = [qs.next() for _ in range(3)]
    main = torch.cuda.Stream()
    with torch.cuda.stream(main):
        lay.w_in.copy_(wt.to(dev))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=main):
        lay.step(stream=main)
    torch.cuda.synchronize()
    lay.reset()
    hb = _bits(host)
    for t in range(3):
        with torch.cuda.stream(main):
            lay.q_in.copy_(qq[t].to(dev))
            lay.mla_q.copy_(mq[t].to(dev))
            graph.replay()
        torch.cuda.synchronize()
        assert int(lay.status.item()) == 0
        scores = lay.scores.cpu().numpy()
        out = lay.attn_out.cpu().numpy()
        lse = lay.attn_lse.cpu().numpy()
        qb = _bits(mq[t])
        for b in range(w.B):
            idx, _ = orc.topk(scores[off[b]:off[b + 1]], w.k)
            assert np.array_equal(idx, lay.sel_idx[b].cpu().numpy())
            ref, ref_lse, mass = orc.mla_decode(qb[b], hb[off[b]:off[b + 1]], idx, lay.mla_scale)
            assert np.all(np.abs(out[b] - ref) <= 5e-3 * mass + 1e-5), (t, b)
            assert np.all(np.abs(lse[b] - ref_lse) <= 3e-3 * np.maximum(1.0, np.abs(ref_lse)))


@pytest.mark.parametrize("k", [1, 31, 33])
def test_tiny_selections(orc, k):
    # one tile, or fewer tiles than the gather ring keeps in flight, or a ragged second tile
    B, C = 2, 64
    r = _run(B, C, k, 1.0, 10 + k)
    _check(*r, C, orc)


def test_maximum_selection_wraps_the_ring(orc):
    # k = 8192: 8 splits of 1024 tokens, 32 tiles each -- the four-stage ring wraps eight times
    B, C, k = 1, 9000, 8192
    r = _run(B, C, k, 0.97, 21)
    _check(*r, C, orc)


def test_only_the_last_entry_valid(orc):
    B, C, k = 1, 512, 300
    g = torch.Generator().manual_seed(5)
    q = torch.randn((B, L.MLA_HEADS, L.MLA_DQK), generator=g).to(torch.bfloat16)
    kv = torch.randn((B * C, L.MLA_DQK), generator=g).to(torch.bfloat16)
    sel = np.full((B, k), -1, np.int32)
    sel[0, k - 1] = 77
    out = torch.empty((B, L.MLA_HEADS, L.MLA_DV), dtype=torch.float32, device=dev)
    lse = torch.empty((B, L.MLA_HEADS), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    L.mla_decode(q.to(dev), torch.from_numpy(sel).to(dev), kv.to(dev), C, 0.1, out, lse, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # one valid token: every head's output is that token's first 512 values, lse its score
    row = kv[77, :L.MLA_DV].float().numpy()
    assert np.allclose(out.cpu().numpy()[0], row[None, :], atol=1e-6, rtol=0)
    _check(q, kv, sel, out.cpu().numpy(), lse.cpu().numpy(), 0.1, C, orc)
