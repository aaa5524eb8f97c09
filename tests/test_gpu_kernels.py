"""GPU parity of the single calls against the oracle: query quantisation (bit-exact
E4M3 bytes), the score kernel (fp64 oracle within tolerance, histogram
bit-exact), top-k on crafted scores (bit-exact), the cache step on crafted
selections (bit-exact tables, recalled bytes), status reporting."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from sparse_attention_kv_echo_gb300 import _lib as L
from sparse_attention_kv_echo_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
dev = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.load(build_if_missing=True)


def _quant_gpu(q, w):
    B = q.shape[0]
    q8 = torch.empty((B, 64, 128), dtype=torch.uint8, device=dev)
    qs = torch.empty((B, 64), dtype=torch.float32, device=dev)
    wf = torch.empty((B, 64), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    L.quantize_q(q.to(dev), w.to(dev), q8, qs, wf, st)
    torch.cuda.synchronize()
    return q8.cpu().numpy(), qs.cpu().numpy(), wf.cpu().numpy(), int(st.item())


def test_quantize_bit_exact():
    g = torch.Generator().manual_seed(11)
    B = 37
    q = torch.randn((B, 64, 128), generator=g)
    scale = torch.exp(torch.empty((B, 64, 1)).uniform_(-30, 30, generator=g))
    q = (q * scale).float()
    q[3] = 0.0                                   # all-zero rows: scale 1
    q[4, :, :] = 1e-41                           # subnormal amax: clamped exponent
    q[5, 7, :] = -0.0
    q[6, 1, 9] = 448.0
    q[7, 2, 0] = 1.75
    w = torch.rand((B, 64), generator=g)
    q8, qs, wf, st = _quant_gpu(q, w)
    r8, rs, rw = orc.quantize_q(q.numpy(), w.numpy())
    assert st == 0
    assert np.array_equal(qs, rs)
    assert np.array_equal(wf, rw)
    bad = np.argwhere(q8 != r8)
    assert bad.size == 0, bad[:5]


def test_e4m3_conversion_sweep():
    """Rows whose amax is exactly 448 have scale 1, so q8 = E4M3(q) directly: sweep many
    fp32 bit patterns of every binade the format covers (and beyond, into zero)."""
    vals = []
    for e in range(-20, 9):
        m = np.arange(0, 1 << 23, 61, dtype=np.uint32)
        vals.append(((np.uint32(e + 127) << np.uint32(23)) | m).view(np.float32))
    vals.append(np.array([2.0 ** -10, 3 * 2.0 ** -10, 232.0, 1.0625, 1.1875, 0.0], np.float32))
    x = np.concatenate(vals)
    x = np.concatenate([x, -x])
    x = x[np.abs(x) < 448]
    per_row = 127
    rows = (x.size + per_row - 1) // per_row
    pad = rows * per_row - x.size
    xp = np.concatenate([x, np.zeros(pad, np.float32)]).reshape(rows, per_row)
    full = np.concatenate([np.full((rows, 1), 448.0, np.float32), xp], axis=1)
    B = (rows + 63) // 64
    full = np.concatenate([full, np.full((B * 64 - rows, 128), 448.0, np.float32)])
    q = torch.from_numpy(full.reshape(B, 64, 128).copy())
    w = torch.ones((B, 64))
    assert B <= L.MAX_REQUESTS
    q8, qs, _, st = _quant_gpu(q, w)
    assert st == 0 and np.all(qs == 1.0)
    got = q8.reshape(-1, 128)[:rows, 1:].reshape(-1)[:x.size]
    ref = orc.e4m3_encode(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


def _scores_gpu(off, n, q, w, k8, ks, scores, theta, hist, status, above=None):
    """quantize_q (clears hist) then index_scores, as a step issues them."""
    B = q.shape[0]
    q8 = torch.empty((B, 64, 128), dtype=torch.uint8, device=dev)
    qs = torch.empty((B, 64), dtype=torch.float32, device=dev)
    wf = torch.empty((B, 64), dtype=torch.float32, device=dev)
    L.quantize_q(q, w, q8, qs, wf, status, hist=hist)
    L.index_scores(off, n, q8, wf, k8, ks, scores, theta, hist, status, above=above)


def _score_call(w, layer=0, theta=None, device_keys="cpu"):
    off = wl.tok_offsets(w.lengths)
    k8, ks = wl.make_keys(w, layer, device=device_keys)
    wt = wl.make_weights(w, layer, device=device_keys)
    q = wl.QueryStream(w, layer, device=device_keys).next()
    n = w.total_tokens
    scores = torch.full((max(n, 1) + 64,), float("nan"), device=dev)
    hist = torch.zeros((w.B, 256), dtype=torch.int32, device=dev)
    th = torch.full((w.B,), math.inf if theta is None else theta, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    hist.fill_(12345)                                 # stale contents: quantize_q must clear them
    above = torch.full((L.above_words(w.B, n),), -1, dtype=torch.int32, device=dev)
    _scores_gpu(torch.from_numpy(off).to(dev), n, q.to(dev), wt.to(dev), k8.to(dev), ks.to(dev), scores,
                th, hist, st, above=above)
    torch.cuda.synchronize()
    return off, k8.cpu().numpy(), ks.cpu().numpy(), q.cpu().numpy(), wt.cpu().numpy(), scores.cpu().numpy(), \
        hist.cpu().numpy().view(np.uint32), int(st.item()), th.cpu().numpy(), above.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("lengths,theta", [
    ((8192,), None),                         # tiny: 64 full tiles
    ((1000, 129, 0, 4173, 300, 1), 150.0),   # ragged tails, an empty request, a 1-token request
    ((128 * 300 + 5,), 170.0),               # more tiles than SMs, ragged tail
])
def test_scores_and_hist(lengths, theta):
    from tests._parity import check_scores
    w = wl.scaled(wl.WORKLOADS["tiny"], "s", B=len(lengths), lengths=tuple(lengths))
    off, k8, ks, q, wt, gs, gh, st, th, ab = _score_call(w, theta=theta)
    assert st == 0
    check_scores((off, k8, ks), q, wt, gs)
    for b in range(w.B):
        sc = gs[off[b]:off[b + 1]]
        assert np.array_equal(gh[b], orc.hist256(sc, th[b]))
        # above-threshold bits: request b's words start at 4 * (floor(first row / 128) + b)
        t0 = 4 * (int(off[b]) // 128 + b)
        nb = sc.size
        words = 4 * ((nb + 127) // 128)
        bits = np.unpackbits(ab[t0:t0 + words].view(np.uint8), bitorder="little")[:nb].astype(bool) \
            if words else np.zeros(0, bool)
        want = (sc > th[b]) if np.isfinite(th[b]) else np.zeros(nb, bool)
        assert np.array_equal(bits, want), b
        if words:
            pad = np.unpackbits(ab[t0:t0 + words].view(np.uint8), bitorder="little")[nb:]
            assert not pad.any()
    assert np.all(np.isnan(gs[w.total_tokens:]))      # rows outside every request untouched


def test_scores_integer_exact():
    """Small-integer keys and queries with power-of-two scales: every product and
    partial sum is exact in fp32, so the GPU score equals the oracle exactly."""
    rng = np.random.default_rng(5)
    n = 640
    tab = orc.e4m3_table()
    lut = {float(tab[c]): c for c in range(128) if float(tab[c]).is_integer()}
    lut.update({-v: c | 0x80 for v, c in list(lut.items()) if v > 0})
    ki = rng.integers(-3, 4, (n, 128))
    k8 = np.vectorize(lambda v: lut[float(v)])(ki).astype(np.uint8)
    ks = (2.0 ** rng.integers(-2, 2, n)).astype(np.float32)
    q = rng.integers(-3, 4, (1, 64, 128)).astype(np.float32)
    q[0, :, 0] = 7.0               # amax 7 -> scale 2^-6 exactly; q/scale = 64 * integer, exact in E4M3
    w = (rng.integers(0, 5, (1, 64)) / 4.0).astype(np.float32)
    off = np.array([0, n], np.int64)
    scores = torch.zeros(n, device=dev)
    hist = torch.zeros((1, 256), dtype=torch.int32, device=dev)
    th = torch.full((1,), math.inf, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _scores_gpu(torch.from_numpy(off).to(dev), n, torch.from_numpy(q).to(dev), torch.from_numpy(w).to(dev),
                torch.from_numpy(k8).to(dev), torch.from_numpy(ks).to(dev), scores, th, hist, st)
    torch.cuda.synchronize()
    q8, qs, _ = orc.quantize_q(q, w)
    ref, _ = orc.scores(q8[0], qs[0], w[0], k8, ks)
    assert np.array_equal(scores.cpu().numpy().astype(np.float64), ref)


def _topk_gpu(scores_list, k, theta=None, hist=True):
    lens = [len(s) for s in scores_list]
    off = wl.tok_offsets(lens)
    flat = np.concatenate([np.asarray(s, np.float32) for s in scores_list]) if sum(lens) else np.zeros(1, np.float32)
    B = len(lens)
    th = np.full(B, np.inf if theta is None else theta, np.float32)
    h = np.stack([orc.hist256(flat[off[b]:off[b + 1]], th[b]) for b in range(B)]).astype(np.uint32)
    sc = torch.from_numpy(flat).to(dev)
    tht = torch.from_numpy(th).to(dev)
    ht = torch.from_numpy(h.view(np.int32)).to(dev) if hist else None
    sel = torch.empty((B, k), dtype=torch.int32, device=dev)
    kth = torch.empty(B, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stats = torch.zeros(8, dtype=torch.int32, device=dev)
    L.topk_select(torch.from_numpy(off).to(dev), max(sum(lens), 1), sc, k, ht, tht, 0.5, sel, kth, st, stats=stats)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), kth.cpu().numpy(), tht.cpu().numpy(), int(st.item()), stats.cpu().numpy(), th


@pytest.mark.parametrize("hist", [True, False])
def test_topk_crafted(hist):
    rng = np.random.default_rng(3)
    cases = [
        np.round(rng.standard_normal(5000) * 4).astype(np.float32),   # heavy ties
        np.full(3000, 2.5, np.float32),                               # all equal
        rng.standard_normal(100).astype(np.float32),                  # n < k
        np.zeros(0, np.float32),                                      # empty request
        np.array([-0.0, 0.0, -0.0] * 500, np.float32),                # signed zeros tie
        (rng.standard_normal(70000) * 30 + 140).astype(np.float32),   # boundary bin overflows smem
        -np.abs(rng.standard_normal(4097)).astype(np.float32),        # negative scores
        (rng.standard_normal(140000) * 1e4).astype(np.float32),       # slices too long for shared memory
        np.concatenate([rng.random(35000) * 1e-3,                     # the boundary bin in one slice,
                        0.6 + 0.3 * rng.random(5000)]).astype(np.float32),  # more than a slice lists
    ]
    k = 256
    sel, kth, th_new, st, stats, th = _topk_gpu(cases, k, hist=hist)
    assert st == 0
    for b, s in enumerate(cases):
        idx, kt = orc.topk(s, k)
        assert np.array_equal(sel[b], idx), (b, np.nonzero(sel[b] != idx)[0][:5])
        assert kth[b] == np.float32(kt) or (math.isinf(kt) and math.isinf(kth[b]))
        want = orc.ema(th[b], kt, 0.5)
        assert th_new[b] == np.float32(want) or (math.isinf(want) and math.isinf(th_new[b]))
    assert stats[L.STAT_TOPK_FALLBACK] >= 1


def test_topk_with_prediction_and_bad_hist():
    rng = np.random.default_rng(4)
    s = [(rng.standard_normal(40000) * 30 + 140).astype(np.float32) for _ in range(3)]
    k = 2048
    idx0 = [orc.topk(x, k) for x in s]
    theta = float(np.mean([t for _, t in idx0]))
    sel, kth, th_new, st, stats, _ = _topk_gpu(s, k, theta=theta)
    assert st == 0
    for b in range(3):
        assert np.array_equal(sel[b], idx0[b][0])
        assert th_new[b] == np.float32(orc.ema(np.float32(theta), idx0[b][1], 0.5))
    assert stats[L.STAT_BOUNDARY_MAX] < 4000          # the shift narrows the boundary bin
    # a histogram that does not describe the scores is detected, rebuilt, and the result stays exact
    lens = [x.size for x in s]
    off = wl.tok_offsets(lens)
    flat = np.concatenate(s)
    wrong = np.zeros((3, 256), np.int32)
    wrong[:, 200] = 40000
    sel_t = torch.empty((3, k), dtype=torch.int32, device=dev)
    kth_t = torch.empty(3, device=dev)
    st_t = torch.zeros(1, dtype=torch.int32, device=dev)
    L.topk_select(torch.from_numpy(off).to(dev), flat.size, torch.from_numpy(flat).to(dev), k,
                  torch.from_numpy(wrong).to(dev), None, 0.5, sel_t, kth_t, st_t)
    torch.cuda.synchronize()
    assert int(st_t.item()) == L.ST_BADDATA
    for b in range(3):
        assert np.array_equal(sel_t[b].cpu().numpy(), idx0[b][0])


def test_cache_step_crafted():
    """Random selections of a 3-request batch, C = 2k, through the GPU cache step
    and the oracle's; tables, slots, misses and recalled bytes bit-exact."""
    rng = np.random.default_rng(9)
    lens = (3000, 700, 5000)
    B, C, k = 3, 512, 256
    off = wl.tok_offsets(lens)
    n = int(off[-1])
    host = torch.randint(-30000, 30000, (n, 576), dtype=torch.int16).view(torch.bfloat16).pin_memory()
    cache = L.LayerCache(B, n, C, host)
    t2s = np.full(n, -1, np.int32)
    s2t = np.full(B * C, -1, np.int32)
    tok_off = torch.from_numpy(off).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    host_gpu = host.to(dev)
    for step in range(8):
        sel = np.full((B, k), -1, np.int32)
        for b in range(B):
            m = min(k, lens[b]) if step % 3 else min(k - 7, lens[b])      # some padding too
            sel[b, :m] = np.sort(rng.choice(lens[b], m, replace=False))
        sel_t = torch.from_numpy(sel).to(dev)
        slot_t = torch.empty_like(sel_t)
        L.cache_step(tok_off, n, sel_t, cache, slot_t, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        g_slot = slot_t.cpu().numpy()
        for b in range(B):
            ss, mt, ms, _ = orc.cache_step(sel[b], t2s[off[b]:off[b + 1]], s2t[b * C:(b + 1) * C])
            assert np.array_equal(g_slot[b], ss)
            assert cache.miss_cnt[b].item() == mt.size
            assert np.array_equal(cache.miss_tok[b * C:b * C + mt.size].cpu().numpy(), mt)
            assert np.array_equal(cache.miss_slot[b * C:b * C + mt.size].cpu().numpy(), ms)
        assert np.array_equal(cache.tok2slot.cpu().numpy(), t2s)
        assert np.array_equal(cache.slot2tok.cpu().numpy(), s2t)
        v = sel_t >= 0
        bidx = torch.arange(B, device=dev)[:, None].expand_as(sel_t)
        rows = cache.dev_kv[(bidx * C + slot_t.long())[v]]
        want = host_gpu[(tok_off[:-1, None] + sel_t.long())[v]]
        assert torch.equal(rows.view(torch.int16), want.view(torch.int16))


def test_nan_query_sets_status():
    w = wl.scaled(wl.WORKLOADS["tiny"], "nan", lengths=(1024,))
    off = wl.tok_offsets(w.lengths)
    k8, ks = wl.make_keys(w, 0)
    q = torch.randn((1, 64, 128))
    q[0, 5, 5] = float("nan")
    wt = torch.rand((1, 64))
    scores = torch.zeros(1024, device=dev)
    hist = torch.zeros((1, 256), dtype=torch.int32, device=dev)
    th = torch.full((1,), math.inf, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _scores_gpu(torch.from_numpy(off).to(dev), 1024, q.to(dev), wt.to(dev), k8.to(dev), ks.to(dev), scores,
                th, hist, st)
    torch.cuda.synchronize()
    assert int(st.item()) & L.ST_NAN


def test_bad_offsets_set_status_not_fault():
    """tok_off beyond n_tokens is reported as bad data; nothing reads out of bounds."""
    off = torch.tensor([0, 5000], dtype=torch.int64, device=dev)
    n = 1024
    k8 = torch.zeros((n, 128), dtype=torch.uint8, device=dev)
    ks = torch.ones(n, device=dev)
    scores = torch.zeros(n, device=dev)
    hist = torch.zeros((1, 256), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _scores_gpu(off, n, torch.randn((1, 64, 128), device=dev), torch.rand((1, 64), device=dev), k8, ks,
                scores, None, hist, st)
    sel = torch.empty((1, 16), dtype=torch.int32, device=dev)
    kth = torch.empty(1, device=dev)
    L.topk_select(off, n, scores, 16, hist, None, 0.5, sel, kth, st)
    torch.cuda.synchronize()
    assert int(st.item()) & L.ST_BADDATA
    assert torch.all(sel == -1)
