"""Shared GPU-parity driver: runs decode steps through the C ABI and checks
every output against the CPU oracle fed with the same input bytes.

Checks per step (the oracle keeps its own cache state, never copied from the GPU):
  scores        |gpu - oracle_fp64| <= 1e-3 |oracle| + 1e-6 A   (A = size of the terms)
  hist          bit-exact: oracle histogram of the GPU scores with the same threshold
  early fetch   bit-exact lists, counts and tables
  top-k         bit-exact indices and k-th score on the GPU scores; EMA threshold bit-exact
  cache step    bit-exact tables, slots, miss lists
  recall        device cache rows of every selected token == host rows
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as orc
from sparse_attention_kv_echo_gb300 import DecodeLayer
from sparse_attention_kv_echo_gb300 import _lib as L
from sparse_attention_kv_echo_gb300 import workloads as wl

RTOL, ATOL_REL = 1e-3, 1e-6


def score_tolerance_ok(gpu, ref, absb):
    gpu = np.asarray(gpu, np.float64)
    err = np.abs(gpu - ref)
    lim = RTOL * np.abs(ref) + ATOL_REL * absb
    bad = np.nonzero(err > lim)[0]
    return bad, float((err / np.maximum(np.abs(ref), 1e-30)).max()) if err.size else 0.0


class OracleLayer:
    """The oracle's own state machine for one layer (CPU, numpy)."""

    def __init__(self, B, n_tokens, C):
        self.t2s = np.full(n_tokens, -1, np.int32)
        self.s2t = np.full(B * C, -1, np.int32)
        self.theta = np.full(B, np.inf, np.float32)
        self.C = C


def check_scores(layer_inputs, q, w, gpu_scores, sample=None, rng=None):
    """fp64 oracle scores for all tokens (sample=None) or `sample` random tokens per request."""
    off, k8, ks = layer_inputs
    q8, qs, _ = orc.quantize_q(q, w)
    worst = 0.0
    for b in range(len(off) - 1):
        lo, hi = int(off[b]), int(off[b + 1])
        if hi == lo:
            continue
        if sample is None or hi - lo <= sample:
            tok = np.arange(lo, hi, dtype=np.int64)
        else:
            tok = np.sort(rng.choice(np.arange(lo, hi), sample, replace=False)).astype(np.int64)
        ref, ab = orc.scores(q8[b], qs[b], w[b], k8, ks, tok=tok)
        bad, rel = score_tolerance_ok(gpu_scores[tok], ref, ab)
        assert bad.size == 0, (b, tok[bad[:5]], gpu_scores[tok[bad[:5]]], ref[bad[:5]])
        worst = max(worst, rel)
    return worst


def run_decode(w: wl.Workload, steps: int, predictor: bool, cap: int = -1, score_sample=None,
               check_every_score_step=True, keys_device="cpu", layer: int = 0, resolved: bool = True,
               hold_early: bool = False, cands: bool = True, lazy: bool = False):
    """Runs `steps` decode steps of one layer on the GPU and checks each against the oracle."""
    dev = "cuda"
    off = wl.tok_offsets(w.lengths)
    k8c, ksc = wl.make_keys(w, layer, device=keys_device)
    k8 = k8c.cpu().numpy()
    ks = ksc.cpu().numpy()
    wt = wl.make_weights(w, layer, device=keys_device).cpu()
    host = wl.make_host_pool(w, layer, device=keys_device, pin=True)
    host_before = host.clone()
    lay = DecodeLayer(off, k8c.to(dev), ksc.to(dev), w.k, w.C, host, predictor=predictor, early_cap=cap,
                      resolved=resolved, hold_early=hold_early, cands=cands, lazy=lazy)
    o = OracleLayer(w.B, w.total_tokens, w.C)
    o_free = np.ones(w.B * w.C, np.uint8)   # lazy reuse: 1 = no resident token in the slot
    qsrc = wl.QueryStream(w, layer, device=keys_device)
    rng = np.random.default_rng(7)
    host_gpu = host.to(dev)
    report = dict(worst_rel=0.0, misses=[], early=[], boundary_max=0, revived=0)
    for t in range(steps):
        q = qsrc.next().cpu()
        theta_before = o.theta.copy()
        lay.step(q.to(dev), wt.to(dev))
        torch.cuda.synchronize()
        st = int(lay.status.item())
        assert st == 0, f"device status {st:#x} at step {t}"
        gs = lay.scores.cpu().numpy()[:max(w.total_tokens, 1)]
        if check_every_score_step or t in (0, 1, steps - 1):
            rel = check_scores((off, k8, ks), q.numpy(), wt.numpy(), gs, sample=score_sample, rng=rng)
            report["worst_rel"] = max(report["worst_rel"], rel)
        gh = lay.hist.cpu().numpy().view(np.uint32)
        g_sel = lay.sel_idx.cpu().numpy()
        g_slot = lay.sel_slot.cpu().numpy()
        g_kth = lay.kth.cpu().numpy()
        g_theta = lay.theta.cpu().numpy()
        g_t2s = lay.cache.tok2slot.cpu().numpy()[:w.total_tokens]
        g_s2t = lay.cache.slot2tok.cpu().numpy()
        g_fb = lay.cache.freebits.cpu().numpy().view(np.uint32)
        g_ecnt = lay.cache.early_cnt.cpu().numpy()
        g_etok = lay.cache.early_tok.cpu().numpy()
        g_eslot = lay.cache.early_slot.cpu().numpy()
        g_mcnt = lay.cache.miss_cnt.cpu().numpy()
        g_mtok = lay.cache.miss_tok.cpu().numpy()
        g_mslot = lay.cache.miss_slot.cpu().numpy()
        misses = 0
        for b in range(w.B):
            lo, hi = int(off[b]), int(off[b + 1])
            sc = gs[lo:hi]
            assert np.array_equal(gh[b], orc.hist256(sc, theta_before[b])), (t, b, "hist")
            t2s = o.t2s[lo:hi]
            s2t = o.s2t[b * w.C:(b + 1) * w.C]
            fr = o_free[b * w.C:(b + 1) * w.C]
            et = es = None
            if predictor:
                # the layer's cap: the caller's (holding: capped at C - k, the oracle's rule)
                assert lay.early_cap == (orc.early_cap_for(cap, w.C, w.k) if hold_early else cap)
                if lazy:
                    et, es = orc.lazy_early(sc, theta_before[b], lay.early_cap, t2s, s2t, fr)
                else:
                    et, es = orc.early_fetch(sc, theta_before[b], lay.early_cap, t2s, s2t)
                assert g_ecnt[b] == et.size, (t, b, "early count", g_ecnt[b], et.size)
                assert np.array_equal(g_etok[b * w.C:b * w.C + et.size], et), (t, b, "early tok")
                assert np.array_equal(g_eslot[b * w.C:b * w.C + et.size], es), (t, b, "early slot")
                report["early"].append(int(et.size))
            idx, kth = orc.topk(sc, w.k)
            assert np.array_equal(g_sel[b], idx), (t, b, "topk", np.nonzero(g_sel[b] != idx)[0][:5])
            assert g_kth[b] == np.float32(kth) or (math.isinf(kth) and math.isinf(g_kth[b])), (t, b, "kth")
            o.theta[b] = orc.ema(theta_before[b], kth, 0.5)
            assert g_theta[b] == o.theta[b] or (np.isinf(o.theta[b]) and np.isinf(g_theta[b])), \
                (t, b, "theta", g_theta[b], o.theta[b])
            if lazy:
                sel_slot, mt, ms, rev = orc.lazy_cache_step(idx, t2s, s2t, fr, et, es)
                report["revived"] += rev
            else:
                sel_slot, mt, ms, _ = orc.cache_step(idx, t2s, s2t, early_tok=et, hold_early=hold_early)
            assert np.array_equal(g_slot[b], sel_slot), (t, b, "sel_slot")
            assert g_mcnt[b] == mt.size, (t, b, "miss count", g_mcnt[b], mt.size)
            assert np.array_equal(g_mtok[b * w.C:b * w.C + mt.size], mt), (t, b, "miss tok")
            assert np.array_equal(g_mslot[b * w.C:b * w.C + mt.size], ms), (t, b, "miss slot")
            misses += mt.size
        assert np.array_equal(g_t2s, o.t2s), (t, "tok2slot")
        assert np.array_equal(g_s2t, o.s2t), (t, "slot2tok")
        free = (o_free.astype(bool) if lazy else (o.s2t < 0)).reshape(-1, 32)
        want_fb = (free.astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(1).astype(np.uint32)
        assert np.array_equal(g_fb, want_fb), (t, "freebits")
        # recalled bytes: every selected token's device row equals its host row
        sel_t = torch.from_numpy(g_sel).to(dev).long()
        slot_t = torch.from_numpy(g_slot).to(dev).long()
        valid = sel_t >= 0
        bidx = torch.arange(w.B, device=dev)[:, None].expand_as(sel_t)
        offs = torch.from_numpy(off[:-1]).to(dev)[:, None]
        rows_dev = lay.cache.dev_kv[(bidx * w.C + slot_t)[valid]]
        rows_host = host_gpu[(offs + sel_t)[valid]]
        assert torch.equal(rows_dev.view(torch.int16), rows_host.view(torch.int16)), (t, "recall bytes")
        if lazy:  # every present token's bytes, ghosts' included, are its host row
            for b in range(w.B):
                lo, hi = int(off[b]), int(off[b + 1])
                pres = np.nonzero(o.t2s[lo:hi] >= 0)[0]
                sl_t = torch.from_numpy(b * w.C + o.t2s[lo:hi][pres]).long().to(dev)
                tk_t = torch.from_numpy(lo + pres).long().to(dev)
                assert torch.equal(lay.cache.dev_kv[sl_t].view(torch.int16), host_gpu[tk_t].view(torch.int16)), \
                    (t, b, "present rows")
        report["misses"].append(misses)
    report["boundary_max"] = int(lay.stats[L.STAT_BOUNDARY_MAX].item())
    report["fallbacks"] = int(lay.stats[L.STAT_TOPK_FALLBACK].item())
    report["cand_miss"] = int(lay.stats[L.STAT_CAND_MISS].item())
    report["revived_gpu"] = int(lay.stats[L.STAT_REVIVED].item())
    assert torch.equal(host.view(torch.int16), host_before.view(torch.int16))  # no write-back
    return report


def run_decode_growing(w: wl.Workload, steps: int, room: int, hold_early: bool = False, seed: int = 5):
    """Decode steps on growing contexts: request b's region holds its w.lengths[b] tokens plus `room`
    free rows; after each step one new token per request is appended (GPU: echo_append_tokens; the
    oracle: its own append on its own copies of the keys, the host pool and the tables).  Every step
    is checked as in run_decode over each request's current tokens, and every append bit-exactly."""
    dev = "cuda"
    lens = np.asarray(w.lengths, np.int64)
    off = np.concatenate([[0], np.cumsum(lens + room)]).astype(np.int64)
    n = int(off[-1])
    end = off[:-1] + lens
    big = wl.scaled(w, w.name + "_room", lengths=tuple(int(x) for x in lens + room))
    k8c, ksc = wl.make_keys(big, 0)
    wt = wl.make_weights(big, 0).cpu()
    host = wl.make_host_pool(big, 0, pin=True)
    # the rows after each request's end are not tokens yet
    k8 = k8c.numpy().copy()
    ks = ksc.numpy().copy()
    for b in range(w.B):
        k8[end[b]:off[b + 1]] = 0
        ks[end[b]:off[b + 1]] = 0
        host[end[b]:off[b + 1]] = 0
    lay = DecodeLayer(off, torch.from_numpy(k8).to(dev), torch.from_numpy(ks).to(dev), w.k, w.C, host,
                      hold_early=hold_early, tok_end=torch.from_numpy(end), device=dev)
    o = OracleLayer(w.B, n, w.C)
    o_end = end.copy()
    o_host = host.view(torch.uint8).numpy().copy()
    o_dev = np.zeros((w.B * w.C, o_host.shape[1]), np.uint8)
    qsrc = wl.QueryStream(big, 0)
    rng = np.random.default_rng(seed)
    for t in range(steps):
        q = qsrc.next().cpu()
        theta_before = o.theta.copy()
        lay.step(q.to(dev), wt.to(dev))
        torch.cuda.synchronize()
        assert int(lay.status.item()) == 0, f"status {int(lay.status.item()):#x} at step {t}"
        gs = lay.scores.cpu().numpy()
        g_sel, g_slot, g_kth = lay.sel_idx.cpu().numpy(), lay.sel_slot.cpu().numpy(), lay.kth.cpu().numpy()
        q8, qs, _ = orc.quantize_q(q.numpy(), wt.numpy())
        for b in range(w.B):
            lo, hi = int(off[b]), int(o_end[b])
            tok = np.arange(lo, hi, dtype=np.int64)
            ref, ab = orc.scores(q8[b], qs[b], wt.numpy()[b], k8, ks, tok=tok)
            bad, _ = score_tolerance_ok(gs[lo:hi], ref, ab)
            assert bad.size == 0, (t, b, "scores")
            sc = gs[lo:hi]
            t2s = o.t2s[lo:hi]
            s2t = o.s2t[b * w.C:(b + 1) * w.C]
            et, _ = orc.early_fetch(sc, theta_before[b], lay.early_cap, t2s, s2t)
            idx, kth = orc.topk(sc, w.k)
            assert np.array_equal(g_sel[b], idx), (t, b, "topk")
            assert g_kth[b] == np.float32(kth), (t, b, "kth")
            o.theta[b] = orc.ema(theta_before[b], kth, 0.5)
            sel_slot, mt, ms, _ = orc.cache_step(idx, t2s, s2t, early_tok=et, hold_early=hold_early)
            assert np.array_equal(g_slot[b], sel_slot), (t, b, "sel_slot")
            orc.recall(o_host[lo:hi], mt, ms, o_dev[b * w.C:(b + 1) * w.C])
            valid = idx >= 0
            o_dev[b * w.C + sel_slot[valid]] = o_host[lo + idx[valid]]
        assert np.array_equal(lay.cache.tok2slot.cpu().numpy(), o.t2s), (t, "tok2slot")
        assert np.array_equal(lay.cache.slot2tok.cpu().numpy(), o.s2t), (t, "slot2tok")
        # every selected token's device row is its host row
        g_dev = lay.cache.dev_kv.view(torch.uint8).cpu().numpy().reshape(w.B * w.C, -1)
        for b in range(w.B):
            v = g_slot[b] >= 0
            assert np.array_equal(g_dev[b * w.C + g_slot[b][v]], o_host[off[b] + g_sel[b][v]]), (t, b, "rows")
        # ---- append one token per request
        k_new = rng.standard_normal((w.B, L.DIM), dtype=np.float32)
        kv_new = rng.integers(-2**15, 2**15, (w.B, o_host.shape[1] // 2), dtype=np.int16)
        lay.append(torch.from_numpy(k_new).to(dev), torch.from_numpy(kv_new).to(dev))
        torch.cuda.synchronize()
        full = orc.append_tokens(off, o_end, k_new, kv_new.view(np.uint8), k8, ks, o_host, w.C, o.t2s, o.s2t,
                                 o_dev)
        want = L.ST_FULL if full.any() else 0
        assert int(lay.status.item()) == want, (t, "append status")
        lay.status.zero_()
        assert np.array_equal(lay.tok_end.cpu().numpy(), o_end), (t, "tok_end")
        assert np.array_equal(lay.k8.cpu().numpy(), k8) and np.array_equal(lay.ks.cpu().numpy(), ks), (t, "keys")
        assert np.array_equal(host.view(torch.uint8).numpy(), o_host), (t, "host pool")
        assert np.array_equal(lay.cache.tok2slot.cpu().numpy(), o.t2s), (t, "append tok2slot")
        assert np.array_equal(lay.cache.slot2tok.cpu().numpy(), o.s2t), (t, "append slot2tok")
    return o_end - end


def run_stack(w: wl.Workload, steps: int, n_layers: int, cross_layer: bool, hold_early: bool = False,
              graph: bool = True, keys_device: str = "cpu", predictor: bool = True, score_steps=None,
              score_sample: int = 64, threads: int = 1):
    """A DecodeStack of n_layers layers (each its own keys, weights, queries, host pool and cache),
    optionally captured as one CUDA graph; every step of every layer is checked against the oracle:
    layer 0's early set by the threshold predictor, the others' (cross_layer) from the previous
    layer's selection.  Per step and layer: histograms, early lists, top-k, k-th scores, thresholds,
    slots, miss lists, tables, free bits and the rows of every selected token, bit-exact; fp64
    scores of score_sample tokens per request on the steps in score_steps (None: every step).
    threads: the oracle's per-request work in parallel (its C calls release the interpreter).
    Returns the per-layer early counts and misses per step."""
    from concurrent.futures import ThreadPoolExecutor

    from sparse_attention_kv_echo_gb300 import DecodeStack
    dev = "cuda"
    off = wl.tok_offsets(w.lengths)
    lays, inputs, qsrcs, hosts, orcs = [], [], [], [], []
    for l in range(n_layers):
        k8c, ksc = wl.make_keys(w, l, device=keys_device)
        wt = wl.make_weights(w, l, device=keys_device).cpu()
        host = wl.make_host_pool(w, l, device=keys_device, pin=True)
        lays.append(DecodeLayer(off, k8c.to(dev), ksc.to(dev), w.k, w.C, host, hold_early=hold_early,
                                predictor=predictor, cross_layer=cross_layer and l > 0, device=dev))
        inputs.append((k8c.cpu().numpy(), ksc.cpu().numpy(), wt.numpy()))
        qsrcs.append(wl.QueryStream(w, l, device=keys_device))
        hosts.append(host.to(dev))
        orcs.append(OracleLayer(w.B, w.total_tokens, w.C))
        del k8c, ksc
    stack = DecodeStack(lays, cross_layer=cross_layer)
    main = torch.cuda.Stream()
    for l, lay in enumerate(lays):
        with torch.cuda.stream(main):
            lay.w_in.copy_(torch.from_numpy(inputs[l][2]).to(dev))
    torch.cuda.synchronize()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            stack.step([lay.q_in for lay in lays], [lay.w_in for lay in lays], stream=main)
        torch.cuda.synchronize()
        for lay in lays:
            lay.reset()
        torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    report = dict(early=[[] for _ in lays], misses=[[] for _ in lays])
    pool = ThreadPoolExecutor(max_workers=max(1, threads))
    for t in range(steps):
        qs = [qsrcs[l].next().cpu() for l in range(n_layers)]
        with torch.cuda.stream(main):
            for l, lay in enumerate(lays):
                lay.q_in.copy_(qs[l].to(dev))
            if graph:
                g.replay()
            else:
                stack.step([lay.q_in for lay in lays], [lay.w_in for lay in lays], stream=main)
        torch.cuda.synchronize()
        prev_sel = None   # the oracle's own selection of the layer before
        for l, lay in enumerate(lays):
            assert int(lay.status.item()) == 0, (t, l, "status")
            o = orcs[l]
            k8, ks, wt = inputs[l]
            gs = lay.scores.cpu().numpy()
            if score_steps is None or t in score_steps:
                check_scores((off, k8, ks), qs[l].numpy(), wt, gs, sample=score_sample, rng=rng)
            gh = lay.hist.cpu().numpy().view(np.uint32)
            g_sel, g_slot = lay.sel_idx.cpu().numpy(), lay.sel_slot.cpu().numpy()
            g_kth = lay.kth.cpu().numpy()
            g_theta = lay.theta.cpu().numpy()
            g_ecnt = lay.cache.early_cnt.cpu().numpy()
            g_etok, g_eslot = lay.cache.early_tok.cpu().numpy(), lay.cache.early_slot.cpu().numpy()
            g_mcnt = lay.cache.miss_cnt.cpu().numpy()
            g_mtok, g_mslot = lay.cache.miss_tok.cpu().numpy(), lay.cache.miss_slot.cpu().numpy()
            theta_before = o.theta.copy()

            def one(b):
                lo, hi = int(off[b]), int(off[b + 1])
                sc = gs[lo:hi]
                t2s = o.t2s[lo:hi]
                s2t = o.s2t[b * w.C:(b + 1) * w.C]
                assert np.array_equal(gh[b], orc.hist256(sc, theta_before[b])), (t, l, b, "hist")
                et = None
                if cross_layer and l > 0:
                    et, es = orc.early_from_selection(prev_sel[b], hi - lo, lay.early_cap, t2s, s2t)
                elif predictor:
                    et, es = orc.early_fetch(sc, theta_before[b], lay.early_cap, t2s, s2t)
                if et is not None:
                    assert g_ecnt[b] == et.size, (t, l, b, "early count", g_ecnt[b], et.size)
                    assert np.array_equal(g_etok[b * w.C:b * w.C + et.size], et), (t, l, b, "early tok")
                    assert np.array_equal(g_eslot[b * w.C:b * w.C + et.size], es), (t, l, b, "early slot")
                idx, kth = orc.topk(sc, w.k)
                assert np.array_equal(g_sel[b], idx), (t, l, b, "topk")
                assert g_kth[b] == np.float32(kth) or (math.isinf(kth) and math.isinf(g_kth[b])), (t, l, b, "kth")
                o.theta[b] = orc.ema(theta_before[b], kth, 0.5)
                assert g_theta[b] == o.theta[b] or (np.isinf(o.theta[b]) and np.isinf(g_theta[b])), \
                    (t, l, b, "theta")
                sel_slot, mt, ms, _ = orc.cache_step(idx, t2s, s2t, early_tok=et, hold_early=hold_early)
                assert np.array_equal(g_slot[b], sel_slot), (t, l, b, "sel_slot")
                assert g_mcnt[b] == mt.size, (t, l, b, "miss count")
                assert np.array_equal(g_mtok[b * w.C:b * w.C + mt.size], mt), (t, l, b, "miss tok")
                assert np.array_equal(g_mslot[b * w.C:b * w.C + mt.size], ms), (t, l, b, "miss slot")
                return idx, 0 if et is None else int(et.size), int(mt.size)

            res = list(pool.map(one, range(w.B)))
            o_sel = [r[0] for r in res]
            for r in res:
                report["early"][l].append(r[1])
            report["misses"][l].append(sum(r[2] for r in res))
            assert np.array_equal(lay.cache.tok2slot.cpu().numpy()[:w.total_tokens], o.t2s), (t, l, "tok2slot")
            assert np.array_equal(lay.cache.slot2tok.cpu().numpy(), o.s2t), (t, l, "slot2tok")
            free = (o.s2t < 0).reshape(-1, 32)
            want_fb = (free.astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(1).astype(np.uint32)
            assert np.array_equal(lay.cache.freebits.cpu().numpy().view(np.uint32), want_fb), (t, l, "freebits")
            # every selected token's device row is its host row (compared on the device)
            sel_t = torch.from_numpy(g_sel).to(dev).long()
            slot_t = torch.from_numpy(g_slot).to(dev).long()
            valid = sel_t >= 0
            bidx = torch.arange(w.B, device=dev)[:, None].expand_as(sel_t)
            offs = torch.from_numpy(off[:-1]).to(dev)[:, None]
            rows_dev = lay.cache.dev_kv[(bidx * w.C + slot_t)[valid]]
            rows_host = hosts[l][(offs + sel_t)[valid]]
            assert torch.equal(rows_dev.view(torch.int16), rows_host.view(torch.int16)), (t, l, "rows")
            prev_sel = o_sel
    pool.shutdown()
    report["cand_miss"] = [int(lay.stats[L.STAT_CAND_MISS].item()) for lay in lays]
    report["fallbacks"] = [int(lay.stats[L.STAT_TOPK_FALLBACK].item()) for lay in lays]
    return report


def run_pool(w: wl.Workload, steps: int, pool: int, hold_early: bool = False, predictor: bool = True,
             graph: bool = True, cap: int = -1, lazy: bool = False):
    """Decode steps with one cache pool of `pool` slots shared by the batch's requests, checked
    against the oracle's own pool (a cache of one request over every row, token ids global): the
    early set (the requests' marked, non-resident tokens in (request, token) order), top-k per
    request, the pool step on the batch's selection in (request, token) order, tables, rows."""
    dev = "cuda"
    off = wl.tok_offsets(w.lengths)
    n = w.total_tokens
    k8c, ksc = wl.make_keys(w, 0)
    wt = wl.make_weights(w, 0)
    host = wl.make_host_pool(w, 0, pin=True)
    lay = DecodeLayer(off, k8c.to(dev), ksc.to(dev), w.k, w.C, host, predictor=predictor, hold_early=hold_early,
                      early_cap=cap, pool_slots=pool, lazy=lazy, device=dev)
    k8, ks, wn = k8c.numpy(), ksc.numpy(), wt.numpy()
    hb = host.view(torch.uint8).numpy()
    t2s = np.full(n, -1, np.int32)
    s2t = np.full(pool, -1, np.int32)
    fr = np.ones(pool, np.uint8)      # lazy reuse: 1 = no resident token in the slot
    theta = np.full(w.B, np.inf, np.float32)
    qsrc = wl.QueryStream(w, 0)
    main = torch.cuda.Stream()
    with torch.cuda.stream(main):
        lay.w_in.copy_(wt.to(dev))
    torch.cuda.synchronize()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            lay.step(stream=main)
        torch.cuda.synchronize()
        lay.reset()
        torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    report = dict(early=[], misses=[], revived=0)
    for t in range(steps):
        q = qsrc.next().cpu()
        with torch.cuda.stream(main):
            lay.q_in.copy_(q.to(dev))
            if graph:
                g.replay()
            else:
                lay.step(stream=main)
        torch.cuda.synchronize()
        assert int(lay.status.item()) == 0, (t, "status")
        gs = lay.scores.cpu().numpy()
        check_scores((off, k8, ks), q.numpy(), wn, gs, sample=64, rng=rng)
        # the early set: every request's tokens above its threshold, not in the pool, in global order
        marked = []
        for b in range(w.B):
            lo, hi = int(off[b]), int(off[b + 1])
            if predictor and np.isfinite(theta[b]):
                s = np.nonzero(gs[lo:hi] > theta[b])[0] + lo
                marked.extend(int(x) for x in s if t2s[x] < 0)
        if lazy:   # the marked tokens, ascending, through the lazy early rule
            ind = np.zeros(n, np.float32)
            ind[np.array(marked, np.int64)] = 1.0
            et, es = orc.lazy_early(ind, 0.5, lay.early_cap, t2s, s2t, fr)
        else:
            et, es = orc.early_from_selection(np.array(marked, np.int32), n, lay.early_cap, t2s, s2t)
        if predictor:
            g_cnt = int(lay.cache.early_cnt.cpu().numpy()[0])
            assert g_cnt == et.size, (t, "early count", g_cnt, et.size)
            assert np.array_equal(lay.cache.early_tok.cpu().numpy()[:g_cnt], et), (t, "early tok")
            assert np.array_equal(lay.cache.early_slot.cpu().numpy()[:g_cnt], es), (t, "early slot")
        g_sel, g_slot = lay.sel_idx.cpu().numpy(), lay.sel_slot.cpu().numpy()
        glob, counts = [], []
        for b in range(w.B):
            lo, hi = int(off[b]), int(off[b + 1])
            idx, kth = orc.topk(gs[lo:hi], w.k)
            assert np.array_equal(g_sel[b], idx), (t, b, "topk")
            theta[b] = orc.ema(theta[b], kth, 0.5)
            v = idx[idx >= 0]
            glob.extend(int(x) + lo for x in v)
            counts.append(v.size)
        sel_g = np.full(w.B * w.k, -1, np.int32)
        sel_g[:len(glob)] = glob
        if lazy:
            sl_g, mt, ms, rev = orc.lazy_cache_step(sel_g, t2s, s2t, fr, et, es)
            report["revived"] += rev
        else:
            sl_g, mt, ms, _ = orc.cache_step(sel_g, t2s, s2t, early_tok=et, hold_early=hold_early)
        pos = 0
        for b in range(w.B):
            want = np.full(w.k, -1, np.int32)
            want[:counts[b]] = sl_g[pos:pos + counts[b]]
            pos += counts[b]
            assert np.array_equal(g_slot[b], want), (t, b, "sel_slot")
        assert np.array_equal(lay.cache.tok2slot.cpu().numpy(), t2s), (t, "pool tok2slot")
        assert np.array_equal(lay.cache.slot2tok.cpu().numpy(), s2t), (t, "pool slot2tok")
        g_dev = lay.cache.dev_kv.view(torch.uint8).cpu().numpy()
        valid = sel_g >= 0
        assert np.array_equal(g_dev[sl_g[valid]], hb[sel_g[valid]]), (t, "rows")
        if lazy:   # ghosts' bytes too, and the free bits
            pres = np.nonzero(t2s >= 0)[0]
            assert np.array_equal(g_dev[t2s[pres]], hb[pres]), (t, "present rows")
            want_fb = (fr.astype(bool).reshape(-1, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(1)
            assert np.array_equal(lay.cache.freebits.cpu().numpy().view(np.uint32), want_fb.astype(np.uint32)), \
                (t, "pool freebits")
        report["early"].append(int(et.size))
        report["misses"].append(int(mt.size))
    return report
