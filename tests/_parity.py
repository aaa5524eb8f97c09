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
               hold_early: bool = False):
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
                      resolved=resolved, hold_early=hold_early)
    o = OracleLayer(w.B, w.total_tokens, w.C)
    qsrc = wl.QueryStream(w, layer, device=keys_device)
    rng = np.random.default_rng(7)
    host_gpu = host.to(dev)
    report = dict(worst_rel=0.0, misses=[], early=[], boundary_max=0)
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
            et = None
            if predictor:
                # the layer's cap: the caller's (holding: capped at C - k, the oracle's rule)
                assert lay.early_cap == (orc.early_cap_for(cap, w.C, w.k) if hold_early else cap)
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
            sel_slot, mt, ms, _ = orc.cache_step(idx, t2s, s2t, early_tok=et, hold_early=hold_early)
            assert np.array_equal(g_slot[b], sel_slot), (t, b, "sel_slot")
            assert g_mcnt[b] == mt.size, (t, b, "miss count", g_mcnt[b], mt.size)
            assert np.array_equal(g_mtok[b * w.C:b * w.C + mt.size], mt), (t, b, "miss tok")
            assert np.array_equal(g_mslot[b * w.C:b * w.C + mt.size], ms), (t, b, "miss slot")
            misses += mt.size
        assert np.array_equal(g_t2s, o.t2s), (t, "tok2slot")
        assert np.array_equal(g_s2t, o.s2t), (t, "slot2tok")
        free = (o.s2t < 0).reshape(-1, 32)
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
        report["misses"].append(misses)
    report["boundary_max"] = int(lay.stats[L.STAT_BOUNDARY_MAX].item())
    report["fallbacks"] = int(lay.stats[L.STAT_TOPK_FALLBACK].item())
    assert torch.equal(host.view(torch.int16), host_before.view(torch.int16))  # no write-back
    return report
