"""CPU oracle for the ECHO decode hot path -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never imports,
links or calls it; the two share no code.  The arithmetic lives in
``echo_oracle.cpp`` (plain C++, fp64 scores, stable-sort top-k, map/set
cache); this module compiles it with g++ and wraps it with ctypes, with
argument marshalling only.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "echo_oracle.cpp")
_LIB = os.path.join(_HERE, "libecho_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ECAPACITY, ENAN = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle shared library (g++, no fp contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-ffp-contract=off", "-pthread",
               _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _p(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct)) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            c_i64p = ctypes.POINTER(ctypes.c_int64)
            c_i32p = ctypes.POINTER(ctypes.c_int32)
            c_u32p = ctypes.POINTER(ctypes.c_uint32)
            c_u8p = ctypes.POINTER(ctypes.c_uint8)
            c_f32p = ctypes.POINTER(ctypes.c_float)
            c_f64p = ctypes.POINTER(ctypes.c_double)
            c_u16p = ctypes.POINTER(ctypes.c_uint16)
            L.orc_bf16_value.restype = ctypes.c_double
            L.orc_bf16_value.argtypes = [ctypes.c_uint16]
            L.orc_mla_decode.restype = ctypes.c_int
            L.orc_mla_decode.argtypes = [c_u16p, ctypes.c_int, c_u16p, ctypes.c_int64, c_i32p, ctypes.c_int,
                                         ctypes.c_double, c_f64p, c_f64p, c_f64p]
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [ctypes.c_double]
            L.orc_e4m3_encode_f32.restype = None
            L.orc_e4m3_encode_f32.argtypes = [c_f32p, ctypes.c_int64, c_u8p]
            L.orc_order_key.restype = ctypes.c_uint32
            L.orc_order_key.argtypes = [ctypes.c_float]
            L.orc_quantize_q.restype = ctypes.c_int
            L.orc_quantize_q.argtypes = [c_f32p, c_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         c_u8p, c_f32p, c_f32p]
            L.orc_scores.restype = None
            L.orc_scores.argtypes = [c_u8p, c_f32p, c_f32p, ctypes.c_int, ctypes.c_int, c_u8p,
                                     c_f32p, c_i64p, ctypes.c_int64, c_f64p, c_f64p]
            L.orc_hist256.restype = None
            L.orc_hist256.argtypes = [c_f32p, ctypes.c_int64, ctypes.c_float, c_u32p]
            L.orc_topk.restype = ctypes.c_int
            L.orc_topk.argtypes = [c_f32p, ctypes.c_int64, ctypes.c_int, c_i32p, c_f32p]
            L.orc_ema.restype = ctypes.c_float
            L.orc_ema.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_float]
            L.orc_early_fetch.restype = ctypes.c_int
            L.orc_early_fetch.argtypes = [ctypes.c_int64, ctypes.c_int, c_f32p, ctypes.c_float,
                                          ctypes.c_int, c_i32p, c_i32p, c_i32p, c_i32p, c_i32p]
            L.orc_cache_step.restype = ctypes.c_int
            L.orc_cache_step.argtypes = [ctypes.c_int64, ctypes.c_int, c_i32p, c_i32p, c_i32p,
                                         ctypes.c_int, c_i32p, ctypes.c_int32, ctypes.c_int, c_i32p, c_i32p,
                                         c_i32p, c_i32p, c_i32p]
            L.orc_lazy_early.restype = ctypes.c_int
            L.orc_lazy_early.argtypes = [ctypes.c_int64, ctypes.c_int, c_f32p, ctypes.c_float, ctypes.c_int,
                                         c_i32p, c_i32p, c_u8p, c_i32p, c_i32p, c_i32p]
            L.orc_lazy_cache_step.restype = ctypes.c_int
            L.orc_lazy_cache_step.argtypes = [ctypes.c_int64, ctypes.c_int, c_i32p, c_i32p, c_u8p, c_i32p,
                                              ctypes.c_int, c_i32p, c_i32p, ctypes.c_int32, c_i32p, c_i32p,
                                              c_i32p, c_i32p, c_i32p]
            L.orc_early_cap_for.restype = ctypes.c_int
            L.orc_early_cap_for.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
            L.orc_recall.restype = None
            L.orc_recall.argtypes = [c_u8p, ctypes.c_int64, c_i32p, c_i32p, ctypes.c_int32, c_u8p]
            L.orc_prefill_rows.restype = ctypes.c_int
            L.orc_prefill_rows.argtypes = [c_f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
                                           ctypes.c_int, ctypes.c_float, c_i32p, c_f32p, c_u32p,
                                           c_u8p]
            L.orc_early_from_selection.restype = ctypes.c_int
            L.orc_early_from_selection.argtypes = [ctypes.c_int64, ctypes.c_int, c_i32p, ctypes.c_int,
                                                   ctypes.c_int, c_i32p, c_i32p, c_i32p, c_i32p, c_i32p]
            L.orc_append_tokens.restype = ctypes.c_int
            L.orc_append_tokens.argtypes = [ctypes.c_int, c_i64p, c_i64p, c_f32p, ctypes.c_int, c_u8p,
                                            ctypes.c_int64, c_u8p, c_f32p, c_u8p, ctypes.c_int, c_i32p, c_i32p,
                                            c_u8p, c_i32p]
            L.orc_decode_step.restype = ctypes.c_int
            L.orc_decode_step.argtypes = [
                ctypes.c_int, c_i64p, c_f32p, c_f32p, ctypes.c_int, ctypes.c_int, c_u8p, c_f32p,
                ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, c_f32p, ctypes.c_int,
                c_i32p, c_i32p, c_u8p, ctypes.c_int64, c_u8p, c_i32p, c_i32p, c_f32p, c_i32p,
                c_f32p, ctypes.c_int]
            _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


class OracleError(RuntimeError):
    def __init__(self, rc, what):
        super().__init__(f"{what}: oracle return code {rc}")
        self.rc = rc


def _check(rc, what):
    if rc != OK:
        raise OracleError(rc, what)


# ---- thin wrappers (numpy in, numpy out) ------------------------------------

def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code) & 0xFF)


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(x) -> np.ndarray:
    x = _c(x, np.float32).reshape(-1)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_f32(_p(x, ctypes.c_float), x.size, _p(out, ctypes.c_uint8))
    return out


def order_key(x: float) -> int:
    return int(lib().orc_order_key(float(x)))


def quantize_q(q, w):
    """q [B,H,D] f32, w [B,H] f32 -> (q8 [B,H,D] u8, qscale [B,H] f32, wfold [B,H] f32)."""
    q = _c(q, np.float32)
    w = _c(w, np.float32)
    B, H, D = q.shape
    q8 = np.empty((B, H, D), np.uint8)
    qs = np.empty((B, H), np.float32)
    wf = np.empty((B, H), np.float32)
    rc = lib().orc_quantize_q(_p(q, ctypes.c_float), _p(w, ctypes.c_float), B, H, D,
                              _p(q8, ctypes.c_uint8), _p(qs, ctypes.c_float), _p(wf, ctypes.c_float))
    _check(rc, "quantize_q")
    return q8, qs, wf


def scores(q8, qscale, w, k8, ks, tok=None):
    """fp64 indexer scores of one request: q8 [H,D], qscale [H], w [H], keys k8 [*,D], ks [*].

    tok (int64 array) picks the key rows to score; None scores every row.
    Returns (scores [n] f64, absbound [n] f64)."""
    q8 = _c(q8, np.uint8)
    qscale = _c(qscale, np.float32)
    w = _c(w, np.float32)
    k8 = _c(k8, np.uint8)
    ks = _c(ks, np.float32)
    H, D = q8.shape
    if tok is None:
        n = k8.shape[0]
        tp = None
    else:
        tok = _c(tok, np.int64)
        n = tok.size
        tp = _p(tok, ctypes.c_int64)
    out = np.empty(n, np.float64)
    ab = np.empty(n, np.float64)
    lib().orc_scores(_p(q8, ctypes.c_uint8), _p(qscale, ctypes.c_float), _p(w, ctypes.c_float), H, D,
                     _p(k8, ctypes.c_uint8), _p(ks, ctypes.c_float), tp, n,
                     _p(out, ctypes.c_double), _p(ab, ctypes.c_double))
    return out, ab


def hist256(scores_f32, theta: float) -> np.ndarray:
    s = _c(scores_f32, np.float32).reshape(-1)
    h = np.empty(256, np.uint32)
    lib().orc_hist256(_p(s, ctypes.c_float), s.size, float(theta), _p(h, ctypes.c_uint32))
    return h


def topk(scores_f32, k: int):
    """-> (idx [k] int32 ascending, -1 padded; kth float)."""
    s = _c(scores_f32, np.float32).reshape(-1)
    idx = np.empty(k, np.int32)
    kth = ctypes.c_float()
    rc = lib().orc_topk(_p(s, ctypes.c_float), s.size, int(k), _p(idx, ctypes.c_int32),
                        ctypes.byref(kth))
    _check(rc, "topk")
    return idx, kth.value


def ema(theta: float, kth: float, alpha: float) -> float:
    return lib().orc_ema(float(theta), float(kth), float(alpha))


def early_fetch(scores_f32, theta: float, cap: int, tok2slot, slot2tok):
    """Updates tok2slot/slot2tok (numpy int32, in place); -> (early_tok, early_slot)."""
    s = _c(scores_f32, np.float32).reshape(-1)
    assert tok2slot.dtype == np.int32 and slot2tok.dtype == np.int32
    assert tok2slot.flags.c_contiguous and slot2tok.flags.c_contiguous
    n, C = s.size, slot2tok.size
    et = np.empty(max(C, 1), np.int32)
    es = np.empty(max(C, 1), np.int32)
    cnt = ctypes.c_int32()
    rc = lib().orc_early_fetch(n, C, _p(s, ctypes.c_float), float(theta), int(cap),
                               _p(tok2slot, ctypes.c_int32), _p(slot2tok, ctypes.c_int32),
                               _p(et, ctypes.c_int32), _p(es, ctypes.c_int32), ctypes.byref(cnt))
    _check(rc, "early_fetch")
    return et[:cnt.value].copy(), es[:cnt.value].copy()


def early_from_selection(prev_sel, n: int, cap: int, tok2slot, slot2tok):
    """Cross-layer early fetch (the layer-to-layer prefetch, as read here): the previous layer's selection prev_sel
    [m] (-1 padded) minus this layer's residents, ascending, <= min(cap, free).  Updates
    tok2slot [n] / slot2tok [C] (numpy int32, in place); -> (early_tok, early_slot)."""
    sel = _c(prev_sel, np.int32).reshape(-1)
    assert tok2slot.dtype == np.int32 and slot2tok.dtype == np.int32
    assert tok2slot.flags.c_contiguous and slot2tok.flags.c_contiguous and tok2slot.size == n
    C = slot2tok.size
    et = np.empty(max(C, 1), np.int32)
    es = np.empty(max(C, 1), np.int32)
    cnt = ctypes.c_int32()
    rc = lib().orc_early_from_selection(int(n), C, _p(sel, ctypes.c_int32), sel.size, int(cap),
                                        _p(tok2slot, ctypes.c_int32), _p(slot2tok, ctypes.c_int32),
                                        _p(et, ctypes.c_int32), _p(es, ctypes.c_int32), ctypes.byref(cnt))
    _check(rc, "early_from_selection")
    return et[:cnt.value].copy(), es[:cnt.value].copy()


def lazy_early(scores_f32, theta: float, cap: int, tok2slot, slot2tok, free):
    """The early set under lazy-reuse eviction (nothing updated): tokens above theta that are
    not present, ascending, <= min(cap, free slots), with the lowest free slots.  free: uint8
    [C], 1 = the slot holds no resident token.  -> (early_tok, early_slot)."""
    s = _c(scores_f32, np.float32).reshape(-1)
    for a, dt in ((tok2slot, np.int32), (slot2tok, np.int32), (free, np.uint8)):
        assert a.dtype == dt and a.flags.c_contiguous
    n, C = s.size, slot2tok.size
    et = np.empty(max(C, 1), np.int32)
    es = np.empty(max(C, 1), np.int32)
    cnt = ctypes.c_int32()
    rc = lib().orc_lazy_early(n, C, _p(s, ctypes.c_float), float(theta), int(cap), _p(tok2slot, ctypes.c_int32),
                              _p(slot2tok, ctypes.c_int32), _p(free, ctypes.c_uint8), _p(et, ctypes.c_int32),
                              _p(es, ctypes.c_int32), ctypes.byref(cnt))
    _check(rc, "lazy_early")
    return et[:cnt.value].copy(), es[:cnt.value].copy()


def lazy_cache_step(sel, tok2slot, slot2tok, free, early_tok=None, early_slot=None):
    """The cache step under lazy-reuse eviction; updates tok2slot, slot2tok and free (uint8 [C])
    in place.  -> (sel_slot, miss_tok, miss_slot, revived)."""
    sel = _c(sel, np.int32).reshape(-1)
    et = _c(np.zeros(0, np.int32) if early_tok is None else early_tok, np.int32).reshape(-1)
    es = _c(np.zeros(0, np.int32) if early_slot is None else early_slot, np.int32).reshape(-1)
    assert et.size == es.size
    for a, dt in ((tok2slot, np.int32), (slot2tok, np.int32), (free, np.uint8)):
        assert a.dtype == dt and a.flags.c_contiguous
    n, C, m = tok2slot.size, slot2tok.size, sel.size
    sel_slot = np.empty(max(m, 1), np.int32)
    mt = np.empty(max(C, 1), np.int32)
    ms = np.empty(max(C, 1), np.int32)
    nm, nr = ctypes.c_int32(), ctypes.c_int32()
    rc = lib().orc_lazy_cache_step(n, C, _p(tok2slot, ctypes.c_int32), _p(slot2tok, ctypes.c_int32),
                                   _p(free, ctypes.c_uint8), _p(sel, ctypes.c_int32), m, _p(et, ctypes.c_int32),
                                   _p(es, ctypes.c_int32), et.size, _p(sel_slot, ctypes.c_int32),
                                   _p(mt, ctypes.c_int32), _p(ms, ctypes.c_int32), ctypes.byref(nm),
                                   ctypes.byref(nr))
    _check(rc, "lazy_cache_step")
    return sel_slot[:m].copy(), mt[:nm.value].copy(), ms[:nm.value].copy(), nr.value


def early_cap_for(cap: int, C: int, k: int) -> int:
    """The early-set cap of the held-slot variant of a decode step with selection width k
    (C - k on top of cap)."""
    return int(lib().orc_early_cap_for(int(cap), int(C), int(k)))


def cache_step(sel, tok2slot, slot2tok, early_tok=None, hold_early=False):
    """Updates the tables in place; early_tok: the tokens this step's early fetch made
    resident; hold_early: the held-slot variant (their slots are held through the miss
    placement).  -> (sel_slot, miss_tok, miss_slot, nfreed)."""
    sel = _c(sel, np.int32).reshape(-1)
    et = _c(np.zeros(0, np.int32) if early_tok is None else early_tok, np.int32).reshape(-1)
    assert tok2slot.dtype == np.int32 and slot2tok.dtype == np.int32
    n, C, m = tok2slot.size, slot2tok.size, sel.size
    sel_slot = np.empty(m, np.int32)
    mt = np.empty(max(m, 1), np.int32)
    ms = np.empty(max(m, 1), np.int32)
    nm = ctypes.c_int32()
    nf = ctypes.c_int32()
    rc = lib().orc_cache_step(n, C, _p(tok2slot, ctypes.c_int32), _p(slot2tok, ctypes.c_int32),
                              _p(sel, ctypes.c_int32), m, _p(et, ctypes.c_int32) if et.size else None,
                              et.size, int(bool(hold_early)), _p(sel_slot, ctypes.c_int32),
                              _p(mt, ctypes.c_int32), _p(ms, ctypes.c_int32), ctypes.byref(nm),
                              ctypes.byref(nf))
    _check(rc, "cache_step")
    return sel_slot, mt[:nm.value].copy(), ms[:nm.value].copy(), nf.value


def recall(host_rows, tok, slot, dev_rows):
    """host_rows [n, row_bytes] u8, dev_rows [C, row_bytes] u8 (updated in place)."""
    host_rows = _c(host_rows, np.uint8)
    assert dev_rows.dtype == np.uint8 and dev_rows.flags.c_contiguous
    tok = _c(tok, np.int32)
    slot = _c(slot, np.int32)
    lib().orc_recall(_p(host_rows, ctypes.c_uint8), host_rows.shape[1], _p(tok, ctypes.c_int32),
                     _p(slot, ctypes.c_int32), tok.size, _p(dev_rows, ctypes.c_uint8))


def append_tokens(tok_off, tok_end, k_new, kv_new, k8, ks, host_rows, C, tok2slot, slot2tok, dev_rows):
    """One new token per request (the offload write path, as read here).  tok_off [B+1] int64 (regions),
    tok_end [B] int64 (updated), k_new [B,D] f32, kv_new [B,row_bytes] u8; k8 [n,D] u8, ks [n]
    f32, host_rows [n,row_bytes] u8, tok2slot [n] / slot2tok [B*C] int32, dev_rows
    [B*C,row_bytes] u8 are updated in place.  -> full [B] int32 (1: region had no room)."""
    tok_off = _c(tok_off, np.int64)
    k_new = _c(k_new, np.float32)
    kv_new = _c(kv_new, np.uint8)
    for a, dt in ((tok_end, np.int64), (k8, np.uint8), (ks, np.float32), (host_rows, np.uint8),
                  (tok2slot, np.int32), (slot2tok, np.int32), (dev_rows, np.uint8)):
        assert a.dtype == dt and a.flags.c_contiguous
    B, D = k_new.shape
    full = np.zeros(B, np.int32)
    rc = lib().orc_append_tokens(B, _p(tok_off, ctypes.c_int64), _p(tok_end, ctypes.c_int64),
                                 _p(k_new, ctypes.c_float), D, _p(kv_new, ctypes.c_uint8), kv_new.shape[1],
                                 _p(k8, ctypes.c_uint8), _p(ks, ctypes.c_float), _p(host_rows, ctypes.c_uint8),
                                 int(C), _p(tok2slot, ctypes.c_int32), _p(slot2tok, ctypes.c_int32),
                                 _p(dev_rows, ctypes.c_uint8), _p(full, ctypes.c_int32))
    _check(rc, "append_tokens")
    return full


def prefill_rows(scores_rows, row0: int, k: int, theta: float):
    """scores_rows [R, W] f32 (W >= row0+R) -> (sel [R,k], kth [R], hist [R,256], union [row0+R] u8)."""
    s = _c(scores_rows, np.float32)
    R, W = s.shape
    sel = np.empty((R, k), np.int32)
    kth = np.empty(R, np.float32)
    hist = np.empty((R, 256), np.uint32)
    un = np.empty(row0 + R, np.uint8)
    rc = lib().orc_prefill_rows(_p(s, ctypes.c_float), W, R, int(row0), int(k), float(theta),
                                _p(sel, ctypes.c_int32), _p(kth, ctypes.c_float),
                                _p(hist, ctypes.c_uint32), _p(un, ctypes.c_uint8))
    _check(rc, "prefill_rows")
    return sel, kth, hist, un


def decode_step(tok_off, q, w, k8, ks, k, alpha, predictor, cap, theta, C, tok2slot, slot2tok,
                host_rows, dev_rows, nthreads=1, want_scores=False):
    """One oracle decode step of one layer for all requests (state updated in place).

    -> dict(sel_idx [B,k], sel_slot [B,k], kth [B], nmiss [B], scores [N] or None)."""
    tok_off = _c(tok_off, np.int64)
    q = _c(q, np.float32)
    w = _c(w, np.float32)
    k8 = _c(k8, np.uint8)
    ks = _c(ks, np.float32)
    B, H, D = q.shape
    for a, dt in ((theta, np.float32), (tok2slot, np.int32), (slot2tok, np.int32),
                  (dev_rows, np.uint8)):
        assert a.dtype == dt and a.flags.c_contiguous
    host_rows = _c(host_rows, np.uint8)
    sel_idx = np.empty((B, k), np.int32)
    sel_slot = np.empty((B, k), np.int32)
    kth = np.empty(B, np.float32)
    nmiss = np.zeros(B, np.int32)
    sc = np.empty(int(tok_off[-1]), np.float32) if want_scores else None
    rc = lib().orc_decode_step(
        B, _p(tok_off, ctypes.c_int64), _p(q, ctypes.c_float), _p(w, ctypes.c_float), H, D,
        _p(k8, ctypes.c_uint8), _p(ks, ctypes.c_float), int(k), float(alpha), int(predictor),
        int(cap), _p(theta, ctypes.c_float), int(C), _p(tok2slot, ctypes.c_int32),
        _p(slot2tok, ctypes.c_int32), _p(host_rows, ctypes.c_uint8), host_rows.shape[1],
        _p(dev_rows, ctypes.c_uint8), _p(sel_idx, ctypes.c_int32), _p(sel_slot, ctypes.c_int32),
        _p(kth, ctypes.c_float), _p(nmiss, ctypes.c_int32),
        _p(sc, ctypes.c_float) if sc is not None else None, int(nthreads))
    _check(rc, "decode_step")
    return dict(sel_idx=sel_idx, sel_slot=sel_slot, kth=kth, nmiss=nmiss, scores=sc)


def bf16_value(bits: int) -> float:
    return float(lib().orc_bf16_value(int(bits)))


def mla_decode(q_bits, kv_bits, slots, scale: float):
    """Sparse MLA decode attention of one request (fp64).  q_bits [H,576] and kv_bits
    [rows,576] are bf16 bit patterns (uint16); slots [k] int32 (-1: padding).
    -> (out [H,512] f64, lse [H] f64, mass [H,512] f64)."""
    q = _c(q_bits, np.uint16)
    kv = _c(kv_bits, np.uint16)
    sl = _c(slots, np.int32).reshape(-1)
    H = q.shape[0]
    assert q.shape[1] == 576 and kv.shape[1] == 576
    out = np.empty((H, 512), np.float64)
    lse = np.empty(H, np.float64)
    mass = np.empty((H, 512), np.float64)
    rc = lib().orc_mla_decode(_p(q, ctypes.c_uint16), H, _p(kv, ctypes.c_uint16), kv.shape[0],
                              _p(sl, ctypes.c_int32), sl.size, float(scale), _p(out, ctypes.c_double),
                              _p(lse, ctypes.c_double), _p(mass, ctypes.c_double))
    _check(rc, "mla_decode")
    return out, lse, mass
