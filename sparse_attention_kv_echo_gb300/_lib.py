"""ctypes binding of libecho -- argument marshalling only.

Every call takes torch CUDA tensors (or None where the C ABI allows NULL),
passes their device addresses and the current CUDA stream to the library and
returns.  Nothing here computes: all work runs in the library's kernels.  The
library must be built (``build()``); there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

ECHO_OK, ECHO_EINVAL, ECHO_ECAPACITY, ECHO_EUNSUPPORTED, ECHO_ECUDA, ECHO_ETOOLARGE = 0, -1, -2, -3, -4, -5
PREFILL_STATIC_SCRATCH_BYTES = 32 << 20
ST_TIMEOUT, ST_NAN, ST_NOSLOT, ST_BADDATA, ST_FULL = 0x1, 0x2, 0x4, 0x8, 0x10
STAT_TOPK_FALLBACK, STAT_BOUNDARY_MAX, STAT_EARLY, STAT_MISSES, STAT_EARLY_USED, STAT_CAND_MISS = 0, 1, 2, 3, 4, 5
STAT_REVIVED = 6
STATS_N = 8
HEADS, DIM, MAX_REQUESTS = 64, 128, 4096
CACHE_HOLD_EARLY, CACHE_LAZY = 1, 2   # echo_cache_step flags
TOPK_CACHED_MAX_SLOTS = 32768  # C limit of echo_topk_select_cached and of the cached form of echo_topk_select_cands
CAND_CAP = 16384             # candidate-list entries per request top-k keeps in shared memory
EARLY_FETCH_BLOCKS = 24      # CTAs of the early-fetch and late-recall kernels

EXPORTS = ("echo_above_words", "echo_append_tokens", "echo_cache_step", "echo_cache_step_resolved",
           "echo_debug_stall_epilogue", "echo_device_sm_count",
           "echo_early_fetch", "echo_host_device_alias", "echo_index_scores", "echo_index_scores_cands", "echo_mla_decode", "echo_pool_above", "echo_pool_select",
           "echo_pool_slots", "echo_prefill_block",
           "echo_prefill_block_static", "echo_prefill_scores", "echo_prefill_workspace_size", "echo_quantize_q", "echo_seed_early",
           "echo_topk_select", "echo_topk_select_cached", "echo_topk_select_cands")

_vp = ctypes.c_void_p


class EchoCacheStruct(ctypes.Structure):
    _fields_ = [("tok2slot", _vp), ("slot2tok", _vp), ("freebits", _vp), ("miss_tok", _vp),
                ("miss_slot", _vp), ("miss_cnt", _vp), ("early_tok", _vp), ("early_slot", _vp),
                ("early_cnt", _vp), ("free_snap", _vp), ("host_kv", _vp), ("dev_kv", _vp), ("row_bytes", ctypes.c_int64),
                ("C", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class EchoCandsStruct(ctypes.Structure):
    _fields_ = [("key", _vp), ("idx", _vp), ("cnt", _vp), ("cut", _vp), ("cap", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class EchoError(RuntimeError):
    def __init__(self, call, rc):
        super().__init__(f"{call} returned {rc}")
        self.rc = rc


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libecho.so (raises when it is missing and not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            if not build_if_missing:
                raise RuntimeError(f"libecho is not built ({_build.LIB}); run "
                                   "python -m sparse_attention_kv_echo_gb300.build")
            _build.build()
        L = ctypes.CDLL(_build.LIB)
        i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
        L.echo_quantize_q.restype = i32
        L.echo_quantize_q.argtypes = [i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        L.echo_above_words.restype = ctypes.c_size_t
        L.echo_above_words.argtypes = [i32, i64]
        L.echo_index_scores.restype = i32
        L.echo_index_scores.argtypes = [i32, _vp, _vp, i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                        ctypes.POINTER(EchoCacheStruct), i32, _vp, _vp]
        L.echo_index_scores_cands.restype = i32
        L.echo_index_scores_cands.argtypes = [i32, _vp, _vp, i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                              ctypes.POINTER(EchoCacheStruct), ctypes.POINTER(EchoCandsStruct),
                                              i32, _vp, _vp]
        L.echo_topk_select_cands.restype = i32
        L.echo_topk_select_cands.argtypes = [i32, _vp, _vp, i64, _vp, i32, _vp, _vp, f32,
                                             ctypes.POINTER(EchoCandsStruct), _vp, _vp, _vp, i32,
                                             ctypes.POINTER(EchoCacheStruct), _vp, _vp, _vp, _vp]
        L.echo_early_fetch.restype = i32
        L.echo_early_fetch.argtypes = [i32, _vp, _vp, i64, _vp, i32, ctypes.POINTER(EchoCacheStruct), _vp, _vp]
        L.echo_topk_select.restype = i32
        L.echo_topk_select.argtypes = [i32, _vp, _vp, i64, _vp, i32, _vp, _vp, f32, _vp, _vp, _vp, _vp, _vp]
        L.echo_cache_step.restype = i32
        L.echo_cache_step.argtypes = [i32, _vp, _vp, i64, _vp, i32, _vp, i32, ctypes.POINTER(EchoCacheStruct), _vp,
                                      _vp, _vp, _vp, _vp, i32]
        L.echo_mla_decode.restype = i32
        L.echo_mla_decode.argtypes = [i32, i32, _vp, _vp, _vp, i64, f32, _vp, _vp, _vp, _vp]
        L.echo_pool_above.restype = i32
        L.echo_pool_above.argtypes = [i32, _vp, _vp, i64, _vp, ctypes.POINTER(EchoCacheStruct), _vp, _vp, _vp]
        L.echo_pool_select.restype = i32
        L.echo_pool_select.argtypes = [i32, _vp, _vp, i32, _vp, _vp]
        L.echo_pool_slots.restype = i32
        L.echo_pool_slots.argtypes = [i32, _vp, i32, _vp, _vp, _vp]
        L.echo_seed_early.restype = i32
        L.echo_seed_early.argtypes = [i32, _vp, _vp, i64, _vp, i32, _vp, ctypes.POINTER(EchoCacheStruct), _vp, _vp]
        L.echo_append_tokens.restype = i32
        L.echo_append_tokens.argtypes = [i32, _vp, _vp, i64, _vp, _vp, _vp, _vp, ctypes.POINTER(EchoCacheStruct),
                                         _vp, _vp]
        L.echo_topk_select_cached.restype = i32
        L.echo_topk_select_cached.argtypes = [i32, _vp, _vp, i64, _vp, i32, _vp, _vp, f32, _vp, _vp, _vp, i32,
                                              ctypes.POINTER(EchoCacheStruct), _vp, _vp, _vp, _vp]
        L.echo_cache_step_resolved.restype = i32
        L.echo_cache_step_resolved.argtypes = [i32, _vp, _vp, i64, _vp, i32, ctypes.POINTER(EchoCacheStruct), _vp, _vp,
                                               _vp, _vp, _vp, i32]
        L.echo_prefill_scores.restype = i32
        L.echo_prefill_scores.argtypes = [i32, i64, i64, _vp, _vp, _vp, _vp, _vp, i64, _vp, _vp, _vp, _vp]
        L.echo_prefill_workspace_size.restype = ctypes.c_size_t
        L.echo_prefill_workspace_size.argtypes = [i32, i64]
        L.echo_prefill_block.restype = i32
        L.echo_prefill_block.argtypes = [i32, i64, i64, _vp, _vp, _vp, _vp, i32, _vp, f32, _vp, i64, _vp, _vp,
                                         _vp, _vp, _vp, _vp, ctypes.POINTER(EchoCacheStruct), _vp, _vp,
                                         ctypes.c_size_t, _vp, _vp, _vp, _vp]
        L.echo_prefill_block_static.restype = i32
        L.echo_prefill_block_static.argtypes = [i32, i64, i64, _vp, _vp, _vp, _vp, i32, _vp, f32, _vp, i64, _vp,
                                                _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(EchoCacheStruct), _vp, _vp,
                                                _vp, _vp, _vp]
        L.echo_host_device_alias.restype = i32
        L.echo_host_device_alias.argtypes = [_vp, ctypes.POINTER(_vp)]
        L.echo_debug_stall_epilogue.restype = i32
        L.echo_debug_stall_epilogue.argtypes = [i64]
        L.echo_device_sm_count.restype = i32
        L.echo_device_sm_count.argtypes = []
        _lib = L
        return L


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(call, rc):
    if rc != ECHO_OK:
        raise EchoError(call, rc)


def host_device_alias(host_tensor: torch.Tensor) -> int:
    out = _vp()
    _check("echo_host_device_alias", load().echo_host_device_alias(host_tensor.data_ptr(), ctypes.byref(out)))
    return out.value


class _CudaArray:
    def __init__(self, iface):
        self.__cuda_array_interface__ = iface


_TYPESTR = {torch.int32: "<i4", torch.float32: "<f4", torch.uint8: "|u1", torch.int64: "<i8"}


def host_alias_tensor(host: torch.Tensor, device) -> torch.Tensor:
    """A CUDA tensor over the device alias of a pinned, contiguous host tensor (kernels
    read and write the host memory directly).  The caller keeps `host` alive."""
    if host.device.type != "cpu" or not host.is_pinned() or not host.is_contiguous():
        raise ValueError("host_alias_tensor needs a pinned, contiguous CPU tensor")
    iface = {"shape": tuple(host.shape), "typestr": _TYPESTR[host.dtype],
             "data": (host_device_alias(host), False), "version": 2, "strides": None}
    with torch.cuda.device(device):
        return torch.as_tensor(_CudaArray(iface), device=device)


def debug_stall_epilogue(limit_ns: int) -> None:
    """echo_debug_stall_epilogue: >= 0, every score call first waits on a barrier nothing arrives
    on and gives up after limit_ns (tests of the timeout path); < 0 turns that off."""
    _check("echo_debug_stall_epilogue", load().echo_debug_stall_epilogue(int(limit_ns)))


def sm_count() -> int:
    return load().echo_device_sm_count()


def quantize_q(q, w, q8, qscale, wfold, status, hist=None, stream=None, cand_cnt=None):
    """echo_quantize_q; q and w may be pinned host tensors, read by the kernel through their
    device alias; cand_cnt: the counts of a Cands (cleared with the histogram)."""
    B = q.shape[0]
    qp = host_device_alias(q) if q.device.type == "cpu" else _ptr(q)
    wp = host_device_alias(w) if w.device.type == "cpu" else _ptr(w)
    _check("echo_quantize_q", load().echo_quantize_q(B, qp, wp, _ptr(q8), _ptr(qscale),
                                                    _ptr(wfold), _ptr(hist), _ptr(cand_cnt), _ptr(status),
                                                    _stream(stream)))


def above_words(B: int, n_tokens: int) -> int:
    return int(load().echo_above_words(int(B), int(n_tokens)))


def index_scores(tok_off, n_tokens, q8, wfold, k8, ks, scores, theta_hat, hist, status, above=None,
                 cache=None, stream=None, ctas=0, tok_end=None, cands=None):
    """echo_index_scores; cache: a LayerCache whose residents `above` leaves out (and whose free bits
    are snapshotted for early_fetch); tok_end: the requests' current ends (None: full regions);
    cands: a Cands (or a view of one) to fill: echo_index_scores_cands."""
    B = q8.shape[0]
    cs = ctypes.byref(cache.struct) if cache is not None else None
    if cands is not None:
        _check("echo_index_scores_cands", load().echo_index_scores_cands(
            B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(q8), _ptr(wfold), _ptr(k8), _ptr(ks), _ptr(scores),
            _ptr(theta_hat), _ptr(hist), _ptr(above), cs, ctypes.byref(cands.struct), int(ctas), _ptr(status),
            _stream(stream)))
        return
    _check("echo_index_scores", load().echo_index_scores(
        B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(q8), _ptr(wfold), _ptr(k8), _ptr(ks), _ptr(scores),
        _ptr(theta_hat), _ptr(hist), _ptr(above), cs, int(ctas), _ptr(status), _stream(stream)))


def topk_select_cands(tok_off, n_tokens, scores, k, hist, theta_hat, alpha, cands, sel_idx, kth, status, stats=None,
                      stream=None, cache=None, sel_slot=None, above=None, early_cap=-1, tok_end=None):
    """echo_topk_select_cands: top-k from the candidate lists of `cands` (None: from all the
    scores), one block per request; with cache (and sel_slot) the cached form (slots of the
    selected tokens as echo_topk_select_cached gives them)."""
    B = tok_off.shape[0] - 1
    _check("echo_topk_select_cands", load().echo_topk_select_cands(
        B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(scores), int(k), _ptr(hist), _ptr(theta_hat),
        float(alpha), ctypes.byref(cands.struct) if cands is not None else None, _ptr(sel_idx), _ptr(kth),
        _ptr(above), int(early_cap), ctypes.byref(cache.struct) if cache is not None else None, _ptr(sel_slot),
        _ptr(status), _ptr(stats), _stream(stream)))


def early_fetch(tok_off, n_tokens, above, early_cap, cache, status, stream=None, tok_end=None):
    """echo_early_fetch: copy the rows of the early set (the tables learn it in cache_step)."""
    B = tok_off.shape[0] - 1
    _check("echo_early_fetch", load().echo_early_fetch(
        B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(above), int(early_cap), ctypes.byref(cache.struct), _ptr(status),
        _stream(stream)))


def topk_select(tok_off, n_tokens, scores, k, hist, theta_hat, alpha, sel_idx, kth, status, stats=None,
                stream=None, tok_end=None):
    B = tok_off.shape[0] - 1
    _check("echo_topk_select", load().echo_topk_select(
        B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(scores), int(k), _ptr(hist), _ptr(theta_hat), float(alpha),
        _ptr(sel_idx), _ptr(kth), _ptr(status), _ptr(stats), _stream(stream)))


def cache_step(tok_off, n_tokens, sel, cache, sel_slot, status, stats=None, stream=None, copy_stream=None,
               above=None, early_cap=-1, hold_early=False, tok_end=None, lazy=False):
    """echo_cache_step; above/early_cap: the early set of this step (as given to early_fetch);
    hold_early: ECHO_CACHE_HOLD_EARLY; lazy: ECHO_CACHE_LAZY (lazy-reuse eviction)."""
    B = tok_off.shape[0] - 1
    m = sel.shape[-1]
    st = _stream(stream)
    cst = _stream(copy_stream) if copy_stream is not None else st
    _check("echo_cache_step", load().echo_cache_step(
        B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(sel), int(m), _ptr(above), int(early_cap),
        ctypes.byref(cache.struct), _ptr(sel_slot), _ptr(status), _ptr(stats), st, cst,
        (CACHE_HOLD_EARLY if hold_early else 0) | (CACHE_LAZY if lazy else 0)))


def topk_select_cached(tok_off, n_tokens, scores, k, hist, theta_hat, alpha, sel_idx, kth, cache, sel_slot,
                       status, stats=None, stream=None, above=None, early_cap=-1, tok_end=None):
    """echo_topk_select_cached: top-k plus each selected token's slot at the cache step's start
    (resident or early; -1: a miss); finish with cache_step_resolved."""
    B = tok_off.shape[0] - 1
    _check("echo_topk_select_cached", load().echo_topk_select_cached(
        B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(scores), int(k), _ptr(hist), _ptr(theta_hat), float(alpha),
        _ptr(sel_idx), _ptr(kth), _ptr(above), int(early_cap), ctypes.byref(cache.struct), _ptr(sel_slot),
        _ptr(status), _ptr(stats), _stream(stream)))


def cache_step_resolved(tok_off, n_tokens, sel, cache, sel_slot, status, stats=None, stream=None, copy_stream=None,
                        hold_early=False, tok_end=None):
    """echo_cache_step_resolved: the cache step after topk_select_cached (sel_slot in/out)."""
    B = tok_off.shape[0] - 1
    m = sel.shape[-1]
    st = _stream(stream)
    cst = _stream(copy_stream) if copy_stream is not None else st
    _check("echo_cache_step_resolved", load().echo_cache_step_resolved(
        B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(sel), int(m), ctypes.byref(cache.struct), _ptr(sel_slot),
        _ptr(status), _ptr(stats), st, cst, CACHE_HOLD_EARLY if hold_early else 0))


def pool_above(tok_off, n_tokens, above_req, pool, above_pool, status, stream=None, tok_end=None):
    """echo_pool_above: per-request above words -> the shared pool's global marks (residents left
    out) and the pool's free-bit snapshot."""
    B = tok_off.shape[0] - 1
    _check("echo_pool_above", load().echo_pool_above(
        B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(above_req), ctypes.byref(pool.struct),
        _ptr(above_pool), _ptr(status), _stream(stream)))


def pool_select(tok_off, sel, sel_pool, stream=None):
    """echo_pool_select: sel [B,k] (request-local) -> sel_pool [B*k] (global, ascending, padding last)."""
    B, k = sel.shape
    _check("echo_pool_select", load().echo_pool_select(B, _ptr(tok_off), _ptr(sel), int(k), _ptr(sel_pool),
                                                       _stream(stream)))


def pool_slots(sel, slot_pool, sel_slot, stream=None):
    """echo_pool_slots: the pool step's slots of sel_pool -> sel_slot [B,k] aligned with sel."""
    B, k = sel.shape
    _check("echo_pool_slots", load().echo_pool_slots(B, _ptr(sel), int(k), _ptr(slot_pool), _ptr(sel_slot),
                                                     _stream(stream)))


def seed_early(tok_off, n_tokens, prev_sel, above, cache, status, stream=None, tok_end=None):
    """echo_seed_early: this layer's early set from the previous layer's selection prev_sel [B,m]
    (above words + cache free-bit snapshot); follow with early_fetch on the same above words."""
    B = tok_off.shape[0] - 1
    _check("echo_seed_early", load().echo_seed_early(
        B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(prev_sel), int(prev_sel.shape[-1]), _ptr(above),
        ctypes.byref(cache.struct), _ptr(status), _stream(stream)))


def append_tokens(tok_off, tok_end, n_tokens, k_new, kv_new, k8, ks, cache, status, stream=None):
    """echo_append_tokens: one new token per request (k_new [B,128] f32, kv_new [B,576] bf16, device)
    into its region at tok_end[b] (updated): E4M3 key + scale, host-pool row, and the lowest free
    cache slot when one is free."""
    B = tok_off.shape[0] - 1
    _check("echo_append_tokens", load().echo_append_tokens(
        B, _ptr(tok_off), _ptr(tok_end), int(n_tokens), _ptr(k_new), _ptr(kv_new), _ptr(k8), _ptr(ks),
        ctypes.byref(cache.struct), _ptr(status), _stream(stream)))


MLA_HEADS, MLA_DQK, MLA_DV, MLA_MAX_K = 128, 576, 512, 8192


def mla_decode(q, sel_slot, dev_kv, C, scale, out, lse, status, stream=None):
    """echo_mla_decode: q [B,128,576] bf16, sel_slot [B,k] int32, dev_kv [B*C,576] bf16 (the
    cache's rows) -> out [B,128,512] f32, lse [B,128] f32."""
    B, k = sel_slot.shape
    _check("echo_mla_decode", load().echo_mla_decode(
        int(B), int(k), _ptr(q), _ptr(sel_slot), _ptr(dev_kv), int(C), float(scale), _ptr(out), _ptr(lse),
        _ptr(status), _stream(stream)))


def prefill_scores(R, row0, n_keys, q8, wfold, k8, ks, scores, W, theta_hat, hist, status, stream=None):
    _check("echo_prefill_scores", load().echo_prefill_scores(
        int(R), int(row0), int(n_keys), _ptr(q8), _ptr(wfold), _ptr(k8), _ptr(ks), _ptr(scores), int(W),
        _ptr(theta_hat), _ptr(hist), _ptr(status), _stream(stream)))


def prefill_workspace_size(R: int, W: int) -> int:
    return int(load().echo_prefill_workspace_size(int(R), int(W)))


def prefill_block(R, row0, n_keys, q, w, k8, ks, k, theta_hat, alpha, scores, W, hist, sel_idx, kth,
                  union_list, union_count, union_bits, cache, sel_slot, ws, status, stats=None, stream=None,
                  copy_stream=None):
    st = _stream(stream)
    cst = _stream(copy_stream) if copy_stream is not None else st
    _check("echo_prefill_block", load().echo_prefill_block(
        int(R), int(row0), int(n_keys), _ptr(q), _ptr(w), _ptr(k8), _ptr(ks), int(k), _ptr(theta_hat),
        float(alpha), _ptr(scores), int(W), _ptr(hist), _ptr(sel_idx), _ptr(kth), _ptr(union_list),
        _ptr(union_count), _ptr(union_bits), ctypes.byref(cache.struct) if cache is not None else None,
        _ptr(sel_slot), _ptr(ws), ws.numel() * ws.element_size(), _ptr(status), _ptr(stats), st, cst))


def prefill_block_static(R, row0, n_keys, q, w, k8, ks, k, theta_hat, alpha, scores, W, hist, sel_idx, kth,
                         union_list, union_count, union_bits, cache, sel_slot, status, stats=None, stream=None,
                         copy_stream=None):
    """echo_prefill_block with the library's fixed device scratch instead of a workspace."""
    st = _stream(stream)
    cst = _stream(copy_stream) if copy_stream is not None else st
    _check("echo_prefill_block_static", load().echo_prefill_block_static(
        int(R), int(row0), int(n_keys), _ptr(q), _ptr(w), _ptr(k8), _ptr(ks), int(k), _ptr(theta_hat),
        float(alpha), _ptr(scores), int(W), _ptr(hist), _ptr(sel_idx), _ptr(kth), _ptr(union_list),
        _ptr(union_count), _ptr(union_bits), ctypes.byref(cache.struct) if cache is not None else None,
        _ptr(sel_slot), _ptr(status), _ptr(stats), st, cst))


class Cands:
    """Candidate lists of decode top-k for B requests (torch-owned, int32 storage): key / idx
    [B*cap], cnt [B] (cleared by quantize_q when passed as cand_cnt), cut [B] (all ones = no
    list yet; top-k writes the next step's)."""

    def __init__(self, B: int, cap: int = CAND_CAP, device="cuda"):
        i32 = dict(dtype=torch.int32, device=device)
        self.B, self.cap, self.b0 = int(B), int(cap), 0
        self.key = torch.zeros(max(self.B * self.cap, 1), **i32)
        self.idx = torch.zeros(max(self.B * self.cap, 1), **i32)
        self.cnt = torch.zeros(max(self.B, 1), **i32)
        self.cut = torch.full((max(self.B, 1),), -1, **i32)
        self.struct = self._struct(0)

    def _struct(self, b0: int) -> EchoCandsStruct:
        # b0: absolute first request in the storage of the lists this object was made from
        root = getattr(self, "_parent", self)
        s = EchoCandsStruct()
        s.key, s.idx = _ptr(root.key[b0 * self.cap:]), _ptr(root.idx[b0 * self.cap:])
        s.cnt, s.cut = _ptr(root.cnt[b0:]), _ptr(root.cut[b0:])
        s.cap, s.reserved = self.cap, 0
        return s

    def view(self, b0: int, b1: int) -> "Cands":
        """The lists of requests [b0, b1) of this object (shared storage)."""
        root = getattr(self, "_parent", self)
        a0, a1 = self.b0 + int(b0), self.b0 + int(b1)
        v = Cands.__new__(Cands)
        v._parent = root
        v.B, v.cap, v.b0 = a1 - a0, self.cap, a0
        v.key, v.idx = root.key, root.idx
        v.cnt, v.cut = root.cnt[a0:a1], root.cut[a0:a1]
        v.struct = v._struct(a0)
        return v

    def reset(self):
        self.cnt.zero_()
        self.cut.fill_(-1)


class LayerCache:
    """The fixed-size GPU cache tensors of one layer for B requests (torch-owned).

    host_pool: pinned host tensor [n_tokens, row_bytes/2] bf16 (the per-layer
    host copy of every token's KV row)."""

    def __init__(self, B: int, n_tokens: int, C: int, host_pool: torch.Tensor, device="cuda"):
        if C % 32:
            raise ValueError("C must be a multiple of 32")
        assert host_pool.is_pinned()
        self.B, self.C, self.n_tokens = B, C, n_tokens
        self.row_bytes = host_pool.shape[1] * host_pool.element_size()
        i32 = dict(dtype=torch.int32, device=device)
        self.tok2slot = torch.full((max(n_tokens, 1),), -1, **i32)
        self.slot2tok = torch.full((B * C,), -1, **i32)
        self.freebits = torch.full((B * C // 32,), -1, **i32)   # all bits set: every slot free
        self.miss_tok = torch.zeros((B * C,), **i32)
        self.miss_slot = torch.zeros((B * C,), **i32)
        self.miss_cnt = torch.zeros((B,), **i32)
        self.early_tok = torch.zeros((B * C,), **i32)
        self.early_slot = torch.zeros((B * C,), **i32)
        self.early_cnt = torch.zeros((B,), **i32)
        self.free_snap = torch.zeros((B * C // 32,), **i32)
        self.dev_kv = torch.zeros((B * C, host_pool.shape[1]), dtype=host_pool.dtype, device=device)
        self.host_pool = host_pool
        self.host_alias = host_device_alias(host_pool)
        s = EchoCacheStruct()
        s.tok2slot, s.slot2tok, s.freebits = _ptr(self.tok2slot), _ptr(self.slot2tok), _ptr(self.freebits)
        s.miss_tok, s.miss_slot, s.miss_cnt = _ptr(self.miss_tok), _ptr(self.miss_slot), _ptr(self.miss_cnt)
        s.early_tok, s.early_slot, s.early_cnt = (_ptr(self.early_tok), _ptr(self.early_slot),
                                                  _ptr(self.early_cnt))
        s.free_snap = _ptr(self.free_snap)
        s.host_kv, s.dev_kv = self.host_alias, _ptr(self.dev_kv)
        s.row_bytes, s.C, s.reserved = self.row_bytes, C, 0
        self.struct = s

    def view(self, b0: int, b1: int) -> "CacheView":
        """The tables of requests [b0, b1) as a cache of b1 - b0 requests (shared storage)."""
        return CacheView(self, b0, b1)

    def reset(self):
        self.tok2slot.fill_(-1)
        self.slot2tok.fill_(-1)
        self.freebits.fill_(-1)
        self.miss_cnt.zero_()
        self.early_cnt.zero_()


class CacheView:
    """Requests [b0, b1) of a LayerCache: per-request arrays offset to b0, tok2slot and the host
    pool shared (token rows are global).  Holds the parent so its storage stays alive."""

    def __init__(self, parent: LayerCache, b0: int, b1: int):
        self.parent, self.b0, self.b1 = parent, int(b0), int(b1)
        C, words = parent.C, parent.C // 32
        s = EchoCacheStruct()
        s.tok2slot = _ptr(parent.tok2slot)
        s.slot2tok = _ptr(parent.slot2tok[b0 * C:])
        s.freebits = _ptr(parent.freebits[b0 * words:])
        s.miss_tok, s.miss_slot = _ptr(parent.miss_tok[b0 * C:]), _ptr(parent.miss_slot[b0 * C:])
        s.miss_cnt = _ptr(parent.miss_cnt[b0:])
        s.early_tok, s.early_slot = _ptr(parent.early_tok[b0 * C:]), _ptr(parent.early_slot[b0 * C:])
        s.early_cnt = _ptr(parent.early_cnt[b0:])
        s.free_snap = _ptr(parent.free_snap[b0 * words:])
        s.host_kv, s.dev_kv = parent.host_alias, _ptr(parent.dev_kv[b0 * C:])
        s.row_bytes, s.C, s.reserved = parent.row_bytes, C, 0
        self.struct = s
