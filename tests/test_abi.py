"""The C-ABI library builds, loads and exports every entry point its header
declares; host-side argument checks answer without touching a GPU (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "echo.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(echo_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    from sparse_attention_kv_echo_gb300 import build, lib
    build.build()
    return lib.load()


def test_header_declares_the_calls():
    names = _declared()
    for want in ("echo_index_scores", "echo_topk_select", "echo_cache_step", "echo_quantize_q",
                 "echo_early_fetch", "echo_prefill_block"):
        assert want in names


def test_every_declared_symbol_is_exported(L):
    from sparse_attention_kv_echo_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (echo_\w+)", out))
    for name in _declared():
        assert name in exported, name
        assert hasattr(L, name)


def test_binding_lists_every_export(L):
    from sparse_attention_kv_echo_gb300 import lib
    assert sorted(lib.EXPORTS) == _declared()


def test_host_checks_reject_bad_arguments(L):
    """These return before any CUDA call, so they run without a GPU."""
    from sparse_attention_kv_echo_gb300 import lib
    v = ctypes.c_void_p
    dummy = v(0x1000)
    # index_scores(B, tok_off, tok_end, n_tokens, q8, wfold, k8, ks, scores, theta, hist, above, cache, ctas,
    #              status, stream)
    def scores_call(B=1, n=10, q8=dummy, k8=dummy, above=None, cache=None):
        return L.echo_index_scores(B, dummy, None, n, q8, dummy, k8, dummy, dummy, None, None, above, cache, 0, dummy,
                                   None)
    assert scores_call(B=0) == lib.ECHO_EINVAL
    assert scores_call(B=lib.MAX_REQUESTS + 1) == lib.ECHO_EUNSUPPORTED
    assert scores_call(q8=None) == lib.ECHO_EINVAL                     # missing q8
    assert scores_call(k8=v(0x1001)) == lib.ECHO_EINVAL                # keys must be 16-byte aligned
    assert scores_call(n=-5) == lib.ECHO_EINVAL                        # negative token count
    assert scores_call(n=0) == lib.ECHO_OK                             # no tokens: nothing enqueued
    # a cache needs the above-threshold words, a complete struct and the snapshot
    c = lib.EchoCacheStruct()
    for f, _ in lib.EchoCacheStruct._fields_:
        if f not in ("row_bytes", "C", "reserved"):
            setattr(c, f, 0x1000)
    c.row_bytes, c.C = 1152, 64
    cache = ctypes.byref(c)
    assert scores_call(above=None, cache=cache) == lib.ECHO_EINVAL
    c.free_snap = None
    assert scores_call(above=dummy, cache=cache) == lib.ECHO_EINVAL
    # early_fetch(B, tok_off, tok_end, n_tokens, above, early_cap, cache, status, stream)
    assert L.echo_early_fetch(1, dummy, None, 10, dummy, -1, cache, dummy, None) == lib.ECHO_EINVAL   # no snapshot
    c.free_snap = 0x1000
    assert L.echo_early_fetch(1, dummy, None, 10, None, -1, cache, dummy, None) == lib.ECHO_EINVAL    # no above words
    assert L.echo_early_fetch(1, dummy, None, 10, dummy, -1, None, dummy, None) == lib.ECHO_EINVAL    # no cache
    assert L.echo_early_fetch(0, dummy, None, 10, dummy, -1, cache, dummy, None) == lib.ECHO_EINVAL
    assert L.echo_early_fetch(1, dummy, None, 0, dummy, -1, cache, dummy, None) == lib.ECHO_OK        # nothing to do
    assert L.echo_early_fetch(1, dummy, None, 10, dummy, 0, cache, dummy, None) == lib.ECHO_OK        # cap 0: nothing
    c.C = 48                                                           # not a multiple of 32
    assert L.echo_early_fetch(1, dummy, None, 10, dummy, -1, cache, dummy, None) == lib.ECHO_ECAPACITY
    assert scores_call(above=dummy, cache=cache) == lib.ECHO_ECAPACITY
    # the bitmask size: four words per 128-token tile of each request, at most
    assert lib.above_words(8, 32768) == 4 * (256 + 8)
    assert lib.above_words(0, 10) == 0
    assert L.echo_topk_select(1, dummy, None, 10, dummy, 0, None, None, 0.5, dummy, dummy, dummy, None,
                              None) == lib.ECHO_EINVAL
    assert L.echo_topk_select(-3, dummy, None, 10, dummy, 4, None, None, 0.5, dummy, dummy, dummy, None,
                              None) == lib.ECHO_EINVAL
    # quantize_q(B, q, w, q8, qscale, wfold, hist, cand_cnt, status, stream)
    assert L.echo_quantize_q(-1, dummy, dummy, dummy, dummy, dummy, None, None, dummy, None) == lib.ECHO_EINVAL
    assert L.echo_quantize_q(1, dummy, dummy, dummy, dummy, v(0x1004), None, None, dummy, None) == lib.ECHO_EINVAL
    assert L.echo_quantize_q(1, dummy, dummy, dummy, dummy, dummy, None, v(0x1002), dummy, None) == lib.ECHO_EINVAL
    assert L.echo_quantize_q(0, None, None, None, None, None, None, None, None, None) == lib.ECHO_OK


def test_candidate_list_checks(L):
    """echo_index_scores_cands needs complete lists; echo_topk_select_cands refuses bad sizes,
    incomplete lists and a cache without sel_slot or above its shared-memory limit."""
    from sparse_attention_kv_echo_gb300 import lib
    v = ctypes.c_void_p
    d = v(0x1000)
    cl = lib.EchoCandsStruct()
    cl.key, cl.idx, cl.cnt, cl.cut, cl.cap = 0x1000, 0x1000, 0x1000, 0x1000, 64
    cands = ctypes.byref(cl)

    def scores(c, n=10):
        return L.echo_index_scores_cands(1, d, None, n, d, d, d, d, d, None, None, None, None, c, 0, d, None)
    assert scores(None) == lib.ECHO_EINVAL
    assert scores(cands, n=0) == lib.ECHO_OK
    cl.cap = 0
    assert scores(cands) == lib.ECHO_EINVAL
    cl.cap, cl.cut = 64, None
    assert scores(cands) == lib.ECHO_EINVAL
    cl.cut = 0x1000

    # topk_select_cands(B, tok_off, tok_end, n, scores, k, hist, theta, alpha, cands, sel, kth, above, cap,
    #                   cache, sel_slot, status, stats, stream)
    def topk(B=1, k=16, c=cands, cache=None, slot=None):
        return L.echo_topk_select_cands(B, d, None, 100, d, k, None, None, 0.5, c, d, d, None, -1, cache, slot, d,
                                        None, None)
    assert topk(B=0) == lib.ECHO_EINVAL
    assert topk(k=0) == lib.ECHO_EINVAL
    assert topk(B=lib.MAX_REQUESTS + 1) == lib.ECHO_EUNSUPPORTED
    cl.idx = None
    assert topk() == lib.ECHO_EINVAL
    cl.idx = 0x1000
    s = lib.EchoCacheStruct()
    for f, _ in lib.EchoCacheStruct._fields_[:12]:
        setattr(s, f, 0x2000)
    s.row_bytes, s.C = 1152, 64
    assert topk(cache=ctypes.byref(s)) == lib.ECHO_EINVAL                    # no sel_slot
    assert topk(k=65, cache=ctypes.byref(s), slot=d) == lib.ECHO_ECAPACITY   # k > C
    s.C = 65536
    assert topk(cache=ctypes.byref(s), slot=d) == lib.ECHO_EUNSUPPORTED      # free bits beyond shared memory


def test_cache_checks(L):
    from sparse_attention_kv_echo_gb300 import lib
    v = ctypes.c_void_p
    s = lib.EchoCacheStruct()
    for f, _ in lib.EchoCacheStruct._fields_[:12]:
        setattr(s, f, 0x2000)
    s.row_bytes, s.C = 1152, 64
    dummy = v(0x1000)
    # k (m) larger than C
    assert L.echo_cache_step(1, dummy, None, 100, dummy, 65, None, 0, ctypes.byref(s), dummy, dummy, None, None,
                             None, 0) == lib.ECHO_ECAPACITY
    s.C = 48   # not a multiple of 32
    assert L.echo_cache_step(1, dummy, None, 100, dummy, 16, None, 0, ctypes.byref(s), dummy, dummy, None, None,
                             None, 0) == lib.ECHO_ECAPACITY
    s.C, s.row_bytes = 64, 1000  # row not a multiple of 16 bytes
    assert L.echo_cache_step(1, dummy, None, 100, dummy, 16, None, 0, ctypes.byref(s), dummy, dummy, None, None,
                             None, 0) == lib.ECHO_EUNSUPPORTED
    s.row_bytes, s.dev_kv = 1152, None
    assert L.echo_cache_step(1, dummy, None, 100, dummy, 16, None, 0, ctypes.byref(s), dummy, dummy, None, None,
                             None, 0) == lib.ECHO_EINVAL
    s.dev_kv = 0x2000
    # unknown flag bits; the held-slot form and lazy reuse together; lazy reuse in the resolved form
    assert L.echo_cache_step(1, dummy, None, 100, dummy, 16, None, 0, ctypes.byref(s), dummy, dummy, None, None,
                             None, 4) == lib.ECHO_EINVAL
    assert L.echo_cache_step(1, dummy, None, 100, dummy, 16, None, 0, ctypes.byref(s), dummy, dummy, None, None,
                             None, lib.CACHE_HOLD_EARLY | lib.CACHE_LAZY) == lib.ECHO_EINVAL
    assert L.echo_cache_step_resolved(1, dummy, None, 100, dummy, 16, ctypes.byref(s), dummy, dummy, None, None,
                                      None, lib.CACHE_LAZY) == lib.ECHO_EINVAL
    assert L.echo_cache_step_resolved(1, dummy, None, 100, dummy, 16, ctypes.byref(s), dummy, dummy, None, None,
                                      None, 4) == lib.ECHO_EINVAL
    # the resolved form: k larger than C; the cached top-k: C above its shared-memory limit
    assert L.echo_cache_step_resolved(1, dummy, None, 100, dummy, 65, ctypes.byref(s), dummy, dummy, None, None,
                                      None, 0) == lib.ECHO_ECAPACITY
    s.C = 65536
    assert L.echo_topk_select_cached(1, dummy, None, 100, dummy, 16, None, None, 0.5, dummy, dummy, None, -1,
                                     ctypes.byref(s), dummy, dummy, None, None) == lib.ECHO_EUNSUPPORTED
    s.C = 64
    assert L.echo_topk_select_cached(1, dummy, None, 100, dummy, 16, None, None, 0.5, dummy, dummy, None, -1,
                                     ctypes.byref(s), None, dummy, None, None) == lib.ECHO_EINVAL   # no sel_slot



def test_append_argument_checks(L):
    """echo_append_tokens(B, tok_off, tok_end, n_tokens, k_new, kv_new, k8, ks, cache, status, stream):
    argument errors return before anything is enqueued (no GPU needed)."""
    from sparse_attention_kv_echo_gb300 import lib
    d = ctypes.c_void_p(0x1000)
    assert L.echo_append_tokens(0, d, d, 10, d, d, d, d, None, d, None) == lib.ECHO_EINVAL
    assert L.echo_append_tokens(1, d, d, 0, d, d, d, d, None, d, None) == lib.ECHO_EINVAL
    assert L.echo_append_tokens(1, None, d, 10, d, d, d, d, None, d, None) == lib.ECHO_EINVAL
    assert L.echo_append_tokens(1, d, None, 10, d, d, d, d, None, d, None) == lib.ECHO_EINVAL
    assert L.echo_append_tokens(1, d, d, 10, d, d, d, d, None, d, None) == lib.ECHO_EINVAL   # no cache
    assert L.echo_append_tokens(lib.MAX_REQUESTS + 1, d, d, 10, d, d, d, d, None, d, None) == lib.ECHO_EUNSUPPORTED


def test_pool_argument_checks(L):
    """echo_pool_above / echo_pool_select / echo_pool_slots refuse bad arguments before any launch."""
    from sparse_attention_kv_echo_gb300 import lib
    d = ctypes.c_void_p(0x1000)
    assert L.echo_pool_above(0, d, None, 10, d, None, d, d, None) == lib.ECHO_EINVAL
    assert L.echo_pool_above(1, d, None, 10, d, None, d, d, None) == lib.ECHO_EINVAL      # no pool
    assert L.echo_pool_select(1, None, d, 8, d, None) == lib.ECHO_EINVAL
    assert L.echo_pool_select(1, d, d, 0, d, None) == lib.ECHO_EINVAL
    assert L.echo_pool_slots(lib.MAX_REQUESTS + 1, d, 8, d, d, None) == lib.ECHO_EUNSUPPORTED
    assert L.echo_seed_early(1, d, None, 10, None, 8, d, None, d, None) == lib.ECHO_EINVAL


def test_pool_layer_refuses_append():
    import torch
    from sparse_attention_kv_echo_gb300 import DecodeLayer
    lay = DecodeLayer.__new__(DecodeLayer)
    lay.tok_end, lay.pool_slots = torch.zeros(1, dtype=torch.int64), 64
    with pytest.raises(ValueError):
        lay.append(torch.zeros((1, 128)), torch.zeros((1, 576)))
