"""The allocation-free prefill block (echo_prefill_block_static).

It exists for callers that cannot give the library device memory: runtimes
that reserve all device memory at start-up and may not allocate later,
embedders without an allocator of their own, and latency-critical threads
that cannot take cudaMalloc's implicit synchronisation.  It must give the
same results as echo_prefill_block with a caller workspace, call after call,
and refuse blocks that do not fit its fixed scratch.  This file is collected
last on purpose; it needs nothing from the other tests.
"""
import numpy as np
import pytest
import torch

from sparse_attention_kv_echo_gb300 import _lib as L
from sparse_attention_kv_echo_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
dev = "cuda"


class _Outputs:
    def __init__(self, R, W, k, n, C, host):
        i32 = dict(dtype=torch.int32, device=dev)
        self.scores = torch.zeros((R, W), dtype=torch.float32, device=dev)
        self.hist = torch.zeros((R, 256), **i32)
        self.sel = torch.full((R, k), -1, **i32)
        self.kth = torch.zeros(R, dtype=torch.float32, device=dev)
        self.theta = torch.full((1,), float("inf"), dtype=torch.float32, device=dev)
        self.ulist = torch.full((W,), -1, **i32)
        self.ucount = torch.zeros(1, **i32)
        self.ubits = torch.zeros((W + 31) // 32, **i32)
        self.slot = torch.full((W,), -1, **i32)
        self.status = torch.zeros(1, **i32)
        self.cache = L.LayerCache(1, n, C, host)


def _block(out, static, i, w, R, n, W, k8, ks, ws=None, stream=None, copy_stream=None):
    q, wt = (t.to(dev) for t in wl.make_prefill_queries(w, i))
    Ri, row0 = q.shape[0], i * R
    args = (Ri, row0, n, q, wt, k8, ks, w.k, out.theta, 0.5, out.scores, W, out.hist, out.sel, out.kth, out.ulist,
            out.ucount, out.ubits, out.cache, out.slot)
    if static:
        L.prefill_block_static(*args, out.status, stream=stream, copy_stream=copy_stream)
    else:
        L.prefill_block(*args, ws, out.status, stream=stream, copy_stream=copy_stream)


def _assert_same(new, ref, what):
    # the same kernels run on the same inputs: every output is bit-identical
    for name in ("scores", "kth", "theta", "hist", "sel", "ulist", "ucount", "ubits", "slot", "status"):
        assert torch.equal(getattr(new, name), getattr(ref, name)), (what, name)
    for name in ("tok2slot", "slot2tok", "freebits", "dev_kv"):
        assert torch.equal(getattr(new.cache, name), getattr(ref.cache, name)), (what, name)


def test_static_scratch_matches_workspace_call_twice():
    L.load(build_if_missing=True)
    w = wl.scaled(wl.WORKLOADS["prefill"], "pf_static", lengths=(3000,), prefill_block=1024, k=256, C=3008)
    k8, ks = (t.to(dev) for t in wl.make_keys(w, 0))
    host = wl.make_host_pool(w, 0, pin=True)
    n, W, R = w.total_tokens, w.total_tokens, w.prefill_block
    ref = _Outputs(R, W, w.k, n, w.C, host)
    new = _Outputs(R, W, w.k, n, w.C, host)
    ws = torch.zeros(L.prefill_workspace_size(R, W), dtype=torch.uint8, device=dev)
    assert ws.numel() <= L.PREFILL_STATIC_SCRATCH_BYTES
    for i in range(2):                                   # two calls in a row
        _block(ref, False, i, w, R, n, W, k8, ks, ws=ws)
        _block(new, True, i, w, R, n, W, k8, ks)
        torch.cuda.synchronize()
        assert int(ref.status.item()) == 0
        _assert_same(new, ref, i)


def test_static_scratch_two_prompts_back_to_back_with_a_copy_stream():
    """Two prompts of different lengths, their blocks interleaved on one stream with the recall
    on a second stream (as PrefillRunner runs them), nothing synchronised in between: a block
    must not rewrite what the previous block's recall still reads."""
    L.load(build_if_missing=True)
    wa = wl.scaled(wl.WORKLOADS["prefill"], "pf_a", lengths=(3000,), prefill_block=1024, k=256, C=3008)
    wb = wl.scaled(wl.WORKLOADS["prefill"], "pf_b", lengths=(1500,), prefill_block=1024, k=256, C=1504, seed=3)
    main, copy = torch.cuda.Stream(), torch.cuda.Stream()
    runs = {}
    for static in (False, True):
        outs = []
        for w in (wa, wb):
            k8, ks = (t.to(dev) for t in wl.make_keys(w, 0))
            host = wl.make_host_pool(w, 0, pin=True)
            n = w.total_tokens
            o = _Outputs(w.prefill_block, n, w.k, n, w.C, host)
            ws = torch.zeros(L.prefill_workspace_size(w.prefill_block, n), dtype=torch.uint8, device=dev)
            outs.append((w, o, k8, ks, ws))
        torch.cuda.synchronize()
        with torch.cuda.stream(main):
            for i in range(3):
                for w, o, k8, ks, ws in outs:
                    n = w.total_tokens
                    if i * w.prefill_block < n:
                        _block(o, static, i, w, w.prefill_block, n, n, k8, ks, ws=ws, stream=main, copy_stream=copy)
            main.wait_stream(copy)
        torch.cuda.synchronize()
        runs[static] = [o for _, o, _, _, _ in outs]
    for a, b in zip(runs[True], runs[False]):
        assert int(b.status.item()) == 0
        _assert_same(a, b, "interleaved")


def test_static_scratch_allocates_nothing():
    """Once warmed up (its kernels loaded, the scratch address known), a call changes neither
    torch's allocated bytes nor the device's free memory."""
    L.load(build_if_missing=True)
    w = wl.scaled(wl.WORKLOADS["prefill"], "pf_mem", lengths=(2048,), prefill_block=1024, k=256, C=2048)
    k8, ks = (t.to(dev) for t in wl.make_keys(w, 0))
    host = wl.make_host_pool(w, 0, pin=True)
    n, R = w.total_tokens, w.prefill_block
    o = _Outputs(R, n, w.k, n, w.C, host)
    _block(o, True, 0, w, R, n, n, k8, ks)            # warm-up
    q, wt = (t.to(dev) for t in wl.make_prefill_queries(w, 1))
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    L.prefill_block_static(q.shape[0], R, n, q, wt, k8, ks, w.k, o.theta, 0.5, o.scores, n, o.hist, o.sel, o.kth,
                           o.ulist, o.ucount, o.ubits, o.cache, o.slot, o.status)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(o.status.item()) == 0


def test_static_scratch_refuses_blocks_that_do_not_fit():
    L.load(build_if_missing=True)
    R, W = 4096, 10_000_000
    assert L.prefill_workspace_size(R, W) > L.PREFILL_STATIC_SCRATCH_BYTES
    d = torch.zeros(16, device=dev)
    s = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = L.load().echo_prefill_block_static(R, 0, W, d.data_ptr(), d.data_ptr(), d.data_ptr(), d.data_ptr(), 16,
                                            d.data_ptr(), 0.5, d.data_ptr(), W, d.data_ptr(), d.data_ptr(),
                                            d.data_ptr(), d.data_ptr(), d.data_ptr(), None, None, None,
                                            s.data_ptr(), None, None, None)
    assert rc == L.ECHO_ETOOLARGE
    torch.cuda.synchronize()
    assert int(s.item()) == 0                            # nothing was enqueued
