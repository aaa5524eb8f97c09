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
from tests._parity import RTOL

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
        q, wt = (t.to(dev) for t in wl.make_prefill_queries(w, i))
        Ri = q.shape[0]
        row0 = i * R
        L.prefill_block(Ri, row0, n, q, wt, k8, ks, w.k, ref.theta, 0.5, ref.scores, W, ref.hist, ref.sel,
                        ref.kth, ref.ulist, ref.ucount, ref.ubits, ref.cache, ref.slot, ws, ref.status)
        L.prefill_block_static(Ri, row0, n, q, wt, k8, ks, w.k, new.theta, 0.5, new.scores, W, new.hist,
                               new.sel, new.kth, new.ulist, new.ucount, new.ubits, new.cache, new.slot, new.status)
        torch.cuda.synchronize()
        assert int(ref.status.item()) == 0 and int(new.status.item()) == 0
        np.testing.assert_allclose(new.scores.cpu().numpy(), ref.scores.cpu().numpy(), rtol=RTOL, atol=0)
        np.testing.assert_allclose(new.kth.cpu().numpy(), ref.kth.cpu().numpy(), rtol=RTOL, atol=0)
        np.testing.assert_allclose(new.theta.cpu().numpy(), ref.theta.cpu().numpy(), rtol=RTOL, atol=0)
        for name in ("hist", "sel", "ulist", "ucount", "ubits", "slot"):
            assert torch.equal(getattr(new, name), getattr(ref, name)), (i, name)
        for name in ("tok2slot", "slot2tok", "freebits", "dev_kv"):
            assert torch.equal(getattr(new.cache, name), getattr(ref.cache, name)), (i, name)


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
