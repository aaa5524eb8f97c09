"""A bounded wait that runs out, on the GPU, without a fault or a hang.

echo_debug_stall_epilogue(limit) makes the score kernel's epilogue first wait
on a barrier that nothing arrives on.  The wait must give up after the limit
and the call report ECHO_ST_TIMEOUT in its status word, while the kernel's
producer and MMA warps drain their copies and MMAs and the tensor memory is
freed; with the stall off again the next call on the same context must run
clean and match the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from sparse_attention_kv_echo_gb300 import _lib as L
from sparse_attention_kv_echo_gb300 import workloads as wl
from tests._parity import score_tolerance_ok

pytestmark = pytest.mark.gpu
dev = "cuda"


def _score(w, off, q, wt, k8, ks, status):
    B, n = w.B, w.total_tokens
    q8 = torch.empty((B, 64, 128), dtype=torch.uint8, device=dev)
    qs = torch.empty((B, 64), dtype=torch.float32, device=dev)
    wf = torch.empty((B, 64), dtype=torch.float32, device=dev)
    hist = torch.zeros((B, 256), dtype=torch.int32, device=dev)
    scores = torch.zeros(n, dtype=torch.float32, device=dev)
    th = torch.full((B,), math.inf, device=dev)
    L.quantize_q(q, wt, q8, qs, wf, status, hist=hist)
    L.index_scores(off, n, q8, wf, k8, ks, scores, th, hist, status)
    torch.cuda.synchronize()
    return scores


def test_epilogue_wait_runs_out_then_the_next_call_is_clean():
    L.load(build_if_missing=True)
    w = wl.scaled(wl.WORKLOADS["tiny"], "timeout", B=2, lengths=(40000, 9000))
    off = torch.from_numpy(wl.tok_offsets(w.lengths)).to(dev)
    k8c, ksc = wl.make_keys(w, 0)
    k8, ks = k8c.to(dev), ksc.to(dev)
    q = wl.QueryStream(w, 0).next()
    wt = wl.make_weights(w, 0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    try:
        L.debug_stall_epilogue(200_000)      # 0.2 ms
        _score(w, off, q.to(dev), wt.to(dev), k8, ks, status)
        assert int(status.item()) & L.ST_TIMEOUT, f"status {int(status.item()):#x}"
    finally:
        L.debug_stall_epilogue(-1)
    # the same context, the default limit: a clean call with correct scores
    status.zero_()
    scores = _score(w, off, q.to(dev), wt.to(dev), k8, ks, status)
    assert int(status.item()) == 0
    gs = scores.cpu().numpy()
    q8, qsc, _ = orc.quantize_q(q.numpy(), wt.numpy())
    lo = wl.tok_offsets(w.lengths)
    for b in range(w.B):
        tok = np.arange(lo[b], lo[b + 1], dtype=np.int64)[::37]
        ref, ab = orc.scores(q8[b], qsc[b], wt.numpy()[b], k8c.numpy(), ksc.numpy(), tok=tok)
        bad, _ = score_tolerance_ok(gs[tok], ref, ab)
        assert bad.size == 0, (b, tok[bad[:5]])
