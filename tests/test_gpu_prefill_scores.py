"""GPU parity of echo_prefill_scores (several query rows per MMA) against the oracle.

Causal scores within the fp64 tolerance, per-row shifted histograms exact against the oracle's
histogram of the GPU scores (added to what the histogram held), and every position past a row's
causal end left untouched.  Cases: fewer rows than one MMA group, row counts that are no multiple
of the 8-row unit, a block that starts mid-prompt, keys ending mid-tile, head weights of both
signs, and a finite or absent block threshold.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from sparse_attention_kv_echo_gb300 import _lib as L
from sparse_attention_kv_echo_gb300 import workloads as wl
from tests._parity import score_tolerance_ok

pytestmark = pytest.mark.gpu
dev = "cuda"
SENTINEL = 0x7FC01234            # a NaN payload the kernel never writes


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.load(build_if_missing=True)


def _inputs(n_keys, R, block_seed, signed=False):
    w = wl.scaled(wl.WORKLOADS["prefill"], f"pfs_{n_keys}", lengths=(n_keys,), prefill_block=R)
    k8, ks = wl.make_keys(w, 0)
    q, wt = wl.make_prefill_queries(w, block_seed)
    q, wt = q[:R].contiguous(), wt[:R].contiguous()
    if signed:
        wt = (wt - 0.5).contiguous()
    return k8, ks, q, wt


def _run(n_keys, R, row0, W=None, theta=None, signed=False, rows_checked=None, hist_init=0):
    W = W if W is not None else row0 + R + 37
    k8, ks, q, wt = _inputs(n_keys, R, block_seed=row0 // max(R, 1), signed=signed)
    q8 = torch.empty((R, 64, 128), dtype=torch.uint8, device=dev)
    qs = torch.empty((R, 64), dtype=torch.float32, device=dev)
    wf = torch.empty((R, 64), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    L.quantize_q(q.to(dev), wt.to(dev), q8, qs, wf, status)
    scores = torch.full((R, W), 0, dtype=torch.int32, device=dev).fill_(SENTINEL).view(torch.float32)
    hist = torch.full((R, 256), hist_init, dtype=torch.int32, device=dev)
    th = None if theta is None else torch.tensor([theta], dtype=torch.float32, device=dev)
    L.prefill_scores(R, row0, n_keys, q8, wf, k8.to(dev), ks.to(dev), scores, W, th, hist, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"status {int(status.item()):#x}"
    gs = scores.cpu().numpy()
    gbits = gs.view(np.uint32)
    gh = hist.cpu().numpy().view(np.uint32)
    oq8, oqs, _ = orc.quantize_q(q.numpy(), wt.numpy())
    k8n, ksn = k8.numpy(), ks.numpy()
    th_o = np.inf if theta is None else theta
    check = range(R) if rows_checked is None else rows_checked
    for r in range(R):
        p = row0 + r
        assert np.all(gbits[r, p + 1:] == SENTINEL), (r, "wrote past its causal end")
        assert not np.any(gbits[r, :p + 1] == SENTINEL), (r, "left a causal position unwritten")
        want = orc.hist256(gs[r, :p + 1], th_o).astype(np.int64) + hist_init
        assert np.array_equal(gh[r].astype(np.int64), want), r
    for r in check:
        p = row0 + r
        ref, ab = orc.scores(oq8[r], oqs[r], wt.numpy()[r], k8n, ksn, tok=np.arange(p + 1, dtype=np.int64))
        bad, _ = score_tolerance_ok(gs[r, :p + 1], ref, ab)
        assert bad.size == 0, (r, bad[:5])


def test_rows_fewer_than_one_mma_group():
    _run(n_keys=3, R=3, row0=0)


def test_ragged_units_from_the_start():
    _run(n_keys=421, R=421, row0=0, signed=True)          # 52 full units + 5 rows; keys end mid-tile


def test_block_mid_prompt_with_threshold():
    _run(n_keys=1900, R=300, row0=1211, theta=0.37, hist_init=3)


def test_one_row_deep_in_the_prompt():
    _run(n_keys=5000, R=1, row0=4999, W=5000)


def test_full_block_shape_sampled_rows():
    # the prompt's block shape: 2048 rows at position 6144 (keys up to 8192), every row's
    # histogram and causal boundary, the scores of sampled rows
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([rng.choice(2048, 12, replace=False), [0, 7, 8, 2047]]))
    _run(n_keys=8192, R=2048, row0=6144, W=8192, theta=-0.5, signed=True, rows_checked=rows)
