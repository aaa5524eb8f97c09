"""GPU parity at the workloads' full sizes, against the CPU oracle:

  - the DeepSeek-V3.2-shaped decode (32 requests x 131072 tokens, 5% hot keys, k = 2048,
    8192 slots) with all 4 layers in one CUDA graph, 16 steps: every (request, layer) of every
    step bit-exact on histograms, early lists, top-k, k-th scores, thresholds, slots, miss
    lists, tables and rows; fp64 scores of sampled tokens on steps {0, 1, last, one more};
  - the skewed mixed batch (64 requests of 4096..262144 tokens, 2 layers, 2560 slots), with the
    predictor on and off, 17 steps: the queries are redrawn at steps 8 and 16 (miss bursts);
  - the chunked prefill of the 102400-token prompt, all 50 blocks of 2048 rows;
  - the query quantiser's E4M3 rounding of every fp32 value below 448 in magnitude.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle as orc
from sparse_attention_kv_echo_gb300 import _lib as L
from sparse_attention_kv_echo_gb300 import workloads as wl
from tests._parity import run_stack

pytestmark = pytest.mark.gpu
dev = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.load(build_if_missing=True)


def _score_steps(steps, seed):
    extra = int(np.random.default_rng(seed).integers(2, steps - 1))
    return {0, 1, steps - 1, extra}


def test_v32_four_layers_in_one_graph():
    w = wl.WORKLOADS["v32"]
    steps = 16
    rep = run_stack(w, steps, w.L, cross_layer=False, keys_device="cuda", score_steps=_score_steps(steps, 0),
                    score_sample=256, threads=16)
    for l in range(w.L):
        assert rep["misses"][l][0] == w.B * w.k          # the first step recalls every selection
        assert rep["fallbacks"][l] <= w.B                 # only the unshifted first step may overflow


@pytest.mark.parametrize("predictor", [True, False])
def test_skewed_both_layers_through_two_redraws(predictor):
    w = wl.scaled(wl.WORKLOADS["skewed"], "skewed", predictor=predictor)
    steps = 17
    rep = run_stack(w, steps, w.L, cross_layer=False, keys_device="cuda", predictor=predictor,
                    score_steps=_score_steps(steps, 1), score_sample=128, threads=16)
    for l in range(w.L):
        m = rep["misses"][l]
        # a redraw (steps 8 and 16) selects mostly new tokens: a burst of misses
        assert m[8] > 2 * m[7] and m[16] > 2 * m[15], m


def test_prefill_full_size_every_block():
    """102400-token prompt, 2048-row blocks, k = 2048, C = 260000: all 50 blocks; sampled rows
    exact against the oracle, the union, threshold, tables and rows every block."""
    from tests.test_gpu_prefill import _run
    _run(wl.WORKLOADS["prefill"], full_rows=False, row_sample=6, blocks=None, keys_device="cuda")


def test_e4m3_every_pattern_below_448():
    """Rows whose largest magnitude is 448 get the power-of-two scale 1, so the quantiser's
    codes are E4M3(q) itself: every fp32 bit pattern of magnitude below 448 (both signs,
    2.28e9 values, 127 per row) against the oracle's OCP rounding."""
    per_row, B = 127, L.MAX_REQUESTS
    chunk = B * L.HEADS * per_row
    top = 0x43E00000                                         # the bits of 448.0
    q8 = torch.empty((B, L.HEADS, L.DIM), dtype=torch.uint8, device=dev)
    qs = torch.empty((B, L.HEADS), dtype=torch.float32, device=dev)
    wf = torch.empty((B, L.HEADS), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    w = torch.ones((B, L.HEADS), device=dev)
    q = torch.empty((B * L.HEADS, L.DIM), dtype=torch.float32, device=dev)
    pool = ThreadPoolExecutor(max_workers=16)
    checked = 0
    for sign in (0, 0x80000000):
        for m0 in range(0, top, chunk):
            m1 = min(top, m0 + chunk)
            cnt = m1 - m0
            rows = (cnt + per_row - 1) // per_row
            bits = (torch.arange(m0, m1, dtype=torch.int64, device=dev) | sign)
            x = bits.to(torch.int32).view(torch.float32) if sign == 0 else \
                (bits - (1 << 32)).to(torch.int32).view(torch.float32)
            q.fill_(448.0)
            pad = torch.zeros(rows * per_row, dtype=torch.float32, device=dev)
            pad[:cnt] = x
            q[:rows, 1:] = pad.view(rows, per_row)
            L.quantize_q(q.view(B, L.HEADS, L.DIM), w, q8, qs, wf, st)
            got = q8.view(-1, L.DIM)[:rows, 1:].reshape(-1)[:cnt].cpu().numpy()
            xs = (np.arange(m0, m1, dtype=np.uint64) | np.uint64(sign)).astype(np.uint32).view(np.float32)
            parts = np.array_split(xs, 16)
            ref = np.concatenate(list(pool.map(orc.e4m3_encode, parts)))
            bad = np.nonzero(got != ref)[0]
            assert bad.size == 0, (hex(int(xs.view(np.uint32)[bad[0]])), got[bad[:4]], ref[bad[:4]])
            checked += cnt
    pool.shutdown()
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and bool(torch.all(qs == 1.0))
    assert checked == 2 * top
