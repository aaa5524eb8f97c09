"""GPU parity of whole decode steps (scores -> early fetch -> top-k -> cache step
-> recall) over many steps against the oracle's own state machine, on the
workloads' shapes: every step bit-exact on histograms, selections, thresholds,
tables, slots and recalled bytes; scores within the fp64 tolerance."""
import numpy as np
import pytest
import torch

from sparse_attention_kv_echo_gb300 import DecodeLayer
from sparse_attention_kv_echo_gb300 import _lib as L
from sparse_attention_kv_echo_gb300 import workloads as wl
from tests._parity import run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.load(build_if_missing=True)


def test_tiny_workload_all_steps():
    w = wl.WORKLOADS["tiny"]
    rep = run_decode(w, w.steps, predictor=True)
    assert sum(rep["early"]) > 0                       # the predictor fetched something early
    assert rep["misses"][0] == w.k                     # first step: everything misses


def test_tiny_workload_table_look_up_in_the_cache_step():
    """The decode step with the look-up in the cache step (echo_topk_select + echo_cache_step)
    instead of in top-k."""
    w = wl.WORKLOADS["tiny"]
    rep = run_decode(w, w.steps, predictor=True, resolved=False)
    assert sum(rep["early"]) > 0


def test_batch_workload_table_look_up_in_the_cache_step():
    w = wl.WORKLOADS["batch"]
    run_decode(w, 4, predictor=True, score_sample=256, check_every_score_step=False, resolved=False)


def test_tiny_workload_held_early_slots():
    """The held-slot variant (ECHO_CACHE_HOLD_EARLY): misses never take this step's early slots, the
    late recall runs right after the cache step."""
    w = wl.WORKLOADS["tiny"]
    rep = run_decode(w, w.steps, predictor=True, hold_early=True)
    assert sum(rep["early"]) > 0


def test_batch_workload_held_early_slots_both_look_ups():
    w = wl.WORKLOADS["batch"]
    run_decode(w, 4, predictor=True, score_sample=256, check_every_score_step=False, hold_early=True)
    run_decode(w, 4, predictor=True, score_sample=256, check_every_score_step=False, hold_early=True,
               resolved=False)


def test_tiny_predictor_off():
    w = wl.WORKLOADS["tiny"]
    rep = run_decode(w, 6, predictor=False)
    assert rep["early"] == []


@pytest.mark.parametrize("cap", [0, 16])
def test_early_cap(cap):
    w = wl.scaled(wl.WORKLOADS["tiny"], "cap", lengths=(6000,))
    run_decode(w, 5, predictor=True, cap=cap)


def test_ragged_batch_edge_cases():
    # a request shorter than k, an empty one, a 1-token one, ragged tile tails
    w = wl.scaled(wl.WORKLOADS["tiny"], "ragged", B=6, lengths=(3000, 200, 0, 1, 4173, 129), k=256, C=320)
    run_decode(w, 6, predictor=True)


def test_c_equals_k():
    w = wl.scaled(wl.WORKLOADS["tiny"], "ck", B=2, lengths=(5000, 2500), k=256, C=256)
    run_decode(w, 5, predictor=True)


def test_redraw_bursts():
    w = wl.scaled(wl.WORKLOADS["skewed"], "burst", B=4, lengths=(9000, 4096, 20000, 5000), C=2560)
    run_decode(w, 10, predictor=True)


def test_early_set_larger_than_one_staging_round():
    """A query redraw with a large k and cache: one request fetches more than 4096 rows early, so the
    early fetch stages its (token, slot) pairs in several rounds."""
    w = wl.scaled(wl.WORKLOADS["skewed"], "rounds", B=2, lengths=(32768, 3000), k=6144, C=16384)
    rep = run_decode(w, 10, predictor=True, score_sample=2048)
    assert max(rep["early"]) > 4096, rep["early"]


def test_walking_cache_step_with_large_early_sets():
    """C above the look-up form's limit (2^17 slots): the cache step walks the early set, which a
    query redraw makes larger than the 4096 pairs it keeps in shared memory."""
    w = wl.scaled(wl.WORKLOADS["skewed"], "walk", B=1, lengths=(200000,), k=6144, C=140000)
    rep = run_decode(w, 10, predictor=True, score_sample=1024)
    assert max(rep["early"]) > 4096, rep["early"]


def test_batch_workload_full_size():
    """8 x 32768, k=2048, C=4096: every table/selection bit-exact, scores sampled."""
    w = wl.WORKLOADS["batch"]
    rep = run_decode(w, 6, predictor=True, score_sample=1024)
    # the unshifted first step's boundary bin is larger than shared memory: a second round of
    # bins resolves it without passes over the scores
    assert rep["boundary_max"] > 16384 and rep["fallbacks"] == 0


def test_hot_set_workload_one_layer():
    """The DeepSeek-V3.2-shaped workload (32 x 131072, hot set), one layer, a few steps."""
    w = wl.WORKLOADS["v32"]
    rep = run_decode(w, 3, predictor=True, score_sample=256, keys_device="cuda")
    assert rep["misses"][0] == w.B * w.k


def test_skewed_workload_both_predictor_modes():
    w = wl.WORKLOADS["skewed"]
    a = run_decode(w, 3, predictor=True, score_sample=256, check_every_score_step=False, keys_device="cuda")
    b = run_decode(w, 3, predictor=False, score_sample=256, check_every_score_step=False, keys_device="cuda")
    assert a["misses"][0] == b["misses"][0]


def test_graph_replay_equals_eager():
    """One captured decode step, replayed, gives the same bytes as eager steps."""
    w = wl.scaled(wl.WORKLOADS["batch"], "graph", B=3, lengths=(9000, 20000, 4000), k=512, C=1024)
    dev = "cuda"
    off = wl.tok_offsets(w.lengths)
    k8, ks = wl.make_keys(w, 0)
    wt = wl.make_weights(w, 0)
    host = wl.make_host_pool(w, 0, pin=True)
    eager = DecodeLayer(off, k8.to(dev), ks.to(dev), w.k, w.C, host)
    graph = DecodeLayer(off, k8.to(dev), ks.to(dev), w.k, w.C, host)
    qs = wl.QueryStream(w, 0)
    queries = [qs.next() for _ in range(6)]
    for lay in (eager, graph):
        lay.q_in.copy_(queries[0].to(dev))
        lay.w_in.copy_(wt.to(dev))
        lay.step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            graph.step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for t in range(1, 6):
        eager.q_in.copy_(queries[t].to(dev))
        eager.step()
        graph.q_in.copy_(queries[t].to(dev))
        g.replay()
        torch.cuda.synchronize()
        for name in ("scores", "hist", "theta", "sel_idx", "sel_slot", "kth"):
            assert torch.equal(getattr(eager, name), getattr(graph, name)), (t, name)
        for name in ("tok2slot", "slot2tok", "freebits", "dev_kv"):
            assert torch.equal(getattr(eager.cache, name), getattr(graph.cache, name)), (t, name)
        assert eager.status.item() == 0 and graph.status.item() == 0


def test_host_io_graph_equals_eager():
    """A step captured with its host I/O (pinned inputs in, slots and k-th scores out)
    gives the same outputs and tables as eager steps."""
    w = wl.scaled(wl.WORKLOADS["batch"], "hostio", B=2, lengths=(12000, 7000), k=512, C=1024)
    dev = "cuda"
    off = wl.tok_offsets(w.lengths)
    k8, ks = wl.make_keys(w, 0)
    wt = wl.make_weights(w, 0)
    host = wl.make_host_pool(w, 0, pin=True)
    eager = DecodeLayer(off, k8.to(dev), ks.to(dev), w.k, w.C, host)
    hio = DecodeLayer(off, k8.to(dev), ks.to(dev), w.k, w.C, host)
    qs = wl.QueryStream(w, 0)
    queries = [qs.next() for _ in range(5)]
    q_host = torch.empty_like(hio.q_in, device="cpu").pin_memory()
    w_host = wt.clone().pin_memory()
    slot_host = torch.empty_like(hio.sel_slot, device="cpu").pin_memory()
    kth_host = torch.empty_like(hio.kth, device="cpu").pin_memory()
    for lay in (eager, hio):
        lay.q_in.copy_(queries[0].to(dev))
        lay.w_in.copy_(wt.to(dev))
        lay.step()
    torch.cuda.synchronize()
    g = hio.capture_host_step(q_host, w_host, slot_host, kth_host)
    for t in range(1, 5):
        eager.q_in.copy_(queries[t].to(dev))
        eager.step()
        q_host.copy_(queries[t])
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(slot_host, eager.sel_slot.cpu()), t
        assert torch.equal(kth_host, eager.kth.cpu()), t
        for name in ("tok2slot", "slot2tok", "freebits", "dev_kv"):
            assert torch.equal(getattr(eager.cache, name), getattr(hio.cache, name)), (t, name)
        assert eager.status.item() == 0 and hio.status.item() == 0
    with pytest.raises(ValueError):
        hio.capture_host_step(q_host.to(dev), w_host, slot_host, kth_host)


@pytest.mark.parametrize("hold_early", [False, True])
def test_cross_layer_stack_in_one_graph(hold_early):
    # three layers in one CUDA graph; layers 1 and 2 fetch early what the layer before selected
    from tests._parity import run_stack
    w = wl.scaled(wl.WORKLOADS["tiny"], "xlayer", B=2, lengths=(3000, 5000), k=256, C=1024)
    rep = run_stack(w, steps=4, n_layers=3, cross_layer=True, hold_early=hold_early)
    # the seeded layers fetch early every selected token of the layer before that is not resident
    assert all(e > 0 for e in rep["early"][1][:2]) and all(e > 0 for e in rep["early"][2][:2])


def test_threshold_stack_eager():
    from tests._parity import run_stack
    w = wl.scaled(wl.WORKLOADS["tiny"], "stack", B=2, lengths=(3000, 1200), k=256, C=1024)
    run_stack(w, steps=3, n_layers=2, cross_layer=False, graph=False)


@pytest.mark.parametrize("hold_early", [False, True])
def test_shared_pool_in_one_graph(hold_early):
    # one pool of slots shared by the batch's requests; the pool smaller than B x C would be
    from tests._parity import run_pool
    w = wl.scaled(wl.WORKLOADS["batch"], "pool", B=3, lengths=(9000, 2000, 6000), k=512, C=1024)
    rep = run_pool(w, steps=5, pool=2048, hold_early=hold_early)
    assert sum(rep["early"]) > 0 and sum(rep["misses"]) > 0


def test_shared_pool_large_predictor_off_and_cap():
    # a pool above 2^17 slots (the walking cache step), predictor off; then a capped early set
    from tests._parity import run_pool
    w = wl.scaled(wl.WORKLOADS["batch"], "pool_big", B=2, lengths=(70000, 65000), k=2048, C=4096)
    run_pool(w, steps=3, pool=140032, predictor=False, graph=False)
    # more than 4096 selections (the walking step's wider per-thread chunks), predictor on
    w3 = wl.scaled(wl.WORKLOADS["batch"], "pool_big3", B=3, lengths=(70000, 65000, 30000), k=2048, C=4096)
    rep = run_pool(w3, steps=4, pool=140032)
    assert sum(rep["early"]) > 0
    w2 = wl.scaled(wl.WORKLOADS["batch"], "pool_cap", B=2, lengths=(8000, 5000), k=256, C=1024)
    run_pool(w2, steps=4, pool=1024, cap=100)


def test_shared_pool_ragged_batch():
    # an empty request, one shorter than k, and long ones sharing one pool
    from tests._parity import run_pool
    w = wl.scaled(wl.WORKLOADS["batch"], "pool_ragged", B=4, lengths=(7000, 0, 150, 3000), k=256, C=1024)
    run_pool(w, steps=4, pool=1024)
