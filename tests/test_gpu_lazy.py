"""GPU parity of the lazy-reuse eviction variant (ECHO_CACHE_LAZY) against the oracle's own lazy
cache: a freed slot keeps its token (a ghost) until the slot is handed out, a selected ghost is a
hit.  Every step bit-exact on early lists, top-k, slots, miss lists, tables and free bits; every
present token's device row (ghosts included) equals its host row; the GPU's revival count equals
the oracle's."""
import pytest

from sparse_attention_kv_echo_gb300 import _lib as L
from sparse_attention_kv_echo_gb300 import workloads as wl
from tests._parity import run_decode, run_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.load(build_if_missing=True)


def test_lazy_tiny_workload_all_steps():
    w = wl.WORKLOADS["tiny"]
    rep = run_decode(w, w.steps, predictor=True, lazy=True)
    assert rep["revived"] == rep["revived_gpu"]
    assert rep["revived"] > 0                # early-fetched tokens top-k skipped, selected later


def test_lazy_ragged_batch_and_redraws():
    w = wl.scaled(wl.WORKLOADS["skewed"], "lazy_burst", B=4, lengths=(9000, 4096, 20000, 5000), C=2560)
    rep = run_decode(w, 10, predictor=True, lazy=True, score_sample=512)
    assert rep["revived"] == rep["revived_gpu"]
    w2 = wl.scaled(wl.WORKLOADS["tiny"], "lazy_ragged", B=5, lengths=(3000, 200, 0, 1, 4173), k=256, C=320)
    run_decode(w2, 6, predictor=True, lazy=True)


def test_lazy_predictor_off_and_a_cap():
    w = wl.scaled(wl.WORKLOADS["tiny"], "lazy_cap", lengths=(6000,))
    run_decode(w, 6, predictor=False, lazy=True)
    rep = run_decode(w, 6, predictor=True, cap=40, lazy=True)
    assert rep["revived"] == rep["revived_gpu"]


def test_lazy_shared_pool():
    """The batch's shared pool with lazy reuse (one cache of one request over every row)."""
    w = wl.scaled(wl.WORKLOADS["batch"], "lazy_pool", B=3, lengths=(9000, 20000, 4000), k=512, C=1024)
    rep = run_pool(w, steps=6, pool=4096, lazy=True)
    assert min(rep["misses"][1:]) >= 0
