"""GPU parity of the append path (echo_append_tokens) against the oracle: key
codes and scales, host-pool rows, the cache insert (lowest free slot, full
cache: host only), a full region, repeated appends; bit-exact throughout."""
import numpy as np
import pytest
import torch

from sparse_attention_kv_echo_gb300 import _lib as L

pytestmark = pytest.mark.gpu
dev = "cuda"
D, ROW = 128, 576


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.load(build_if_missing=True)


def _freebits_from(s2t, B, C):
    free = (s2t.reshape(B, C) == -1)
    words = np.zeros((B, C // 32), np.uint32)
    for j in range(32):
        words |= free[:, j::32].astype(np.uint32) << np.uint32(j)
    return words.reshape(-1)


def test_append_matches_oracle(orc):
    rng = np.random.default_rng(3)
    regions = [40, 9, 25, 3, 64]
    B, C = len(regions), 64
    off = np.concatenate([[0], np.cumsum(regions)]).astype(np.int64)
    n = int(off[-1])
    end = np.array([off[0] + 5, off[1] + 9, off[2] + 0, off[3] + 2, off[4] + 30], np.int64)   # request 1 full
    # cache state: request 2's slots all taken (host only), the others partly
    s2t = np.full(B * C, -1, np.int32)
    t2s = np.full(n, -1, np.int32)
    for b in range(B):
        used = np.arange(C) if b == 2 else rng.choice(C, int(rng.integers(0, C - 4)), replace=False)
        s2t[b * C + used] = 0    # occupied (the owner does not matter to the append)
    k8 = rng.integers(0, 256, (n, D), dtype=np.uint8)
    ks = rng.random(n, dtype=np.float32)
    host = torch.empty((n, ROW), dtype=torch.bfloat16).pin_memory()
    host.view(torch.int16).copy_(torch.from_numpy(rng.integers(-2**15, 2**15, (n, ROW), dtype=np.int16)))
    cache = L.LayerCache(B, n, C, host, device=dev)
    cache.slot2tok.copy_(torch.from_numpy(s2t))
    cache.tok2slot.copy_(torch.from_numpy(t2s))
    cache.freebits.copy_(torch.from_numpy(_freebits_from(s2t, B, C).view(np.int32)))
    dev_rows0 = rng.integers(-2**15, 2**15, (B * C, ROW), dtype=np.int16)
    cache.dev_kv.view(torch.int16).copy_(torch.from_numpy(dev_rows0))
    k8_d, ks_d = torch.from_numpy(k8).to(dev), torch.from_numpy(ks).to(dev)
    off_d, end_d = torch.from_numpy(off).to(dev), torch.from_numpy(end).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    # the oracle's copies
    o = dict(k8=k8.copy(), ks=ks.copy(), host=host.view(torch.uint8).numpy().copy(), t2s=t2s.copy(),
             s2t=s2t.copy(), dev=dev_rows0.view(np.uint8).reshape(B * C, -1).copy(), end=end.copy())
    for rep in range(3):
        k_new = rng.standard_normal((B, D), dtype=np.float32) * np.float32(3.0)
        k_new[3] = 0.0                                  # zero key: scale 0
        k_new[4, :] *= np.float32(1e30) if rep == 1 else np.float32(1.0)
        k_new[0, :] *= np.float32(1e-39 / 3.0) if rep == 2 else np.float32(1.0)   # a subnormal scale
        kv_new = rng.integers(-2**15, 2**15, (B, ROW), dtype=np.int16)
        L.append_tokens(off_d, end_d, n, torch.from_numpy(k_new).to(dev),
                        torch.from_numpy(kv_new).to(dev), k8_d, ks_d, cache, st)
        torch.cuda.synchronize()
        want_full = [int(o["end"][b] == off[b + 1]) for b in range(B)]   # request 1 from the start, 3 later
        full = orc.append_tokens(off, o["end"], k_new, kv_new.view(np.uint8), o["k8"], o["ks"], o["host"], C,
                                 o["t2s"], o["s2t"], o["dev"])
        assert full.tolist() == want_full and want_full[1] == 1
        assert int(st.item()) == L.ST_FULL
        assert np.array_equal(end_d.cpu().numpy(), o["end"])
        assert np.array_equal(k8_d.cpu().numpy(), o["k8"])
        assert np.array_equal(ks_d.cpu().numpy().view(np.uint32), o["ks"].view(np.uint32))
        assert np.array_equal(host.view(torch.uint8).numpy(), o["host"])
        assert np.array_equal(cache.tok2slot.cpu().numpy(), o["t2s"])
        assert np.array_equal(cache.slot2tok.cpu().numpy(), o["s2t"])
        assert np.array_equal(cache.freebits.cpu().numpy().view(np.uint32), _freebits_from(o["s2t"], B, C))
        assert np.array_equal(cache.dev_kv.view(torch.uint8).cpu().numpy().reshape(B * C, -1), o["dev"])
        st.zero_()


def test_append_rejects_nonfinite_key():
    B, C, n = 1, 32, 8
    off = torch.tensor([0, n], dtype=torch.int64, device=dev)
    end = torch.tensor([2], dtype=torch.int64, device=dev)
    host = torch.zeros((n, ROW), dtype=torch.bfloat16).pin_memory()
    cache = L.LayerCache(B, n, C, host, device=dev)
    k8 = torch.zeros((n, D), dtype=torch.uint8, device=dev)
    ks = torch.zeros(n, dtype=torch.float32, device=dev)
    k = torch.zeros((B, D), dtype=torch.float32, device=dev)
    k[0, 5] = float("nan")
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    L.append_tokens(off, end, n, k, torch.ones((B, ROW), dtype=torch.bfloat16, device=dev), k8, ks, cache, st)
    torch.cuda.synchronize()
    assert int(st.item()) == L.ST_NAN and int(end.item()) == 2
    assert not k8.any() and not host.view(torch.int16).any() and int(cache.slot2tok.max().item()) == -1


@pytest.mark.parametrize("hold_early", [False, True])
def test_decode_on_growing_contexts(hold_early):
    # decode steps and appends interleaved on regions with room for 3 more tokens, so the last
    # append of the 4-step run finds every region full (ECHO_ST_FULL, nothing written)
    from sparse_attention_kv_echo_gb300 import workloads as wl
    from tests._parity import run_decode_growing
    w = wl.scaled(wl.WORKLOADS["tiny"], "grow", B=3, lengths=(3000, 200, 5000), k=256, C=1024)
    grown = run_decode_growing(w, steps=4, room=3, hold_early=hold_early)
    assert grown.tolist() == [3, 3, 3]


def test_context_growing_from_empty():
    # request 0 starts with no token (its first append lands on its region's first row); request 1
    # is shorter than k; three decode steps with appends in between, checked step by step
    from sparse_attention_kv_echo_gb300 import workloads as wl
    from tests._parity import run_decode_growing
    w = wl.scaled(wl.WORKLOADS["tiny"], "grow0", B=2, lengths=(0, 180), k=256, C=1024)
    grown = run_decode_growing(w, steps=3, room=5)
    assert grown.tolist() == [3, 3]
