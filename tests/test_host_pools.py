"""Host-side logic of the page-locked host pools and the bench's host counters (CPU only: nothing
here registers memory with CUDA).  The pools are private anonymous mappings aligned to the
transparent huge page size and advised for huge pages; the share of a range on huge pages is read
from /proc/self/smaps."""
import mmap

import numpy as np
import pytest
import torch

from sparse_attention_kv_echo_gb300 import workloads as wl


def test_huge_page_size_is_a_power_of_two_or_zero():
    hp = wl._huge_page_bytes()
    assert hp >= 0
    if hp:
        assert hp & (hp - 1) == 0 and hp % mmap.PAGESIZE == 0


def test_mapping_is_aligned_sized_and_zeroed_where_touched():
    hp = wl._huge_page_bytes()
    if not hp or not hasattr(mmap, "MADV_HUGEPAGE"):
        pytest.skip("no transparent huge pages on this kernel")
    nbytes = 2 * hp + 12345
    region, buf = wl._huge_mapping(nbytes, hp)
    assert buf.size == nbytes and buf.dtype == np.uint8
    assert buf.ctypes.data % hp == 0
    assert np.all(buf[::mmap.PAGESIZE] == 0)
    buf[-1] = 7                      # the whole range is writable
    share = wl._huge_share_range(buf.ctypes.data, buf.ctypes.data + nbytes)
    assert share == -1.0 or 0.0 <= share <= 1.0
    del buf, region


def test_share_of_ordinary_memory():
    t = torch.ones(1 << 16)
    s = wl.huge_page_share(t)
    assert s == -1.0 or 0.0 <= s <= 1.0
    assert wl._huge_share_range(0, 4096) in (0.0, -1.0)     # nothing of this process is mapped there


def test_vmstat_counters_and_deltas():
    import bench
    a = bench.vmstat()
    assert all(isinstance(v, int) for v in a.values())
    b = {k: v + 3 for k, v in a.items()}
    assert bench.vm_delta(a, b) == {k: 3 for k in a}
