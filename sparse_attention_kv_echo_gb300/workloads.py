"""Seeded synthetic inputs shaped like the ECHO evaluation workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path and the CPU oracle consume the bytes
it produces.  Keys are stored the way a DeepSeek-V3.2 index cache stores them
(E4M3 bytes with one fp32 scale per token); the cast to E4M3 is torch's own
``float8_e4m3fn`` conversion, a library routine shared with neither side.

Workloads (all seeded, seed 0 unless stated):
  tiny     1 request x 8192 tokens, 1 layer, k=256, 1024 slots, 16 steps
  batch    8 x 32768, 1 layer, k=2048, 4096 slots/request, 64 steps
  v32      32 x 131072, 4 layers (independent keys and pools), k=2048,
           8192 slots/request/layer, 5% hot tokens (+2.0 before quantising), 128 steps
  prefill  1 x 102400-token prompt, 2048-row query blocks, k=2048 per row, 260000 slots
  skewed   64 requests, lengths log-uniform in [4096, 262144], 2 layers, k=2048,
           2560 slots/request, queries re-drawn every 8 steps, 96 steps
  layers   8 x 32768, 4 layers whose keys and queries are correlated layer to layer
           (rho = 0.9: layer l = rho * layer l-1 + sqrt(1 - rho^2) * fresh N(0,1)),
           k=2048, 4096 slots/request/layer, 64 steps -- the shape the cross-layer
           prefetch assumes (consecutive layers select mostly the same tokens)
Queries q ~ N(0,1) [64,128] fp32 drift as q_t = 0.9 q_{t-1} + 0.44 eps_t; head
weights w ~ U(0,1); host KV rows are 576 bf16 values ~ N(0,1) (1152 bytes).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

H = 64          # index heads
D = 128         # index head dim
KV_DIM = 576    # bf16 values per KV row
ROW_BYTES = KV_DIM * 2


@dataclass(frozen=True)
class Workload:
    name: str
    B: int                      # requests
    L: int                      # layers (independent keys, pools and caches)
    lengths: tuple              # tokens per request
    k: int
    C: int                      # GPU slots per request per layer
    steps: int
    drift: str = "ar"           # "ar": AR(0.9) every step; "redraw8": i.i.d. redraw every 8 steps
    hot_frac: float = 0.0
    hot_offset: float = 0.0
    predictor: bool = True
    prefill_block: int = 0      # > 0: chunked prefill with this many rows per block
    seed: int = 0
    layer_rho: float = 0.0      # > 0: keys, queries and weights correlated from layer to layer

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))


def _skewed_lengths(B: int, seed: int) -> tuple:
    rng = np.random.default_rng(seed * 1000003 + 4)
    u = rng.uniform(math.log(4096), math.log(262144), size=B)
    return tuple(int(round(math.exp(x))) for x in u)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, (8192,), 256, 1024, 16),
    "batch": Workload("batch", 8, 1, (32768,) * 8, 2048, 4096, 64),
    "layers": Workload("layers", 8, 4, (32768,) * 8, 2048, 4096, 64, layer_rho=0.995),
    "v32": Workload("v32", 32, 4, (131072,) * 32, 2048, 8192, 128, hot_frac=0.05, hot_offset=2.0),
    "prefill": Workload("prefill", 1, 1, (102400,), 2048, 260000, 50, prefill_block=2048),
    "skewed": Workload("skewed", 64, 2, _skewed_lengths(64, 0), 2048, 2560, 96, drift="redraw8"),
}


def scaled(w: Workload, name: str, **kw) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    d = dict(w.__dict__)
    d.update(kw)
    d["name"] = name
    return Workload(**d)


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + stream)
    return g


def tok_offsets(lengths) -> np.ndarray:
    off = np.zeros(len(lengths) + 1, np.int64)
    off[1:] = np.cumsum(np.asarray(lengths, np.int64))
    return off


def make_keys(w: Workload, layer: int, device="cpu", requests=None):
    """E4M3 index keys [sum N, 128] (uint8) and per-token fp32 scales [sum N] of one layer.

    Each key row ~ N(0,1) (plus hot_offset on a hot subset of hot_frac of each
    request's tokens, drawn uniformly without replacement), then stored as
    E4M3 bytes with scale amax/448 per token.  requests: only these requests'
    rows, concatenated in the order given (each request has its own generator,
    so its bytes are the same as in the full set)."""
    rows = []
    scales = []
    for b in (range(w.B) if requests is None else requests):
        n = w.lengths[b]
        g = _gen(device, w.seed, 10_000 + 1000 * layer + b)
        if w.layer_rho > 0:
            kf = _correlated((n, D), w, layer, 10_000 + b, device)
        else:
            kf = torch.randn((n, D), generator=g, device=device, dtype=torch.float32)
        if w.hot_frac > 0:
            nh = int(round(w.hot_frac * n))
            perm = torch.randperm(n, generator=g, device=device)[:nh]
            kf[perm] += w.hot_offset
        amax = kf.abs().amax(dim=1)
        amax = torch.where(amax > 0, amax, torch.ones_like(amax))
        s = amax / 448.0
        k8 = (kf / s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        rows.append(k8)
        scales.append(s)
    return torch.cat(rows, 0).contiguous(), torch.cat(scales, 0).contiguous()


def _correlated(shape, w: Workload, layer: int, sub: int, device) -> torch.Tensor:
    """N(0,1) draws of `layer` that correlate rho with the same draws of layer - 1."""
    x = torch.randn(shape, generator=_gen(device, w.seed, sub), device=device, dtype=torch.float32)
    c = math.sqrt(1.0 - w.layer_rho ** 2)
    for j in range(1, layer + 1):
        z = torch.randn(shape, generator=_gen(device, w.seed, sub + 1000 * j), device=device, dtype=torch.float32)
        x = w.layer_rho * x + c * z
    return x


def make_weights(w: Workload, layer: int, device="cpu") -> torch.Tensor:
    """Per-head weights w ~ U(0,1), [B, 64] fp32 (the same for every layer when layer_rho > 0)."""
    g = _gen(device, w.seed, 20_000 + (0 if w.layer_rho > 0 else layer))
    return torch.rand((w.B, H), generator=g, device=device, dtype=torch.float32)


class QueryStream:
    """Index queries [B, 64, 128] fp32 of one layer, step after step."""

    def __init__(self, w: Workload, layer: int, device="cpu"):
        self.w = w
        self.g = _gen(device, w.seed, 30_000 + layer)
        self.device = device
        self.t = 0
        self.q = torch.randn((w.B, H, D), generator=self.g, device=device, dtype=torch.float32)
        # correlated layers: this layer's query = rho * the layer before's + sqrt(1 - rho^2) * its own
        self.prev = None
        if w.layer_rho > 0 and layer > 0:
            self.prev = QueryStream(w, layer - 1, device)

    def next(self) -> torch.Tensor:
        """The query of the current step; advances the stream."""
        out = self.q.clone()
        if self.prev is not None:
            out = self.w.layer_rho * self.prev.next() + math.sqrt(1.0 - self.w.layer_rho ** 2) * out
        self.t += 1
        eps = torch.randn(self.q.shape, generator=self.g, device=self.device, dtype=torch.float32)
        if self.w.drift == "redraw8" and self.t % 8 == 0:
            self.q = eps
        else:
            self.q = 0.9 * self.q + 0.44 * eps
        return out


def _huge_page_bytes() -> int:
    """The transparent huge page size of this kernel (0 when it has none)."""
    try:
        with open("/sys/kernel/mm/transparent_hugepage/enabled") as f:
            if "[never]" in f.read():
                return 0
        with open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size") as f:
            return int(f.read().strip())
    except (OSError, ValueError):
        return 0


def _madvise_collapse(addr: int, length: int) -> None:
    import ctypes
    if length <= 0:
        return
    try:
        libc = ctypes.CDLL(None, use_errno=True)
        libc.madvise.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
        libc.madvise(ctypes.c_void_p(addr), ctypes.c_size_t(length), 25)   # MADV_COLLAPSE
    except (OSError, AttributeError):
        pass


def _huge_mapping(nbytes: int, hp: int):
    """A private anonymous mapping of nbytes, aligned to the huge page size hp and advised for
    huge pages, its pages faulted in; returns (mapping, byte view)."""
    import mmap
    region = mmap.mmap(-1, nbytes + hp, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    whole = np.frombuffer(region, dtype=np.uint8)
    off = (-whole.ctypes.data) % hp
    region.madvise(mmap.MADV_HUGEPAGE, off, len(region) - off)
    buf = whole[off:off + nbytes]
    # fault the pages in, then ask the kernel to collapse what did not come as huge pages
    # (MADV_COLLAPSE, Linux 6.1+; a refusal leaves the small pages in place)
    buf[::mmap.PAGESIZE] = 0
    _madvise_collapse(buf.ctypes.data, nbytes - nbytes % hp)
    # then keep the kernel's background collapsing away from these pages: once registered they
    # cannot move, and repeated attempts on them only disturb the GPU's host reads
    if hasattr(mmap, "MADV_NOHUGEPAGE"):
        region.madvise(mmap.MADV_NOHUGEPAGE, off, len(region) - off)
    return region, buf


def pinned_empty(shape, dtype) -> torch.Tensor:
    """An uninitialised host tensor whose pages are locked and mapped for the GPU
    (cudaHostRegister), sized exactly: torch's pinned allocator rounds every
    block up to a power of two, which for a multi-GB host pool nearly doubles
    the locked memory.  A buffer of at least one transparent huge page is a
    private anonymous mapping advised for huge pages (aligned to their size), so
    that the GPU's random row reads over the host link touch few page
    translations; smaller ones are a numpy buffer.  The tensor's storage keeps
    the bytes alive (views included); the registration is dropped just before
    they are freed."""
    import mmap
    import weakref
    nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    if nbytes == 0:
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    hp = _huge_page_bytes()
    if hp and nbytes >= hp and hasattr(mmap, "MADV_HUGEPAGE"):
        # After other work has fragmented memory a mapping may get only part of its huge pages
        # (and the GPU's host reads from the rest are slow and easily congested).  Each try
        # compacts memory further; the earlier tries stay mapped until the end so that a new
        # one cannot get their small pages back: up to six tries, keeping the best
        tries = []
        for _ in range(6):
            region, buf = _huge_mapping(nbytes, hp)
            tries.append((_huge_share_range(buf.ctypes.data, buf.ctypes.data + nbytes), region, buf))
            if tries[-1][0] >= 1.0:
                break
        _, region, buf = max(tries, key=lambda t: t[0])
        del tries
    else:
        buf = np.empty(nbytes, np.uint8)
    rt = torch.cuda.cudart()
    rc = rt.cudaHostRegister(buf.ctypes.data, nbytes, 3)   # portable | mapped
    if int(rc) != 0:
        raise RuntimeError(f"cudaHostRegister failed ({int(rc)})")
    weakref.finalize(buf, rt.cudaHostUnregister, buf.ctypes.data)
    return torch.from_numpy(buf).view(dtype).view(shape)


def _huge_share_range(lo: int, hi: int) -> float:
    """Share of the bytes [lo, hi) of this process that sit on transparent huge pages (from
    /proc/self/smaps; -1 when that cannot be read)."""
    try:
        huge = 0
        with open("/proc/self/smaps") as f:
            start = end = None
            for line in f:
                head = line.split()
                if "-" in head[0] and len(head) > 4 and not head[0].endswith(":"):
                    a, b = head[0].split("-")
                    start, end = int(a, 16), int(b, 16)
                elif head[0] == "AnonHugePages:" and start is not None and start < hi and end > lo:
                    huge += int(head[1]) * 1024
        return min(1.0, huge / max(1, hi - lo))
    except (OSError, ValueError, IndexError):
        return -1.0


def huge_page_share(t: torch.Tensor) -> float:
    """Share of a host tensor's bytes that sit on transparent huge pages (-1: unknown)."""
    lo = t.data_ptr()
    return _huge_share_range(lo, lo + t.numel() * t.element_size())


def make_host_pool(w: Workload, layer: int, device="cpu", pin: bool = False, rows: int | None = None) -> torch.Tensor:
    """Host KV pool [sum N, 576] bf16 ~ N(0,1) of one layer (pinned when pin=True).

    With device='cuda' the values are drawn on the GPU and copied to host memory.
    rows: only the first `rows` rows, a multiple of the 65536-row draw (the same
    values as in the whole pool: the draws are made in that order)."""
    g = _gen(device, w.seed, 40_000 + layer)
    chunk = 1 << 16
    n = w.total_tokens if rows is None else int(rows)
    if n != w.total_tokens and n % chunk:
        raise ValueError("a partial host pool takes a multiple of 65536 rows")
    if pin:
        out = pinned_empty((n, KV_DIM), torch.bfloat16)
    else:
        out = torch.empty((n, KV_DIM), dtype=torch.bfloat16)
    for r0 in range(0, n, chunk):
        r1 = min(n, r0 + chunk)
        out[r0:r1].copy_(torch.randn((r1 - r0, KV_DIM), generator=g, device=device,
                                     dtype=torch.float32).to(torch.bfloat16))
    return out


def make_prefill_queries(w: Workload, block: int, device="cpu"):
    """Queries [R, 64, 128] fp32 (i.i.d. N(0,1) per row) and weights [R, 64] U(0,1) of one block."""
    R = min(w.prefill_block, w.total_tokens - block * w.prefill_block)
    g = _gen(device, w.seed, 50_000 + block)
    q = torch.randn((R, H, D), generator=g, device=device, dtype=torch.float32)
    wt = torch.rand((R, H), generator=g, device=device, dtype=torch.float32)
    return q, wt
