"""Chunked prefill through the libecho C ABI: one prompt, blocks of query rows.

A PrefillRunner owns the fixed-size buffers of one prompt (the row-strided
score workspace, per-row histograms and selections, the union of a block's
selections, the GPU cache over the whole prompt) and issues one
echo_prefill_block call per block: the block's recall runs on a copy stream
while the next block is scored.
"""
from __future__ import annotations

import math

import torch

from . import _lib as L


class PrefillRunner:
    def __init__(self, k8: torch.Tensor, ks: torch.Tensor, k: int, C: int, host_pool: torch.Tensor,
                 block_rows: int, alpha: float = 0.5, device="cuda"):
        self.n_keys = int(k8.shape[0])
        self.W = self.n_keys                      # row stride: the whole prompt
        self.R = int(block_rows)
        self.k, self.C, self.alpha = int(k), int(C), float(alpha)
        if self.C < self.W:
            raise ValueError("the prompt's cache needs C >= prompt length")
        self.k8, self.ks = k8, ks
        f32 = dict(dtype=torch.float32, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        self.scores = torch.zeros((self.R, self.W), **f32)
        self.hist = torch.zeros((self.R, 256), **i32)
        self.sel_idx = torch.full((self.R, self.k), -1, **i32)
        self.kth = torch.zeros(self.R, **f32)
        self.theta = torch.full((1,), math.inf, **f32)
        self.union_list = torch.full((self.W,), -1, **i32)
        self.union_count = torch.zeros(1, **i32)
        self.union_bits = torch.zeros((self.W + 31) // 32, **i32)
        self.sel_slot = torch.full((self.W,), -1, **i32)
        self.ws = torch.zeros(L.prefill_workspace_size(self.R, self.W), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, **i32)
        self.stats = torch.zeros(L.STATS_N, **i32)
        self.cache = L.LayerCache(1, self.n_keys, self.C, host_pool, device=device)
        self.copy = torch.cuda.Stream(device=device)

    def blocks(self):
        return (self.n_keys + self.R - 1) // self.R

    def block(self, i: int, q: torch.Tensor, w: torch.Tensor, stream=None):
        """Enqueue block i (q [R_i,64,128], w [R_i,64] on the device)."""
        row0 = i * self.R
        R = min(self.R, self.n_keys - row0)
        assert q.shape[0] == R and w.shape[0] == R
        L.prefill_block(R, row0, self.n_keys, q, w, self.k8, self.ks, self.k, self.theta, self.alpha,
                        self.scores, self.W, self.hist, self.sel_idx, self.kth, self.union_list,
                        self.union_count, self.union_bits, self.cache, self.sel_slot, self.ws, self.status,
                        stats=self.stats, stream=stream, copy_stream=self.copy)
        return row0, R

    def wait_recall(self, stream=None):
        (torch.cuda.current_stream() if stream is None else stream).wait_stream(self.copy)
