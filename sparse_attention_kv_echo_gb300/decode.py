"""One layer's decode step through the libecho C ABI, on fixed-size buffers.

A DecodeLayer owns the torch tensors one layer needs for B requests (scores,
histogram, threshold state, selection, the GPU cache and its lists, the
quantised query) and issues the calls of a step:
    echo_quantize_q    -> E4M3 query, folded head weights, cleared histogram
    echo_index_scores  -> scores, shifted-score histogram, above-threshold bits,
                          free-bit snapshot
    echo_early_fetch   -> rows of the tokens above the predicted threshold,
                          copied from the host pool on the step's stream
                          (programmatic dependent of the score kernel) while
    echo_topk_select   -> exact top-k indices, k-th score, EMA threshold, and
    echo_cache_step    -> early set into the tables, free / allocate, slot of
                          every selection run on a side stream; the late-miss
                          recall joins the step's stream after both.
Every buffer keeps its address and size, so ``step`` can be captured into a
CUDA graph and replayed; ``q_in``/``w_in`` are the inputs a graph reads.
"""
from __future__ import annotations

import math

import torch

from . import _lib as L


class DecodeLayer:
    def __init__(self, tok_off, k8: torch.Tensor, ks: torch.Tensor, k: int, C: int,
                 host_pool: torch.Tensor, alpha: float = 0.5, predictor: bool = True,
                 early_cap: int = -1, device="cuda"):
        tok_off = torch.as_tensor(tok_off, dtype=torch.int64)
        self.B = int(tok_off.numel() - 1)
        self.n_tokens = int(k8.shape[0])
        self.k, self.C, self.alpha = int(k), int(C), float(alpha)
        self.predictor, self.early_cap = bool(predictor), int(early_cap)
        self.tok_off = tok_off.to(device)
        self.k8, self.ks = k8, ks
        f32 = dict(dtype=torch.float32, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        self.scores = torch.zeros(max(self.n_tokens, 1), **f32)
        self.hist = torch.zeros((self.B, 256), **i32)
        self.theta = torch.full((self.B,), math.inf, **f32)
        self.sel_idx = torch.full((self.B, self.k), -1, **i32)
        self.sel_slot = torch.full((self.B, self.k), -1, **i32)
        self.kth = torch.zeros((self.B,), **f32)
        self.above = torch.zeros(max(L.above_words(self.B, self.n_tokens), 1), **i32)
        self.q8 = torch.zeros((self.B, L.HEADS, L.DIM), dtype=torch.uint8, device=device)
        self.qscale = torch.zeros((self.B, L.HEADS), **f32)
        self.wfold = torch.zeros((self.B, L.HEADS), **f32)
        self.status = torch.zeros(1, **i32)
        self.stats = torch.zeros(L.STATS_N, **i32)
        self.q_in = torch.zeros((self.B, L.HEADS, L.DIM), **f32)
        self.w_in = torch.zeros((self.B, L.HEADS), **f32)
        self.cache = L.LayerCache(self.B, self.n_tokens, self.C, host_pool, device=device)
        self.side = torch.cuda.Stream(device=device)

    def reset(self):
        self.cache.reset()
        self.theta.fill_(math.inf)
        self.status.zero_()
        self.stats.zero_()

    def step(self, q: torch.Tensor | None = None, w: torch.Tensor | None = None, stream=None):
        """Enqueue one decode step (q [B,64,128] f32, w [B,64] f32; defaults q_in / w_in).

        stream: the step's stream (default: current).  Everything, the row copies
        included, is ordered before whatever is enqueued on `stream` next."""
        q = self.q_in if q is None else q
        w = self.w_in if w is None else w
        main = torch.cuda.current_stream() if stream is None else stream
        above = self.above if self.predictor else None
        L.quantize_q(q, w, self.q8, self.qscale, self.wfold, self.status, hist=self.hist, stream=main)
        L.index_scores(self.tok_off, self.n_tokens, self.q8, self.wfold, self.k8, self.ks, self.scores,
                       self.theta, self.hist, self.status, above=above,
                       cache=self.cache if self.predictor else None, stream=main)
        if self.predictor:
            # the early rows stream over the host link on `main` while top-k and
            # the table update run on the side stream
            self.side.wait_stream(main)
            L.early_fetch(self.tok_off, self.n_tokens, self.above, self.early_cap, self.cache, self.status,
                          stream=main)
            work = self.side
        else:
            work = main
        L.topk_select(self.tok_off, self.n_tokens, self.scores, self.k, self.hist, self.theta, self.alpha,
                      self.sel_idx, self.kth, self.status, stats=self.stats, stream=work)
        L.cache_step(self.tok_off, self.n_tokens, self.sel_idx, self.cache, self.sel_slot, self.status,
                     stats=self.stats, stream=work, copy_stream=main, above=above, early_cap=self.early_cap)

    def kernel_launches_per_step(self) -> int:
        # quantize + score (+ early fetch) + top-k + cache step + late recall
        return 2 + (1 if self.predictor else 0) + 1 + 2
