"""One layer's decode step through the libecho C ABI, on fixed-size buffers.

A DecodeLayer owns the torch tensors one layer needs for B requests (scores,
histogram, threshold state, selection, the GPU cache and its lists, the
quantised query) and issues the calls of a step:
    echo_quantize_q    -> E4M3 query, folded head weights, cleared histogram
    echo_index_scores  -> scores, shifted-score histogram, above-threshold bits,
                          free-bit snapshot, and (cands; by default when the
                          requests average 65536 tokens or more) each
                          request's candidate list for top-k
    echo_early_fetch   -> rows of the tokens above the predicted threshold,
                          copied from the host pool on the step's stream
                          (programmatic dependent of the score kernel) while
    echo_topk_select   -> exact top-k indices, k-th score, EMA threshold, and
    echo_cache_step    -> early set into the tables, free / allocate, slot of
                          every selection run on a side stream; the late-miss
                          recall joins the step's stream after both;
    echo_mla_decode    -> (attention=True) sparse MLA attention of each request
                          group over its selected slots, as soon as the group's
                          rows are in the cache.
Every buffer keeps its address and size, so ``step`` can be captured into a
CUDA graph and replayed; ``q_in``/``w_in`` are the inputs a graph reads.
``capture_host_step`` captures the step together with its host I/O (inputs
from pinned host buffers, selection slots and k-th scores back to pinned host
buffers), so one graph launch carries a whole step end to end.
"""
from __future__ import annotations

import math

import torch

from . import _lib as L


class DecodeLayer:
    def __init__(self, tok_off, k8: torch.Tensor, ks: torch.Tensor, k: int, C: int,
                 host_pool: torch.Tensor, alpha: float = 0.5, predictor: bool = True,
                 early_cap: int = -1, groups: int | None = None, first_share: float | None = None,
                 resolved: bool = True, hold_early: bool = False, attention: bool = False,
                 mla_scale: float = 1.0 / math.sqrt(192.0), tok_end=None, cross_layer: bool = False,
                 pool_slots: int = 0, cands: bool | None = None, cand_cap: int = L.CAND_CAP, lazy: bool = False,
                 device="cuda"):
        tok_off = torch.as_tensor(tok_off, dtype=torch.int64)
        self.B = int(tok_off.numel() - 1)
        self.n_tokens = int(k8.shape[0])
        self.k, self.C, self.alpha = int(k), int(C), float(alpha)
        self.predictor = bool(predictor)
        # top-k looks up the selected tokens' slots itself (the cache step then frees and places
        # the misses) when the request's free bits fit its shared memory
        # lazy: lazy-reuse eviction (a freed slot keeps its token until the slot is handed out); the
        # cache step then does the slot look-up itself
        self.lazy = bool(lazy)
        if self.lazy and hold_early:
            raise ValueError("lazy reuse goes with the contract's early slots, not the held-slot form")
        self.resolved = bool(resolved) and self.C <= L.TOPK_CACHED_MAX_SLOTS and not self.lazy
        # hold_early: the cache step holds the slots of unselected early tokens until the misses
        # are placed, so the late recall need not wait for the early copy; the early set is then
        # capped at C - k on top of the caller's cap (selected tokens plus held slots within C)
        self.hold_early = bool(hold_early)
        # (shared pool: the batch's selections and the held slots share the pool)
        room = (int(pool_slots) - self.B * self.k) if pool_slots else (self.C - self.k)
        if self.hold_early and (early_cap < 0 or early_cap > room):
            early_cap = room
        self.early_cap = int(early_cap)
        self.tok_off = tok_off.to(device)
        # growing contexts: request b's region is [tok_off[b], tok_off[b+1]) and tok_end[b] its current end
        # (append() adds a token); None: every region is full
        self.tok_end = None if tok_end is None else torch.as_tensor(tok_end, dtype=torch.int64).to(device)
        self.k8, self.ks = k8, ks
        f32 = dict(dtype=torch.float32, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        self.scores = torch.zeros(max(self.n_tokens, 1), **f32)
        self.hist = torch.zeros((self.B, 256), **i32)
        self.theta = torch.full((self.B,), math.inf, **f32)
        self.sel_idx = torch.full((self.B, self.k), -1, **i32)
        self.sel_slot = torch.full((self.B, self.k), -1, **i32)
        self.kth = torch.zeros((self.B,), **f32)
        # Requests are scored in groups (contiguous request ranges): the early fetch of group g
        # streams over the host link while group g+1 is scored, so the link starts sooner.
        # cross_layer: this layer's early set comes from the previous layer's selection (seed_from),
        # fetched before this layer scores; one request group
        self.cross_layer = bool(cross_layer) and self.predictor
        # pool_slots > 0: one cache pool of that many slots shared by every request (the worker's
        # device cache) instead of C slots per request; one request group
        self.pool_slots = int(pool_slots)
        if self.pool_slots and (cross_layer or attention):
            raise ValueError("the shared pool goes with neither cross_layer nor attention")
        if self.cross_layer or self.pool_slots:
            groups = 1
        if groups is None:
            # the early fetch of a group streams while the groups after it are scored: more groups
            # start the host link sooner (32 x 131072: 1 group 389, 2 629, 3 693, 4 737, 8 387 steps/s;
            # 8 x 32768: 2 groups best)
            groups = (4 if self.B >= 16 else 2) if (self.predictor and self.B >= 2) else 1
        groups = max(1, min(int(groups), self.B))
        bounds = [self.B * g // groups for g in range(groups + 1)]
        if first_share is not None and groups >= 2:
            # the first group's share of the requests (the rest split evenly): a smaller first group
            # starts the host link sooner
            f = min(self.B - (groups - 1), max(1, round(self.B * first_share)))
            bounds = [0] + [f + (self.B - f) * g // (groups - 1) for g in range(groups)]
        self.groups = [(bounds[g], bounds[g + 1]) for g in range(groups) if bounds[g + 1] > bounds[g]]
        # each group's above-threshold words: the groups' word ranges may overlap
        self.above_g = [torch.zeros(max(L.above_words(b1 - b0, self.n_tokens), 1), **i32)
                        for b0, b1 in self.groups]
        self.q8 = torch.zeros((self.B, L.HEADS, L.DIM), dtype=torch.uint8, device=device)
        self.qscale = torch.zeros((self.B, L.HEADS), **f32)
        self.wfold = torch.zeros((self.B, L.HEADS), **f32)
        self.status = torch.zeros(1, **i32)
        self.stats = torch.zeros(L.STATS_N, **i32)
        self.q_in = torch.zeros((self.B, L.HEADS, L.DIM), **f32)
        self.w_in = torch.zeros((self.B, L.HEADS), **f32)
        if self.pool_slots:
            # the pool is the cache of one request spanning every row: token ids are global
            self.cache = L.LayerCache(1, self.n_tokens, self.pool_slots, host_pool, device=device)
            self.tok_off_pool = torch.tensor([0, self.n_tokens], dtype=torch.int64, device=device)
            self.above_req = torch.zeros(max(L.above_words(self.B, self.n_tokens), 1), **i32)
            self.above_pool = torch.zeros(max(L.above_words(1, self.n_tokens), 1), **i32)
            self.sel_pool = torch.full((1, self.B * self.k), -1, **i32)
            self.slot_pool = torch.full((1, self.B * self.k), -1, **i32)
            self.resolved = False
        else:
            self.cache = L.LayerCache(self.B, self.n_tokens, self.C, host_pool, device=device)
        # sparse MLA attention over the selected slots (the cache rows are its 576-dim KV rows)
        self.attention, self.mla_scale = bool(attention), float(mla_scale)
        if self.attention:
            if self.cache.row_bytes != 2 * L.MLA_DQK:
                raise ValueError("attention needs 576-dim bf16 cache rows")
            self.mla_q = torch.zeros((self.B, L.MLA_HEADS, L.MLA_DQK), dtype=torch.bfloat16, device=device)
            self.attn_out = torch.zeros((self.B, L.MLA_HEADS, L.MLA_DV), **f32)
            self.attn_lse = torch.zeros((self.B, L.MLA_HEADS), **f32)
        self.views = [] if self.pool_slots else [self.cache.view(b0, b1) for b0, b1 in self.groups]
        # candidate lists: the score kernel lists each request's tokens above a cut that top-k sets
        # for the next step, and top-k selects among them when they hold the top-k
        # (default: lists when the requests average 65536 tokens or more -- at 32768 a list holds a
        # quarter of a request, and the 8-CTA clusters select faster)
        if cands is None:
            cands = self.n_tokens >= 65536 * self.B
        self.cands = L.Cands(self.B, cand_cap, device=device) if cands else None
        self.cands_g = ([self.cands.view(b0, b1) for b0, b1 in self.groups] if self.cands is not None
                        else [None] * len(self.groups))
        self.sides = [torch.cuda.Stream(device=device) for _ in self.groups]
        self.side = self.sides[0]
        # scoring streams of the groups after the first (the first uses the step's stream);
        # low priority, so the early fetch of the group before is placed first
        lo, _ = torch.cuda.Stream.priority_range()
        self.gstreams = [torch.cuda.Stream(device=device, priority=lo) for _ in self.groups[1:]]
        self.selected_evs = []     # after each group's top-k in the last enqueued step
        if self.cross_layer:
            self.above_seed = torch.zeros(max(L.above_words(self.B, self.n_tokens), 1), **i32)
            self.xfer = torch.cuda.Stream(device=device)
            self.seed_ev = None

    def reset(self):
        self.cache.reset()
        if self.cands is not None:
            self.cands.reset()
        self.theta.fill_(math.inf)
        self.status.zero_()
        self.stats.zero_()

    def seed_from(self, prev: "DecodeLayer"):
        """Cross-layer early fetch of this layer from the previous layer's selection (enqueue after
        prev.step and before this layer's step(seeded=True)): on this layer's transfer stream, after
        prev's top-k, the seed kernel marks prev's selected tokens that are not resident here and
        snapshots the free bits, and the early fetch streams their rows into this layer's cache
        while this layer has not scored yet.  The caller orders the transfer stream after this
        layer's previous step (DecodeStack forks it from the step's stream)."""
        if not self.cross_layer:
            raise ValueError("seed_from needs cross_layer=True")
        x = self.xfer
        for ev in prev.selected_evs:
            x.wait_event(ev)
        L.seed_early(self.tok_off, self.n_tokens, prev.sel_idx, self.above_seed, self.cache, self.status, stream=x,
                     tok_end=self.tok_end)
        self.seed_ev = torch.cuda.Event()
        self.seed_ev.record(x)
        L.early_fetch(self.tok_off, self.n_tokens, self.above_seed, self.early_cap, self.cache, self.status,
                      stream=x, tok_end=self.tok_end)

    def _quantize(self, q, w, stream):
        L.quantize_q(q, w, self.q8, self.qscale, self.wfold, self.status, hist=self.hist, stream=stream,
                     cand_cnt=None if self.cands is None else self.cands.cnt)

    def _select(self, off, b0, b1, cands, stream, cache=None, above=None, early_cap=-1, end=None):
        """Top-k of requests [b0, b1) on `stream` (off: their tok_off); with cache the cached form,
        which also writes sel_slot."""
        sl = slice(b0, b1)
        if self.cands is not None:
            L.topk_select_cands(off, self.n_tokens, self.scores, self.k, self.hist[sl], self.theta[sl], self.alpha,
                                cands, self.sel_idx[sl], self.kth[sl], self.status, stats=self.stats, stream=stream,
                                cache=cache, sel_slot=None if cache is None else self.sel_slot[sl], above=above,
                                early_cap=early_cap, tok_end=end)
        elif cache is not None:
            L.topk_select_cached(off, self.n_tokens, self.scores, self.k, self.hist[sl], self.theta[sl], self.alpha,
                                 self.sel_idx[sl], self.kth[sl], cache, self.sel_slot[sl], self.status,
                                 stats=self.stats, stream=stream, above=above, early_cap=early_cap, tok_end=end)
        else:
            L.topk_select(off, self.n_tokens, self.scores, self.k, self.hist[sl], self.theta[sl], self.alpha,
                          self.sel_idx[sl], self.kth[sl], self.status, stats=self.stats, stream=stream, tok_end=end)

    def _step_pool(self, q, w, main, out_host):
        # per-request scores and marks; the early fetch, top-k's slots and the cache step on the pool
        n, end = self.n_tokens, self.tok_end
        self._quantize(q, w, main)
        L.index_scores(self.tok_off, n, self.q8, self.wfold, self.k8, self.ks, self.scores, self.theta, self.hist,
                       self.status, above=self.above_req if self.predictor else None, stream=main, tok_end=end,
                       cands=self.cands)
        if self.predictor:
            L.pool_above(self.tok_off, n, self.above_req, self.cache, self.above_pool, self.status, stream=main,
                         tok_end=end)
            L.early_fetch(self.tok_off_pool, n, self.above_pool, self.early_cap, self.cache, self.status, stream=main)
        side = self.sides[0]
        side.wait_stream(main)
        copy = side if self.hold_early else main
        self._select(self.tok_off, 0, self.B, self.cands, side, end=end)
        ev = torch.cuda.Event()
        ev.record(side)
        self.selected_evs = [ev]
        L.pool_select(self.tok_off, self.sel_idx, self.sel_pool, stream=side)
        L.cache_step(self.tok_off_pool, n, self.sel_pool, self.cache, self.slot_pool, self.status, stats=self.stats,
                     stream=side, copy_stream=copy, above=self.above_pool if self.predictor else None,
                     early_cap=self.early_cap if self.predictor else 0, hold_early=self.hold_early,
                     lazy=self.lazy)
        L.pool_slots(self.sel_idx, self.slot_pool, self.sel_slot, stream=side)
        if out_host is not None:
            with torch.cuda.stream(side):
                self._write_out(out_host, 0, self.B)
        main.wait_stream(side)

    def _step_seeded(self, q, w, main, out_host, mla_q):
        # scores without threshold bits or snapshot; top-k and the cache step take the seeded set
        self._quantize(q, w, main)
        L.index_scores(self.tok_off, self.n_tokens, self.q8, self.wfold, self.k8, self.ks, self.scores, self.theta,
                       self.hist, self.status, stream=main, tok_end=self.tok_end, cands=self.cands)
        side = self.sides[0]
        side.wait_stream(main)
        if self.seed_ev is not None:
            side.wait_event(self.seed_ev)
        copy = side if self.hold_early else self.xfer
        self._select(self.tok_off, 0, self.B, self.cands, side, cache=self.cache if self.resolved else None,
                     above=self.above_seed, early_cap=self.early_cap, end=self.tok_end)
        ev = torch.cuda.Event()
        ev.record(side)
        self.selected_evs = [ev]
        if self.resolved:
            L.cache_step_resolved(self.tok_off, self.n_tokens, self.sel_idx, self.cache, self.sel_slot, self.status,
                                  stats=self.stats, stream=side, copy_stream=copy, hold_early=self.hold_early,
                                  tok_end=self.tok_end)
        else:
            L.cache_step(self.tok_off, self.n_tokens, self.sel_idx, self.cache, self.sel_slot, self.status,
                         stats=self.stats, stream=side, copy_stream=copy, above=self.above_seed,
                         early_cap=self.early_cap, hold_early=self.hold_early, tok_end=self.tok_end, lazy=self.lazy)
        if out_host is not None:
            with torch.cuda.stream(side):
                self._write_out(out_host, 0, self.B)
        if self.attention:
            copy.wait_stream(self.xfer)
            copy.wait_stream(side)
            self._attend(mla_q, 0, self.B, copy)
        main.wait_stream(side)
        main.wait_stream(self.xfer)

    def step(self, q: torch.Tensor | None = None, w: torch.Tensor | None = None, stream=None, out_host=None,
             mla_q: torch.Tensor | None = None, seeded: bool = False):
        """Enqueue one decode step (q [B,64,128] f32, w [B,64] f32; defaults q_in / w_in; pinned
        host tensors are read by the quantiser directly).

        stream: the step's stream (default: current).  Everything, the row copies
        included, is ordered before whatever is enqueued on `stream` next.
        out_host: optional (slot [B,k] int32, kth [B] f32) CUDA tensors over pinned host
        memory (_lib.host_alias_tensor): each request group's slots and k-th scores are
        written there by a kernel as soon as its cache step is done, while the late misses
        are still being recalled.
        mla_q: with attention=True, the step's MLA queries [B,128,576] bf16 (default
        self.mla_q); attn_out / attn_lse receive the attention of every request.
        seeded: (cross_layer) the early set is the one seed_from enqueued for this step."""
        q = self.q_in if q is None else q
        if self.attention:
            mla_q = self.mla_q if mla_q is None else mla_q
        w = self.w_in if w is None else w
        main = torch.cuda.current_stream() if stream is None else stream
        if self.pool_slots:
            self._step_pool(q, w, main, out_host)
            return
        if seeded:
            if not self.cross_layer:
                raise ValueError("seeded steps need cross_layer=True")
            self._step_seeded(q, w, main, out_host, mla_q)
            return
        self._quantize(q, w, main)
        if not self.predictor:
            L.index_scores(self.tok_off, self.n_tokens, self.q8, self.wfold, self.k8, self.ks, self.scores,
                           self.theta, self.hist, self.status, stream=main, tok_end=self.tok_end, cands=self.cands)
            self._select(self.tok_off, 0, self.B, self.cands, main, end=self.tok_end)
            L.cache_step(self.tok_off, self.n_tokens, self.sel_idx, self.cache, self.sel_slot, self.status,
                         stats=self.stats, stream=main, copy_stream=main, tok_end=self.tok_end, lazy=self.lazy)
            if out_host is not None:
                with torch.cuda.stream(main):
                    self._write_out(out_host, 0, self.B)
            if self.attention:
                self._attend(mla_q, 0, self.B, main)
            return
        sms = torch.cuda.get_device_properties(main.device).multi_processor_count
        scored, gstream = None, []
        end = (lambda b0, b1: None) if self.tok_end is None else (lambda b0, b1: self.tok_end[b0:b1])
        for g, (b0, b1) in enumerate(self.groups):
            s = main if g == 0 else self.gstreams[g - 1]
            if scored is not None:
                s.wait_event(scored)           # after the previous group's scores
            # while a group's early fetch holds its SMs, the next group's score kernel leaves them
            # (every earlier group's early fetch may still be copying)
            ctas = 0 if g == 0 else max(sms - L.EARLY_FETCH_BLOCKS * g, sms // 4)
            L.index_scores(self.tok_off[b0:b1 + 1], self.n_tokens, self.q8[b0:b1], self.wfold[b0:b1], self.k8,
                           self.ks, self.scores, self.theta[b0:b1], self.hist[b0:b1], self.status,
                           above=self.above_g[g], cache=self.views[g], stream=s, ctas=ctas, tok_end=end(b0, b1),
                           cands=self.cands_g[g])
            scored = torch.cuda.Event()
            scored.record(s)
            gstream.append(s)
            # the group's early rows stream over the host link on `s` (programmatic dependent of its
            # score kernel) while the next group is scored
            L.early_fetch(self.tok_off[b0:b1 + 1], self.n_tokens, self.above_g[g], self.early_cap, self.views[g],
                          self.status, stream=s, tok_end=end(b0, b1))
        # top-k and the table update of every group on the groups' side streams once all scores are
        # done (a top-k started earlier would take SMs the next score kernel counts on); the late
        # misses of a group follow its early fetch on the group's stream (a slot fetched early and
        # then freed may go to a miss), or, holding those slots, its cache step on the side stream
        self.selected_evs = []
        for g, (b0, b1) in enumerate(self.groups):
            side = self.sides[g]
            copy = side if self.hold_early else gstream[g]
            side.wait_event(scored)
            off = self.tok_off[b0:b1 + 1]
            if self.resolved:
                # top-k looks up every selected token's slot (resident or early)
                self._select(off, b0, b1, self.cands_g[g], side, cache=self.views[g], above=self.above_g[g],
                             early_cap=self.early_cap, end=end(b0, b1))
                ev = torch.cuda.Event()
                ev.record(side)
                self.selected_evs.append(ev)
                L.cache_step_resolved(off, self.n_tokens, self.sel_idx[b0:b1], self.views[g], self.sel_slot[b0:b1],
                                      self.status, stats=self.stats, stream=side, copy_stream=copy,
                                      hold_early=self.hold_early, tok_end=end(b0, b1))
            else:
                self._select(off, b0, b1, self.cands_g[g], side, end=end(b0, b1))
                ev = torch.cuda.Event()
                ev.record(side)
                self.selected_evs.append(ev)
                L.cache_step(off, self.n_tokens, self.sel_idx[b0:b1], self.views[g], self.sel_slot[b0:b1],
                             self.status, stats=self.stats, stream=side, copy_stream=copy, above=self.above_g[g],
                             early_cap=self.early_cap, hold_early=self.hold_early, tok_end=end(b0, b1),
                             lazy=self.lazy)
            if out_host is not None:
                with torch.cuda.stream(side):
                    self._write_out(out_host, b0, b1)
            if self.attention:
                # after the group's late recall (on `copy`) and its early rows (on its scoring stream)
                if copy is not gstream[g]:
                    copy.wait_stream(gstream[g])
                self._attend(mla_q, b0, b1, copy)
        for gs in self.gstreams:
            main.wait_stream(gs)
        for side in self.sides:
            main.wait_stream(side)

    def append(self, k_new: torch.Tensor, kv_new: torch.Tensor, stream=None):
        """Enqueue the append of one new token per request (k_new [B,128] f32, kv_new [B,576] bf16,
        device): its E4M3 key and scale at tok_end[b], its row in the host pool and, when a slot is
        free, in the cache; tok_end advances (a full region sets ECHO_ST_FULL).  Needs tok_end."""
        if self.tok_end is None:
            raise ValueError("append needs growing contexts (tok_end)")
        if self.pool_slots:
            # echo_append_tokens places each request in its own slot range; a shared pool would
            # need one allocation across the requests
            raise ValueError("append goes with per-request slot ranges, not the shared pool")
        main = torch.cuda.current_stream() if stream is None else stream
        L.append_tokens(self.tok_off, self.tok_end, self.n_tokens, k_new, kv_new, self.k8, self.ks, self.cache,
                        self.status, stream=main)

    def _attend(self, mla_q, b0, b1, stream):
        C = self.C
        L.mla_decode(mla_q[b0:b1], self.sel_slot[b0:b1], self.cache.dev_kv[b0 * C:b1 * C], C, self.mla_scale,
                     self.attn_out[b0:b1], self.attn_lse[b0:b1], self.status, stream=stream)

    def _write_out(self, out_host, b0, b1):
        # elementwise kernels, not copy-engine transfers: their stores go straight to the
        # host memory behind the alias, with no copy-engine launch in the graph
        torch.bitwise_or(self.sel_slot[b0:b1], 0, out=out_host[0][b0:b1])
        torch.mul(self.kth[b0:b1], 1.0, out=out_host[1][b0:b1])

    def capture_host_step(self, q_host: torch.Tensor, w_host: torch.Tensor, slot_host: torch.Tensor,
                          kth_host: torch.Tensor, stream=None) -> torch.cuda.CUDAGraph:
        """A CUDA graph of one step with its host I/O: the quantiser reads q_host [B,64,128]
        f32 and w_host [B,64] f32 (pinned) directly, the step runs, and sel_slot / kth are
        copied out to slot_host [B,k] int32 / kth_host [B] f32 (pinned) per request group
        as soon as they are final.  The buffers are bound to the graph: refill
        q_host/w_host before a replay, read the outputs after it."""
        for t, like in ((q_host, self.q_in), (w_host, self.w_in), (slot_host, self.sel_slot), (kth_host, self.kth)):
            if t.device.type != "cpu" or not t.is_pinned() or t.shape != like.shape or t.dtype != like.dtype:
                raise ValueError("host I/O buffers must be pinned CPU tensors shaped like q_in, w_in, "
                                 "sel_slot and kth")
        cap = torch.cuda.Stream(device=self.q_in.device) if stream is None else stream
        cap.wait_stream(torch.cuda.current_stream(self.q_in.device))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            # the graph reads and writes these buffers through their aliases: keep them alive
            self._host_io = getattr(self, "_host_io", []) + [(q_host, w_host, slot_host, kth_host)]
            out = (L.host_alias_tensor(slot_host, self.q_in.device), L.host_alias_tensor(kth_host, self.q_in.device))
            with torch.cuda.graph(g, stream=cap):
                self.step(q_host, w_host, stream=cap, out_host=out)
        torch.cuda.current_stream(self.q_in.device).wait_stream(cap)
        return g

    def kernel_launches_per_step(self) -> int:
        # quantize, then per group: score (+ early fetch) + top-k + cache step + late recall
        att = 1 if self.attention else 0
        if self.pool_slots:  # quantize, score, top-k, select, cache step, recall, slots (+ marks, early fetch)
            return 7 + (2 if self.predictor else 0)
        if not self.predictor:
            return 5 + att
        if self.cross_layer:  # quantize, score, top-k, cache step, recall + seed, early fetch (seeded steps)
            return 7 + att
        return 1 + (5 + att) * len(self.groups)


class DecodeStack:
    """Several layers of one decode step, in order.  cross_layer: every layer after the first
    takes its early set from the layer before (DecodeLayer.seed_from): its rows stream while the
    earlier layers finish and it scores.  The first layer keeps the threshold predictor."""

    def __init__(self, layers: list[DecodeLayer], cross_layer: bool = False):
        self.layers = layers
        self.cross_layer = bool(cross_layer)
        if self.cross_layer and not all(l.cross_layer for l in layers[1:]):
            raise ValueError("layers after the first need cross_layer=True")

    def step(self, qs, ws, stream=None, between=None, out_host=None):
        """qs / ws: per layer the step's query [B,64,128] and weights [B,64] (f32; pinned host
        tensors are read by the quantisers directly).
        between(stream): optional work enqueued on the step's stream after each layer but the last
        (the rest of a transformer layer -- attention, MLP -- that separates two indexers).
        out_host: optional per layer (slot [B,k] int32, kth [B] f32) CUDA tensors over pinned host
        memory, written as each layer's request groups finish (DecodeLayer.step)."""
        main = torch.cuda.current_stream() if stream is None else stream
        if self.cross_layer:  # the transfer streams follow everything before this step
            for lay in self.layers[1:]:
                lay.xfer.wait_stream(main)
        for i, lay in enumerate(self.layers):
            seeded = self.cross_layer and i > 0
            if seeded:
                lay.seed_from(self.layers[i - 1])
            lay.step(qs[i], ws[i], stream=main, seeded=seeded, out_host=None if out_host is None else out_host[i])
            if between is not None and i + 1 < len(self.layers):
                between(main)

    def capture_host_step(self, q_host: torch.Tensor, w_host: torch.Tensor, slot_host: torch.Tensor,
                          kth_host: torch.Tensor, stream=None) -> torch.cuda.CUDAGraph:
        """A CUDA graph of one step of every layer with its host I/O: layer l's quantiser reads
        q_host[l] [B,64,128] f32 and w_host[l] [B,64] f32 (pinned) directly, and its slots and k-th
        scores go to slot_host[l] [B,k] int32 / kth_host[l] [B] f32 (pinned) as soon as each request
        group's are final.  The buffers are bound to the graph: refill the inputs before a replay,
        read the outputs after it."""
        lays = self.layers
        n = len(lays)
        for t, like in ((q_host, lays[0].q_in), (w_host, lays[0].w_in), (slot_host, lays[0].sel_slot),
                        (kth_host, lays[0].kth)):
            if (t.device.type != "cpu" or not t.is_pinned() or not t.is_contiguous()
                    or tuple(t.shape) != (n,) + tuple(like.shape) or t.dtype != like.dtype):
                raise ValueError("host I/O buffers must be pinned, contiguous CPU tensors shaped like "
                                 "[layers] + q_in, w_in, sel_slot and kth")
        dev = lays[0].q_in.device
        cap = torch.cuda.Stream(device=dev) if stream is None else stream
        cap.wait_stream(torch.cuda.current_stream(dev))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            # the graph reads and writes these buffers through their aliases: keep them alive
            self._host_io = getattr(self, "_host_io", []) + [(q_host, w_host, slot_host, kth_host)]
            outs = [(L.host_alias_tensor(slot_host[i], dev), L.host_alias_tensor(kth_host[i], dev)) for i in range(n)]
            with torch.cuda.graph(g, stream=cap):
                self.step([q_host[i] for i in range(n)], [w_host[i] for i in range(n)], stream=cap, out_host=outs)
        torch.cuda.current_stream(dev).wait_stream(cap)
        return g

    def kernel_launches_per_step(self) -> int:
        return sum(l.kernel_launches_per_step() for l in self.layers)
