/*
 * echo.h -- C ABI of libecho, the GB300 (sm_103a) decode hot path of ECHO,
 * lossless KV-cache offloading for sparse-attention LLMs.
 *
 * Per layer and decode step the path computes, for a batch of B requests:
 *   1. the indexer score of every context token (echo_quantize_q,
 *      echo_index_scores), then the rows of the tokens above the predicted
 *      threshold fetched early (echo_early_fetch) while
 *   2. the exact top-k tokens and the EMA threshold prediction
 *      (echo_topk_select),
 *   3. the GPU-cache step: free unselected slots, allocate slots for the
 *      misses, recall the missing KV rows from the host pool (echo_cache_step);
 * and, for chunked prefill, a block of query rows at once (echo_prefill_block).
 *
 * Sources (page title, then section):
 *   [EXPL] "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs",
 *          section 2 "The top-k dependency" and its panels.
 *   [AE]   "OSDI'26 Artifact Evaluation for ECHO: Efficient KV Cache Offloading
 *          with Lossless Prefetching for Serving Native Sparse Attention LLMs",
 *          sections "Download the model", "Baselines under evaluation",
 *          "Fused Prefetch Kernels (ECHO only)".
 *   [IDX]  The DeepSeek-V3.2 lightning-indexer score computed here:
 *          I[s] = sum_h w[h] * ReLU(q[h] . k[s]), 64 heads x 128 dims, keys
 *          stored as E4M3 bytes with one fp32 scale per token.
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers owned by the caller unless stated.  The
 *     library allocates nothing, keeps no state between calls, never
 *     synchronises the device and never reads device memory from the host;
 *     every call only enqueues work on the given stream(s), so a whole decode
 *     step can be captured into one CUDA graph.
 *   - Requests are ragged (CSR): tok_off[B+1] (int64, device, non-decreasing,
 *     tok_off[0] = 0, tok_off[B] <= n_tokens) gives request b the token rows
 *     [tok_off[b], tok_off[b+1]) of every per-token array.  Token indices in
 *     selections and slot tables are request-local (0 .. N_b - 1).
 *     n_tokens is the number of rows allocated in the per-token arrays; it
 *     is a host value and fixed for a captured graph, the lengths are data.
 *   - Return value: ECHO_OK or a negative ECHO_E* code from host-side
 *     argument checks (nothing is enqueued then).  Conditions found on the
 *     device are OR-ed as ECHO_ST_* bits into *status (int32, device), which
 *     the caller clears and reads when it likes; the kernels never trap.
 *   - stats (optional, may be NULL): uint32 device counters [ECHO_STATS_N],
 *     accumulated (never cleared by the library).
 *   - Every wait inside a kernel is bounded; a wait that runs out sets
 *     ECHO_ST_TIMEOUT and the kernel returns.
 */
#ifndef ECHO_H
#define ECHO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* echo_stream_t; /* a cudaStream_t; NULL = legacy default stream */

/* host-side return codes */
#define ECHO_OK 0
#define ECHO_EINVAL (-1)        /* NULL pointer, negative size, misaligned pointer */
#define ECHO_ECAPACITY (-2)     /* k > C, C not a multiple of 32 */
#define ECHO_EUNSUPPORTED (-3)  /* B above ECHO_MAX_REQUESTS, row size not a multiple of 16 */
#define ECHO_ECUDA (-4)         /* a CUDA launch or driver call failed */
#define ECHO_ETOOLARGE (-5)     /* the call needs more than its fixed device scratch holds */

/* device status bits (OR-ed into *status) */
#define ECHO_ST_TIMEOUT 0x1     /* a bounded wait ran out; outputs of that call are invalid */
#define ECHO_ST_NAN 0x2         /* NaN/Inf in q or w, or a NaN score */
#define ECHO_ST_NOSLOT 0x4      /* a miss found no free slot (cannot happen when k <= C) */
#define ECHO_ST_BADDATA 0x8     /* tok_off/tables/selection/histogram inconsistent with the sizes given */
#define ECHO_ST_FULL 0x10       /* echo_append_tokens: a request's region had no room (nothing written) */

/* stats counters (uint32 each) */
#define ECHO_STAT_TOPK_FALLBACK 0   /* top-k boundary bins too large for shared memory */
#define ECHO_STAT_BOUNDARY_MAX 1    /* largest boundary-bin population seen */
#define ECHO_STAT_EARLY 2           /* tokens fetched early (above the prediction) */
#define ECHO_STAT_MISSES 3          /* tokens recalled after top-k */
#define ECHO_STAT_EARLY_USED 4      /* early-fetched tokens that top-k then selected */
#define ECHO_STAT_CAND_MISS 5       /* top-k given candidate lists that selected from all the scores */
#define ECHO_STAT_REVIVED 6         /* lazy reuse: freed tokens selected again while their slot kept them */
#define ECHO_STATS_N 8

/* echo_cache_step flags */
#define ECHO_CACHE_HOLD_EARLY 1     /* hold the unselected early tokens' slots until the misses are placed */
#define ECHO_CACHE_LAZY 2           /* lazy-reuse eviction: a freed slot keeps its token until handed out */

/*
 * Requests.  tok_off [B+1] (int64, device) gives request b its region of rows
 * [tok_off[b], tok_off[b+1]) in every per-token array (keys, scales, scores,
 * tok2slot, host pool).  tok_end [B] (int64, device, optional: NULL = every
 * region full) gives the request's current end, tok_off[b] <= tok_end[b] <=
 * tok_off[b+1]: a context that grows by echo_append_tokens inside its region.
 * Tokens in [tok_end[b], tok_off[b+1]) are not part of the request; every call
 * of one step must see the same tok_end.  Inconsistent bounds give an empty
 * request and ECHO_ST_BADDATA.
 */
#define ECHO_HEADS 64           /* index heads */
#define ECHO_DIM 128            /* index head dimension (bytes per E4M3 key row) */
#define ECHO_MAX_REQUESTS 4096  /* requests per call */

/*
 * GPU cache of one layer for B requests [EXPL panels "Five fixed-size integer
 * tensors on the GPU" and "One layer, one step: free -> allocate -> recall"].
 * Every array has a fixed size, so nothing changes length from step to step.
 * Initial state: tok2slot and slot2tok all -1, freebits all ones, counts 0.
 *   tok2slot  [n_tokens] int32   slot of each token in its request's slot range, -1 = not resident
 *   slot2tok  [B*C]      int32   request-local token held by each slot, -1 = free
 *   freebits  [B*C/32]   uint32  bit (j%32) of word j/32 set <=> slot j of that request is free
 *   miss_tok  [B*C]      int32   this step's late misses per request (ascending tokens)
 *   miss_slot [B*C]      int32   the slot each late miss was given
 *   miss_cnt  [B]        int32
 *   early_tok [B*C]      int32   this step's early fetches per request (ascending tokens)
 *   early_slot[B*C]      int32   the slot each early fetch was given
 *   early_cnt [B]        int32
 *   free_snap [B*C/32]   uint32  freebits as echo_index_scores found them (echo_early_fetch
 *                                reads this copy while echo_cache_step updates freebits)
 *   host_kv   device-accessible address of the pinned host KV pool [n_tokens, row_bytes]
 *             (cudaHostAlloc'd or registered; the address the device uses for it)
 *   dev_kv    [B*C, row_bytes] device cache rows; request b owns rows [b*C, (b+1)*C)
 * C is a multiple of 32 and at most 524288 (2^19; ECHO_EUNSUPPORTED above);
 * row_bytes a multiple of 16 (1152 for 576 bf16 values).
 * Row copies read the (token, slot) lists of the late misses or free_snap
 * (early fetch), never the live tables, so a table update may overlap them; a consumer of
 * dev_kv must wait for the copy stream.
 */
typedef struct echo_cache {
    int32_t* tok2slot;
    int32_t* slot2tok;
    uint32_t* freebits;
    int32_t* miss_tok;
    int32_t* miss_slot;
    int32_t* miss_cnt;
    int32_t* early_tok;
    int32_t* early_slot;
    int32_t* early_cnt;
    uint32_t* free_snap;
    const void* host_kv;
    void* dev_kv;
    int64_t row_bytes;
    int32_t C;
    int32_t reserved;
} echo_cache;

/*
 * Query quantisation [IDX; the sources only say the score GEMM runs in FP8].
 * Per (request, head): scale = the smallest power of two 2^e with
 * max_d |q[b,h,d]| <= 448 * 2^e (e >= -126; 1 for an all-zero row),
 * q8[b,h,d] = E4M3 round-to-nearest-even(q / scale), and
 * wfold[b,h] = w[b,h] * scale (fp32).
 *   q [B,64,128] f32 (16-byte aligned), w [B,64] f32
 *   -> q8 [B,64,128] u8, qscale [B,64] f32, wfold [B,64] f32 (16-byte aligned).
 *   q and w may be device memory or pinned host memory given by its device
 *   alias (echo_host_device_alias); the kernel reads each element once, so a
 *   step's inputs need no separate host-to-device copy.
 *   hist [B,256] u32 (may be NULL) is set to zero, ready for echo_index_scores;
 *   cand_cnt [B] int32 (may be NULL; the cnt of an echo_cands) is set to zero,
 *   ready for echo_index_scores_cands.
 * NaN/Inf in q or w -> ECHO_ST_NAN.
 */
int echo_quantize_q(int B, const float* q, const float* w, uint8_t* q8, float* qscale,
                    float* wfold, uint32_t* hist, int32_t* cand_cnt, int32_t* status, echo_stream_t stream);

/*
 * Indexer score of every token [IDX] and the 256-bin histogram of the
 * threshold-shifted scores [EXPL panel "Prefill: one-round histogram"].
 *   scores[t] = ks[t] * sum_h wfold[b,h] * max(0, sum_d q8[b,h,d] * k8[t,d])
 *   for every token row t of request b, which equals the definition
 *   sum_h w[h] * ReLU(q[h] . k[t]) over the dequantised E4M3 values.
 *   Inputs: q8 [B,64,128] u8 and wfold [B,64] f32 from echo_quantize_q,
 *   k8 [n_tokens,128] E4M3 bytes, ks [n_tokens] f32 (q8, k8 and ks 16-byte
 *   aligned; with a cache, its tok2slot too).
 *   Outputs: scores [n_tokens] f32 (rows outside every request untouched);
 *   hist [B,256] u32 (may be NULL): ADDS, per request, the counts of
 *   bin = top 8 bits of orderkey(fp32(score - shift)), shift = theta_hat[b]
 *   when finite, else 0, so it must hold zeros on entry (echo_quantize_q
 *   clears it); orderkey maps a float to a uint32 in the same order (-0
 *   counted as +0).  theta_hat [B] f32 may be NULL (no shift).
 *   above (may be NULL): [echo_above_words(B, n_tokens)] u32, the tokens with
 *   score > theta_hat[b] (none when theta_hat[b] is not finite) that are not
 *   resident in `cache` (NULL: residency not considered), for echo_early_fetch.
 *   Request b's words start at 4 * (floor(tok_off[b] / 128) + b); bit j of
 *   its word w is its token 32*w + j; words past its last token hold zeros.
 *   cache (may be NULL; needs above): the layer's cache; its freebits are
 *   also copied to free_snap for echo_early_fetch.
 *   ctas: CTAs of the score kernel, one per SM at most (<= 0: one per SM).
 *   Pass fewer when other kernels will hold SMs while this one runs (e.g. the
 *   early fetch of another group of requests), so that none of its CTAs
 *   waits for an SM.
 */
size_t echo_above_words(int B, int64_t n_tokens);
int echo_index_scores(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, const uint8_t* q8,
                      const float* wfold, const uint8_t* k8, const float* ks, float* scores,
                      const float* theta_hat, uint32_t* hist, uint32_t* above,
                      const echo_cache* cache, int ctas, int32_t* status, echo_stream_t stream);

/*
 * Early fetch [EXPL panel "Decode: fetch above a predicted threshold"], the
 * copy half.  Before top-k is known, the early set of request b is the tokens
 * marked in `above` by echo_index_scores (score > the predicted threshold,
 * not resident), in ascending order, at most min(early_cap, free slots) of
 * them (early_cap < 0: no cap but the free slots); they take the lowest free
 * slots in ascending order (free as in cache->free_snap).  This call copies
 * their rows host_kv[tok_off[b] + t] -> dev_kv[b*C + slot] and lists them in
 * early_tok / early_slot (ranks 0 .. E-1); it touches no table: the tables
 * learn the early set in echo_cache_step (given the same above and
 * early_cap), which may therefore run concurrently with this copy.
 * Enqueue it on the stream of echo_index_scores right after it: it is
 * launched as a programmatic dependent of the score kernel.  It reads neither
 * the scores nor the threshold, so echo_topk_select may run on another stream
 * meanwhile.  The late-miss recall of echo_cache_step must be ordered after
 * it (its copy_stream = this stream), since a slot fetched early and then
 * freed may be handed to a miss, unless the cache step holds those slots
 * (ECHO_CACHE_HOLD_EARLY).
 */
int echo_early_fetch(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, const uint32_t* above,
                     int early_cap,
                     const echo_cache* cache, int32_t* status, echo_stream_t stream);

/*
 * Exact top-k per request [EXPL section 2: "guarantees an exact top-k"] and
 * the EMA threshold update [EXPL panel "Decode: fetch above a predicted
 * threshold": EMA with alpha = 0.5 of the previous k-th score].
 *   sel_idx [B,k] int32: the min(k, N_b) highest scores of request b, equal
 *   scores resolved towards the lower index, written in ascending index
 *   order and padded with -1.  kth [B] f32: the k-th highest score (the
 *   smallest selected one when N_b < k; -inf when N_b = 0).
 *   theta_hat [B] in/out (may be NULL): +inf -> kth; else
 *   alpha*kth + (1-alpha)*theta_hat, each operation rounded in fp32;
 *   unchanged when N_b = 0.
 *   hist [B,256] as written by echo_index_scores with the same theta_hat, or
 *   NULL (then it is computed here).  The selection never depends on the
 *   histogram or the prediction; they only decide how much work it takes (a
 *   histogram that does not describe the scores is rebuilt and flagged
 *   ECHO_ST_BADDATA).
 * The kernel lets a programmatic dependent launch (echo_cache_step) start as
 * soon as it begins; it writes sel_idx, kth and theta_hat only.
 */
int echo_topk_select(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, const float* scores,
                     int k,
                     const uint32_t* hist, float* theta_hat, float alpha, int32_t* sel_idx,
                     float* kth, int32_t* status, uint32_t* stats, echo_stream_t stream);

/*
 * GPU-cache step [EXPL panel "One layer, one step: free -> allocate ->
 * recall"; panel "Decode: fetch above a predicted threshold"]: with sel [B,m]
 * (ascending request-local tokens, -1 padded):
 *   0. with above (may be NULL: no early fetch this step), the early set of
 *      echo_early_fetch (same above and early_cap) becomes resident in the
 *      slots that call copied it to, and early_cnt[b] = its size E (0
 *      without above);
 *   1. every resident token that is not selected is freed (both table
 *      entries -1, its free bit set); its bytes stay, nothing is written
 *      back.  With flags & ECHO_CACHE_HOLD_EARLY, the slot of an early token
 *      of this step is held until step 2 is done instead (its early copy may
 *      still be in flight) and is free after the step;
 *   2. the selected tokens that are not resident (the misses), in ascending
 *      order, take the lowest free slots in ascending order;
 *   3. sel_slot [B,m] = slot of each selected token (-1 for padding);
 *   4. the miss rows are copied host_kv[tok_off[b] + t] -> dev_kv[b*C + slot],
 *      on copy_stream (which may equal stream: then as a programmatic
 *      dependent of steps 0-3; else an event orders it after them).
 * Needs m <= C; holding, also m + (unselected early tokens) <= C, which an
 * early_cap of at most C - m guarantees (else a miss may find no slot:
 * ECHO_ST_NOSLOT).  Holding, the recall may run before echo_early_fetch's
 * copy ends.  flags: 0, ECHO_CACHE_HOLD_EARLY or ECHO_CACHE_LAZY (other bits,
 * or both: ECHO_EINVAL).
 * Lazy-reuse eviction (ECHO_CACHE_LAZY; a variant -- a reading of "freed slots
 * keep their token until overwritten" -- not the contract): a
 * token freed in step 1 keeps its bytes and both table entries (a ghost: its
 * slot is free, the token still maps to it) until its slot is handed to
 * another token, which drops it from the tables; every early token of step 0
 * enters the tables in its slot (dropping the ghost there), a selected one
 * stays resident, an unselected one becomes a ghost; in step 2 a selected
 * ghost is a hit, resident again in its slot with no copy
 * (ECHO_STAT_REVIVED); a miss that takes a ghost's slot drops the ghost.
 * Ghosts map to their slots, so echo_index_scores leaves them out of the
 * early set (their bytes are in the cache).  The tables keep every present
 * token (resident or ghost) mutually inverse; freebits mark the slots no
 * resident token holds.  Not with echo_cache_step_resolved or the held-slot
 * form (ECHO_EUNSUPPORTED / ECHO_EINVAL); the look-up is the cache step's.
 * Steps 0-3 are launched as a programmatic dependent of the
 * kernel before them on `stream`: while that kernel still runs (if it lets
 * dependents start early, as echo_topk_select and echo_index_scores do) they
 * may read slot2tok and freebits, which none of this library's kernels but
 * this step writes; sel and above are read only after that kernel has
 * completed.
 */
int echo_cache_step(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, const int32_t* sel,
                    int m,
                    const uint32_t* above, int early_cap, const echo_cache* cache, int32_t* sel_slot,
                    int32_t* status, uint32_t* stats, echo_stream_t stream, echo_stream_t copy_stream,
                    int flags);

/*
 * The two calls above with the cache step's look-up done by top-k:
 * echo_topk_select_cached is echo_topk_select (m = k) that also writes, for
 * every selected entry, sel_slot[b,i] = the slot the token holds at the
 * start of the cache step (step 0 of echo_cache_step: its resident slot, or
 * for a token of the early set, given above and early_cap as there, the
 * slot echo_early_fetch copied it to, which this call enters into tok2slot
 * and slot2tok), -1 for a miss or padding, and early_cnt[b] = E.  The
 * request's free bits must be as echo_early_fetch saw them (nothing between
 * the two calls changes them).  Needs C <= 32768 (ECHO_EUNSUPPORTED
 * otherwise) and reads the free bits and tables of `cache`.
 * echo_cache_step_resolved then does steps 1-4 of echo_cache_step with those
 * slots (sel_slot in/out, early_cnt in, the same flags), launched the same way; needs
 * C <= 131072.  Together they give exactly the tables, slots, lists and rows
 * of echo_topk_select followed by echo_cache_step.
 */
int echo_topk_select_cached(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                            const float* scores, int k,
                            const uint32_t* hist, float* theta_hat, float alpha, int32_t* sel_idx, float* kth,
                            const uint32_t* above, int early_cap, const echo_cache* cache, int32_t* sel_slot,
                            int32_t* status, uint32_t* stats, echo_stream_t stream);
int echo_cache_step_resolved(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                             const int32_t* sel, int m,
                             const echo_cache* cache, int32_t* sel_slot, int32_t* status, uint32_t* stats,
                             echo_stream_t stream, echo_stream_t copy_stream, int flags);

/*
 * Decode top-k over candidate lists [EXPL section 2 "The top-k dependency":
 * an exact top-k after the scores; what the lists change is only how much of
 * the scores top-k reads].  The score kernel appends, per request, every
 * token whose score has order key >= cut[b] to the request's list; when a
 * request's list holds at least k and at most cap tokens it contains every
 * token of the top-k (the k-th score is then >= the cut), and top-k selects
 * among those alone; otherwise it selects from all the scores as
 * echo_topk_select does.  Top-k sets cut[b] for the next step: the score of
 * rank 4k of this step (from the list, or the lower edge of a histogram bin
 * when the list cannot tell), a guess that only decides which path the next
 * step takes.  Selections, k-th scores, thresholds, slots and tables are the
 * same as without lists.
 *   key [B*cap] u32   order keys of the candidates' scores (request b: [b*cap, (b+1)*cap))
 *   idx [B*cap] int32 request-local token of each candidate, in no particular order
 *   cnt [B]     int32 candidates found; may exceed cap (the list then holds only
 *                     cap of them and top-k reads all the scores); cleared by
 *                     echo_quantize_q before every score call
 *   cut [B]     u32   0xFFFFFFFF = no list (the initial value); written by top-k
 *   cap               entries per request, > 0
 */
typedef struct echo_cands {
    uint32_t* key;
    int32_t* idx;
    int32_t* cnt;
    uint32_t* cut;
    int32_t cap;
    int32_t reserved;
} echo_cands;

/*
 * echo_index_scores that also fills the candidate lists: cands->cnt must hold
 * zeros on entry (echo_quantize_q clears it); cands->cut is read.  A NaN score
 * sets ECHO_ST_NAN here (top-k over a list reads only the list).  All other
 * arguments and outputs as echo_index_scores.
 */
int echo_index_scores_cands(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                            const uint8_t* q8, const float* wfold, const uint8_t* k8, const float* ks,
                            float* scores, const float* theta_hat, uint32_t* hist, uint32_t* above,
                            const echo_cache* cache, const echo_cands* cands, int ctas, int32_t* status,
                            echo_stream_t stream);

/*
 * Top-k from candidate lists, one thread block per request: echo_topk_select
 * (cache NULL; sel_slot, above and early_cap unused) or
 * echo_topk_select_cached (cache given: sel_slot, early_cnt and the early
 * set's table entries as described there, C <= 32768), with the lists the
 * score call filled (cands may be NULL: every request selects from all its
 * scores).  scores, hist and theta_hat as for those calls; hist may be NULL.
 * Selecting from all the scores, the boundary bin's entries are gathered into
 * shared memory (up to 16384 of them; past that the bin is selected by passes
 * over the scores, counted in ECHO_STAT_TOPK_FALLBACK).  A request that had a
 * list (cut < 0xFFFFFFFF) but selected from all its scores is counted in
 * ECHO_STAT_CAND_MISS.  Lets a programmatic dependent launch start as soon as
 * it begins, like echo_topk_select.
 */
int echo_topk_select_cands(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                           const float* scores, int k, const uint32_t* hist, float* theta_hat, float alpha,
                           const echo_cands* cands, int32_t* sel_idx, float* kth, const uint32_t* above,
                           int early_cap, const echo_cache* cache, int32_t* sel_slot, int32_t* status,
                           uint32_t* stats, echo_stream_t stream);

/*
 * Chunked prefill [EXPL panel "Prefill: one-round histogram"; AE section
 * "Fused Prefetch Kernels (ECHO only)", inter-query prefetch].
 *
 * echo_prefill_scores: scores of one block of R query rows against the
 * prompt's keys, causal.  Row r sits at position row0 + r and sees keys
 * [0, row0 + r] (itself included); its scores go to scores[r*W + s] for
 * s <= row0 + r (the rest of the row is untouched), with
 * scores = ks[s] * sum_h wfold[r,h] * max(0, sum_d q8[r,h,d] * k8[s,d]).
 * hist [R,256] (may be NULL) ADDS the per-row counts of the 256 bins of
 * orderkey(fp32(score - theta)) >> 24, theta = *theta_hat when finite else 0
 * (one scalar for the block).  Needs row0 + R <= n_keys and W >= row0 + R.
 */
int echo_prefill_scores(int R, int64_t row0, int64_t n_keys, const uint8_t* q8, const float* wfold,
                        const uint8_t* k8, const float* ks, float* scores, int64_t W,
                        const float* theta_hat, uint32_t* hist, int32_t* status, echo_stream_t stream);

/* Bytes of device workspace echo_prefill_block needs for R rows and row stride W. */
size_t echo_prefill_workspace_size(int R, int64_t W);

/*
 * One prefill block: on `stream`, quantise the R rows q [R,64,128] / w [R,64]
 * (echo_quantize_q), score them (echo_prefill_scores into scores [R,W] and
 * hist [R,256]), select each row's exact top-k over its causal prefix into
 * sel_idx [R,k] (ascending, -1 padded; every token when row0 + r + 1 <= k)
 * with its k-th score in kth [R], then the union of the rows' selections:
 * union_list [W] (ascending, -1 padded), *union_count, union_bits
 * [ceil(W/32)] (may be NULL), and the block threshold update
 * *theta_hat <- EMA(alpha) with the last row's k-th score (+inf: replaced).
 * With a cache (B = 1 over the whole prompt, C >= W): the cache step on the
 * union (free the rest, misses -> lowest free slots; sel_slot [W]) after the
 * previous block's recall has read its lists, and the recall of the misses on
 * copy_stream, which overlaps the next block's scoring on `stream`.
 * ws: echo_prefill_workspace_size(R, W) bytes, 256-byte aligned.
 */
int echo_prefill_block(int R, int64_t row0, int64_t n_keys, const float* q, const float* w,
                       const uint8_t* k8, const float* ks, int k, float* theta_hat, float alpha,
                       float* scores, int64_t W, uint32_t* hist, int32_t* sel_idx, float* kth,
                       int32_t* union_list, int32_t* union_count, uint32_t* union_bits,
                       const echo_cache* cache, int32_t* sel_slot, void* ws, size_t ws_bytes,
                       int32_t* status, uint32_t* stats, echo_stream_t stream,
                       echo_stream_t copy_stream);

/*
 * Allocation-free variant of echo_prefill_block (the pages have no
 * counterpart: this is a library service, not part of the method).
 *
 * For callers that cannot provide device workspace: a runtime that reserves
 * all of its device memory up front and may not allocate again, an embedder
 * without an allocator of its own, or a latency-critical thread that cannot
 * afford the device synchronisation cudaMalloc may imply.  It runs the same
 * block as echo_prefill_block, with the same arguments minus ws / ws_bytes;
 * the workspace lives in a fixed device array inside the library, of
 * ECHO_PREFILL_STATIC_SCRATCH_BYTES, which every GPU that loads the library
 * keeps until the process exits.  It allocates nothing.
 *   - Limit: blocks whose workspace (echo_prefill_workspace_size(R, W)) is
 *     larger than the array return ECHO_ETOOLARGE and enqueue nothing; a
 *     2048-row block of a 102400-token prompt needs about 18 MB.
 *   - The first call on each device looks up the array's device address with
 *     that device current (again after the device's context is replaced, e.g.
 *     by cudaDeviceReset); make that first call before any stream capture: a
 *     lookup that would happen while `stream` is capturing returns
 *     ECHO_EINVAL and enqueues nothing.
 *   - All calls on a device share the one array and it keeps the previous
 *     call's contents; the block clears what must start at zero itself.
 *     Calls whose work overlaps on the GPU (other streams, other threads)
 *     race on the array: order them on one stream or serialise them.  A call
 *     on the stream and copy stream of the previous call is ordered after that
 *     call's recall (still running on the copy stream) before it rewrites
 *     anything the recall reads.
 */
#define ECHO_PREFILL_STATIC_SCRATCH_BYTES (32u << 20)
int echo_prefill_block_static(int R, int64_t row0, int64_t n_keys, const float* q, const float* w,
                              const uint8_t* k8, const float* ks, int k, float* theta_hat, float alpha,
                              float* scores, int64_t W, uint32_t* hist, int32_t* sel_idx, float* kth,
                              int32_t* union_list, int32_t* union_count, uint32_t* union_bits,
                              const echo_cache* cache, int32_t* sel_slot, int32_t* status, uint32_t* stats,
                              echo_stream_t stream, echo_stream_t copy_stream);

/*
 * Failure-path knob, for tests (the pages have no counterpart).  Every wait
 * inside a kernel gives up after a limit (2 s) and reports ECHO_ST_TIMEOUT
 * instead of hanging.  With limit_ns >= 0, the score kernel's epilogue (on the
 * current device) first waits on a barrier that nothing arrives on, giving up
 * after limit_ns: every score call then takes its timeout path -- it sets
 * ECHO_ST_TIMEOUT, its outputs are invalid, and its kernel drains its copies
 * and MMAs before it frees tensor memory and exits, so the next call runs
 * normally.  limit_ns < 0 turns the wait off (the default).  The waits that
 * drain are never shortened.  Synchronous (a copy to device memory); not for
 * use while a score call is in flight.
 */
int echo_debug_stall_epilogue(int64_t limit_ns);

/*
 * Sparse MLA decode attention over the selected slots [EXPL section 2: a
 * decode step attends over the k selected tokens only; the formula is
 * DeepSeek-V3.2's sparse MLA in its absorbed form, the pages give none]:
 * per request b and head h, over the entries i with sel_slot[b,i] >= 0,
 *   s_i = scale * sum_{d<576} q[b,h,d] * kv[b*C + sel_slot[b,i], d],
 *   out[b,h,:] = sum_i softmax(s)_i * kv[b*C + sel_slot[b,i], 0:512],
 *   lse[b,h] = log sum_i exp(s_i)   (out = 0, lse = -inf with no valid slot).
 *   q [B,128,576] bf16 (as uint16 bits), dev_kv [B*C,576] bf16 rows (the
 *   cache's rows, 1152 bytes each), both 16-byte aligned; sel_slot [B,k];
 *   out [B,128,512] f32 (16-byte aligned), lse [B,128] f32.
 *   k <= ECHO_MLA_MAX_K.  No workspace: the selection is cut into at most
 *   ECHO_MLA_MAX_SPLITS splits (one thread-block cluster per request and
 *   output half) that combine on chip.
 *   A device-side wait that gives up sets ECHO_ST_TIMEOUT in *status.
 *   Errors: ECHO_EINVAL (sizes, NULL or misaligned pointers),
 *   ECHO_EUNSUPPORTED (B > ECHO_MAX_REQUESTS or k > ECHO_MLA_MAX_K),
 *   ECHO_ECUDA (launch).
 * Scores are fp32 sums of bf16 products (tensor cores); the softmax weights
 * enter the value sum rounded to bf16.
 */
#define ECHO_MLA_HEADS 128
#define ECHO_MLA_DQK 576
#define ECHO_MLA_DV 512
#define ECHO_MLA_MAX_SPLITS 8
#define ECHO_MLA_MAX_K 8192
int echo_mla_decode(int B, int k, const uint16_t* q, const int32_t* sel_slot, const void* dev_kv, int64_t C,
                    float scale, float* out, float* lse, int32_t* status, echo_stream_t stream);

/*
 * Cross-layer early set [page "ECHO Guide: KV Offloading for Native Sparse Attention",
 * section "Intra-Query Prefetching: Layer-to-Layer Pipeline": layers l+1 and
 * l+2 select mostly what layer l selected; reading: layer l+1's early set is
 * layer l's selection minus layer l+1's residents].  Writes, for this layer's
 * cache, the two inputs of its early set: `above` (echo_above_words(B,
 * n_tokens) words, the layout echo_index_scores writes; bit set = selected by
 * prev_sel [B,m] (-1 padded, request-local) and not resident) and
 * cache->free_snap (this layer's free bits now).  Then call echo_early_fetch
 * with the same `above` at once (it streams the rows while this layer has not
 * scored yet), echo_index_scores of this layer with above = NULL and cache =
 * NULL (no threshold bits, no new snapshot), and this layer's top-k / cache
 * step with the same `above`.  The tables must not change between this call
 * and this layer's cache step.  Errors as echo_early_fetch.
 */
int echo_seed_early(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, const int32_t* prev_sel,
                    int m, uint32_t* above, const echo_cache* cache, int32_t* status, echo_stream_t stream);

/*
 * Shared per-worker pool [AE "Baselines under evaluation" and the decode
 * server's NSA_DEV_CACHE_SIZE: one device pool of slots per layer for the
 * worker's requests].  The pool is an echo_cache of one request spanning all
 * n_tokens rows (tok_off = {0, n_tokens}, token ids global, C = pool slots);
 * the early fetch, cache step and recall run on it unchanged.  Reading: the
 * requests' early sets and misses take the pool's lowest free slots in
 * (request, token) order.  A step: echo_index_scores per request with
 * `above_req` and cache = NULL; echo_pool_above; echo_early_fetch(1,
 * {0, n_tokens}, ..., above_pool, cap, pool); echo_topk_select per request;
 * echo_pool_select; echo_cache_step(1, {0, n_tokens}, ..., sel_pool, B*k,
 * above_pool, cap, pool, slot_pool, ...); echo_pool_slots.
 *   echo_pool_above: above_pool [echo_above_words(1, n_tokens)] = the marks of
 *     above_req [echo_above_words(B, n_tokens)] at global positions, tokens
 *     resident in the pool left out; pool->free_snap = pool->freebits.
 *   echo_pool_select: sel [B,k] (request-local, ascending, -1 padded) ->
 *     sel_pool [B*k] (global ids tok_off[b] + sel, ascending, -1 padding last).
 *   echo_pool_slots: slot_pool [B*k] (the pool step's sel_slot of sel_pool) ->
 *     sel_slot [B,k] aligned with sel.
 * Errors: ECHO_EINVAL (sizes, NULL pointers), ECHO_EUNSUPPORTED, cache errors.
 */
int echo_pool_above(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, const uint32_t* above_req,
                    const echo_cache* pool, uint32_t* above_pool, int32_t* status, echo_stream_t stream);
int echo_pool_select(int B, const int64_t* tok_off, const int32_t* sel, int k, int32_t* sel_pool, echo_stream_t stream);
int echo_pool_slots(int B, const int32_t* sel, int k, const int32_t* slot_pool, int32_t* sel_slot,
                    echo_stream_t stream);

/*
 * Append one new token to each request: the offload write path [EXPL section
 * 2, "One layer, one step": the host holds every token, hence no write-back
 * on eviction; the pages give no append mechanics -- reading below].
 * For request b with pos = tok_end[b]:
 *   pos == tok_off[b+1] (region full): nothing is written, ECHO_ST_FULL;
 *   ks[pos] = amax / 448 (fp32), amax = max_d |k_new[b,d]|;
 *   k8[pos,d] = E4M3 round-to-nearest-even, saturating, of k_new[b,d] / ks[pos]
 *               (fp32 quotient); amax = 0 gives ks = 0 and zero codes;
 *   host pool row pos = kv_new[b] (row_bytes, through cache->host_kv);
 *   the request's lowest free slot s, if any, takes the token: freebits bit
 *   cleared, tok2slot[pos] = s, slot2tok[b*C+s] = pos - tok_off[b], device
 *   row b*C+s = kv_new[b]; with no free slot the token is host-only;
 *   tok_end[b] = pos + 1.
 * A non-finite key component sets ECHO_ST_NAN and leaves that request as it
 * was.  Args: tok_off [B+1] / tok_end [B] int64 device (tok_end updated),
 * k_new [B,128] f32 device, kv_new [B,row_bytes] device (16-byte aligned),
 * k8 [n_tokens,128] u8 and ks [n_tokens] f32 device, cache as above.
 * Enqueue between steps, on the step's stream (every call of the next step
 * must see the new tok_end).  Errors: ECHO_EINVAL (sizes, NULL or misaligned
 * pointers), ECHO_EUNSUPPORTED, cache errors as echo_cache_step.
 */
int echo_append_tokens(int B, const int64_t* tok_off, int64_t* tok_end, int64_t n_tokens, const float* k_new,
                       const void* kv_new, uint8_t* k8, float* ks, const echo_cache* cache, int32_t* status,
                       echo_stream_t stream);

/* Device-accessible address of a pinned host buffer (for echo_cache.host_kv).
 * Returns ECHO_ECUDA when the pointer is not pinned/mapped host memory. */
int echo_host_device_alias(const void* host_ptr, const void** device_ptr);

/* Number of SMs of the current device (for sizing); negative on error. */
int echo_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* ECHO_H */
