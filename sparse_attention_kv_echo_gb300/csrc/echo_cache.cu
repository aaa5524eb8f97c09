// echo_cache.cu -- the per-layer GPU cache step, early fetch and recall.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2:
//   panel "Five fixed-size integer tensors on the GPU": nothing changes
//     length, so a decode step stays inside one CUDA graph;
//   panel "One layer, one step: free -> allocate -> recall": unselected slots
//     are freed (no write-back: the host holds every token), misses get
//     slots, their rows are recalled from the host pool;
//
// Kernels (one CTA of 1024 threads per request for the table work; the early
// selection runs at the end of the score kernel, echo_scores.cu):
//   cache_step_kernel    marks the slots of selected residents in a shared
//                        bitmap, frees the rest one warp per 32-slot word
//                        (ballot -> free-bit word), then a prefix sum of
//                        popcounts over the free-bit words hands the misses,
//                        in ascending order, the lowest free slots: each
//                        thread owns 4 consecutive selection entries, so its
//                        misses take consecutive free slots (one binary search,
//                        then a walk over the free bits).  Independent loads go
//                        out together at the start: two rounds of global
//                        latency for a 2048-entry selection and 4096 slots.
//   recall_kernel        one warp per row (two in flight), 16-byte loads from
//                        the pinned host pool through its device alias
//                        (zero-copy over the host link), 16-byte stores into
//                        the device cache; the rows of all requests form one
//                        list spread over a few large blocks.
#include "echo_common.cuh"
#include "echo_internal.h"
#include "echo_slots.cuh"
#include "echo_cachestep.cuh"

namespace echo {
namespace {

constexpr int kCT = 1024;  // threads of the walking cache step
constexpr int kLT = 1024;  // threads of the look-up cache step (at ~64 registers a block fills an SM's
                           // register file: no copy block, whose loads wait on the host link, shares it)


__device__ __forceinline__ bool request_range(const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, int b,
                                              int64_t* base, int64_t* n) {
    int64_t lo, hi;
    const bool ok = seg_bounds(tok_off, tok_end, n_tokens, b, &lo, &hi);
    *base = lo;
    *n = hi - lo;
    return ok;
}

constexpr int kPer = 4;        // selection entries per thread per chunk
// Above-threshold words per thread per chunk: the early set's ranks do not
// depend on it, so each kernel picks what keeps its threads' walks short
// (1024 words = 32768 tokens per request: one word per thread of the cache
// step, two per thread of the early fetch).
constexpr int kEarlyWordsStep = 1;
constexpr int kEarlyWordsFetch = 2;

constexpr int kES = 4096;  // early (token, slot) pairs kept in shared memory for the table phases

// Shared memory of the cache-step kernel, in 32-bit words.
__host__ __device__ constexpr size_t cache_step_smem_words(int C) {
    return 3 * static_cast<size_t>(C / 32) + 1 + 2 * static_cast<size_t>(kES);
}

// Binary search of v in the ascending a[0, n); -1 when absent.
__device__ __forceinline__ int find_sorted(const int32_t* a, int n, int32_t v) {
    int lo = 0, hi = n - 1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        const int32_t x = a[mid];
        if (x == v) return mid;
        if (x < v)
            lo = mid + 1;
        else
            hi = mid - 1;
    }
    return -1;
}

// ---------------------------------------------------------------- cache step, look-up form
// (echo_cachestep.cuh): the early set is found by rank look-ups, not walked.
// Used when C <= kLookupMaxSlots.
constexpr int kAWC = 8192;                 // above words per chunk held in shared memory
constexpr int kLookupMaxSlots = 1 << 17;   // 4 x 4096 words + the chunk fit shared memory

template <bool kResolved>
__global__ void __launch_bounds__(kLT)
    cache_step_lookup_kernel(const int64_t* __restrict__ tok_off, const int64_t* __restrict__ tok_end, int64_t n_tokens, const int32_t* __restrict__ sel,
                             int m, const uint32_t* __restrict__ above, int early_cap, CacheArgs c,
                             int32_t* sel_slot, int32_t* status, uint32_t* stats, bool hold_early) {
    pdl_launch_dependents();  // the late recall's blocks may be scheduled now; they wait for this kernel
    extern __shared__ uint32_t smem[];
    __shared__ uint32_t scan[40];
    __shared__ uint32_t flags[2];
    CacheStepLookup<kLT, kAWC, kResolved> cs;
    cs.init(tok_off, tok_end, n_tokens, blockIdx.x, sel, m, sel_slot, above, early_cap, c, status, stats, smem, scan, flags,
            hold_early);
    cs.prologue_issue();  // the tables only: they may be read before the kernel before this one ends
    cs.prologue_finish();
    pdl_wait();           // the selection and the above words come from the kernels before this one
    cs.load_selection();
    cs.load_above();
    cs.load_slots();
    cs.above_finish();    // while the slot loads are in flight
    cs.finish();
}

__global__ void __launch_bounds__(kCT) cache_step_kernel(const int64_t* __restrict__ tok_off,
                                                         const int64_t* __restrict__ tok_end, int64_t n_tokens,
                                                         const int32_t* __restrict__ sel, int m,
                                                         const uint32_t* __restrict__ above, int early_cap,
                                                         CacheArgs c, int32_t* __restrict__ sel_slot, int32_t* status,
                                                         uint32_t* stats, bool hold_early, bool lazy) {
    // keep [words]: a selected token lives in the slot | wpre [words + 1] | fbs [words] (free bits)
    // | es_tok [kES] | es_slot [kES] (the early pairs, both ascending)
    extern __shared__ uint32_t keep[];
    __shared__ uint32_t scan[40];
    __shared__ uint32_t s_flags, s_early_used, s_revived;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_launch_dependents();  // the late recall's blocks may be scheduled now; they wait for this kernel
    pdl_wait();  // launched as a programmatic dependent: everything below may depend on the kernel before
    int64_t base, n;
    if (!request_range(tok_off, tok_end, n_tokens, b, &base, &n) && tid == 0) set_status(status, ECHO_ST_BADDATA);
    const int C = c.C, words = C / 32;
    int32_t* t2s = c.tok2slot + base;
    int32_t* s2t = c.slot2tok + static_cast<int64_t>(b) * C;
    uint32_t* fb = c.freebits + static_cast<int64_t>(b) * words;
    const int32_t* sl = sel + static_cast<int64_t>(b) * m;
    int32_t* out = sel_slot + static_cast<int64_t>(b) * m;
    int32_t* mtok = c.miss_tok + static_cast<int64_t>(b) * C;
    int32_t* mslot = c.miss_slot + static_cast<int64_t>(b) * C;
    int32_t* etok = c.early_tok + static_cast<int64_t>(b) * C;
    int32_t* eslot = c.early_slot + static_cast<int64_t>(b) * C;
    uint32_t* wpre = keep + words;
    uint32_t* fbs = wpre + words + 1;
    int32_t* es_tok = reinterpret_cast<int32_t*>(fbs + words);
    int32_t* es_slot = es_tok + kES;
    constexpr int kChunk = kCT * kPer;
    const int chunks = (m + kChunk - 1) / kChunk;
    const bool early = above != nullptr && early_cap != 0 && n > 0;

    // Global latency is what this kernel costs (it runs while the early rows
    // stream over the host link), so the loads go out in two rounds and every
    // later phase works from registers and shared memory.  Round 1: this
    // thread's selection entries (kPer consecutive ones, so its misses have
    // consecutive ranks) and the one after them, the slot owners and free-bit
    // words, the first above-threshold words.
    int32_t s[kPer], j[kPer];
    auto load_sel = [&](int c0) {
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = c0 + kPer * tid + q;
            s[q] = (i < m) ? sl[i] : -1;
        }
    };
    load_sel(0);
    int32_t after0 = (kPer * tid + kPer < m) ? sl[kPer * tid + kPer] : -1;
    constexpr int kPre = 4;  // 32-slot words per warp held in registers
    const bool pre = words <= kPre * (kCT / 32);
    int32_t own[kPre];
#pragma unroll
    for (int r = 0; r < kPre; ++r) {
        const int w = warp + r * (kCT / 32);
        own[r] = (pre && w < words) ? s2t[w * 32 + lane] : -1;
    }
    const uint32_t* ab = early ? above + 4 * (base / 128 + b) : nullptr;
    const int nw = static_cast<int>((n + 31) >> 5);
    const uint32_t tail_mask = (n & 31) ? (1u << (n & 31)) - 1u : ~0u;
    uint32_t v[kEarlyWordsStep];
    if (early) early_words<kEarlyWordsStep>(ab, nw, tail_mask, kEarlyWordsStep * tid, v);
    for (int w = tid; w < words; w += kCT) {
        fbs[w] = fb[w];
        keep[w] = 0u;
    }
    if (tid == 0) {
        s_flags = 0;
        s_early_used = 0;
        s_revived = 0;
    }
    // Round 2: the slots of the selected tokens as the step found them.
    if (chunks == 1) {
#pragma unroll
        for (int q = 0; q < kPer; ++q) j[q] = (s[q] >= 0 && s[q] < n) ? t2s[s[q]] : -1;
    }
    __syncthreads();

    // 0. the early set (the tokens echo_early_fetch copied) and its slots; the
    // slots leave the free bits, the tables learn only the selected early tokens
    // (1a), and the slots of the others are held until the misses are placed
    // (their early copies may still be in flight) and free again after the step
    uint32_t E = 0;
    if (early) {
        const uint32_t F = free_prefix<kCT>(fbs, words, scan, wpre, fbs);
        const uint32_t limit = (early_cap < 0) ? F : min(F, static_cast<uint32_t>(early_cap));
        const uint32_t found = early_assign<kCT, kEarlyWordsStep>(
            ab, nw, tail_mask, limit, 0u, limit, wpre, fbs, words, scan, v, [&](uint32_t r, int tok, int slot) {
                if (slot < 0) {
                    set_status(status, ECHO_ST_BADDATA);
                    return;
                }
                etok[r] = tok;
                eslot[r] = slot;
                if (r < static_cast<uint32_t>(kES)) {
                    es_tok[r] = tok;
                    es_slot[r] = slot;
                }
            });
        E = min(found, limit);
        __syncthreads();  // every walk over fbs is done before its bits change
        take_lowest_free<kCT>(fbs, words, E, wpre);
        __syncthreads();
    }
    // the early pairs are looked up in shared memory when they all fit, else in
    // the early lists just written (this block's own writes)
    const bool es_ok = E <= static_cast<uint32_t>(kES);
    const int32_t* e_tok = es_ok ? es_tok : etok;
    const int32_t* e_slot = es_ok ? es_slot : eslot;
    uint32_t used = 0;
    if (lazy) {
        // lazy reuse: every early token enters the tables in its slot, and the ghost
        // (a token freed earlier whose bytes and entries the slot kept) leaves them
        for (uint32_t e = tid; e < E; e += kCT) {
            const int32_t tok = e_tok[e], slot = e_slot[e];
            if (tok < 0 || tok >= n || slot < 0 || slot >= C) continue;
            const int32_t g = s2t[slot];
            if (g >= 0 && g < n) t2s[g] = -1;
            t2s[tok] = slot;
            s2t[slot] = tok;
        }
        __syncthreads();
    }

    // 1a. slots that hold a selected token are kept; the selection must be
    // ascending with -1 padding last
    for (int ch = 0; ch < chunks; ++ch) {
        const int c0 = ch * kChunk;
        int32_t after = after0;
        if (chunks > 1) {
            load_sel(c0);
            const int inext = c0 + kPer * tid + kPer;
            after = (inext < m) ? sl[inext] : -1;
        }
        uint32_t flags = 0;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int32_t nxt = (q + 1 < kPer) ? s[q + 1] : after;
            if (s[q] >= 0 && s[q] < n) {
                if (nxt >= 0 && nxt <= s[q]) flags |= ECHO_ST_BADDATA;
                if (chunks > 1 || lazy) j[q] = t2s[s[q]];
                if (lazy) {
                    if (j[q] >= 0 && E > 0 && find_sorted(e_tok, static_cast<int>(E), s[q]) >= 0) ++used;
                } else if (j[q] < 0 && E > 0) {  // a selected early token becomes resident in its slot
                    const int e = find_sorted(e_tok, static_cast<int>(E), s[q]);
                    if (e >= 0) {
                        j[q] = e_slot[e];
                        t2s[s[q]] = j[q];
                        s2t[j[q]] = s[q];
                        ++used;
                    }
                }
            } else {
                j[q] = -1;
                if (s[q] >= 0 || nxt >= 0) flags |= ECHO_ST_BADDATA;
            }
        }
        if (flags) atomicOr(&s_flags, flags);
#pragma unroll
        for (int q = 0; q < kPer; ++q)
            if (j[q] >= 0 && j[q] < C) atomicOr(&keep[j[q] >> 5], 1u << (j[q] & 31));
    }
    __syncthreads();

    // 1b. every other occupied slot is freed (bytes stay, nothing is written
    // back), one warp per 32-slot word; the new free-bit words stay in shared memory
    auto free_word = [&](int w, int32_t st) {
        const int slot = w * 32 + lane;
        const bool kept = (keep[w] >> lane) & 1u;
        const bool freeing = st >= 0 && !kept;
        if (freeing && !lazy) {  // lazy reuse: the token stays in the tables as a ghost
            s2t[slot] = -1;
            if (st < n) t2s[st] = -1;
        }
        const unsigned fm = __ballot_sync(0xffffffffu, freeing);
        if (lane == 0) fbs[w] |= fm;
    };
    // (the owners read at the start: early slots were free then, so none of them is freed here)
    if (pre) {
#pragma unroll
        for (int r = 0; r < kPre; ++r) {
            const int w = warp + r * (kCT / 32);
            if (w < words) free_word(w, own[r]);
        }
    } else {
        // C beyond the registers: only the slots that held a resident token at the start (free bit
        // clear in freebits, which this kernel writes at its end only) and are not kept are read,
        // their owners' loads issued together; lazy reuse keeps the entries and reads nothing
        for (int w = tid; w < words; w += kCT) {
            uint32_t occ = ~__ldcg(fb + w) & ~keep[w];
            if (!occ) continue;
            fbs[w] |= occ;
            while (occ && !lazy) {
                int32_t ps[8], po[8];
                int cnt = 0;
                while (occ && cnt < 8) {
                    ps[cnt++] = w * 32 + (__ffs(occ) - 1);
                    occ &= occ - 1;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < cnt) po[i] = s2t[ps[i]];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < cnt) {
                        s2t[ps[i]] = -1;
                        if (po[i] >= 0 && po[i] < n) t2s[po[i]] = -1;
                    }
            }
        }
    }
    if (used) atomicAdd(&s_early_used, used);
    __syncthreads();
    if (lazy) {  // a selected ghost is resident again in its slot: the slot is not free
        uint32_t rev = 0;
        for (int w = tid; w < words; w += kCT) {
            rev += __popc(fbs[w] & keep[w]);
            fbs[w] &= ~keep[w];
        }
        if (rev) atomicAdd(&s_revived, rev);
        __syncthreads();
    }
    if (!hold_early) {  // the unselected early tokens' slots are free for the misses
        for (uint32_t e = tid; e < E; e += kCT) {
            const int32_t es = e_slot[e];
            if (es >= 0 && es < C && !((keep[es >> 5] >> (es & 31)) & 1u)) atomicOr(&fbs[es >> 5], 1u << (es & 31));
        }
        __syncthreads();
    }

    // 2. free-slot prefix over the new free-bit words
    const uint32_t F = free_prefix<kCT>(fbs, words, scan, wpre, fbs);

    // 3. the misses, in ascending token order, take the lowest free slots; the
    // slot of every selected entry is written on the way
    uint32_t found = 0;
    for (int ch = 0; ch < chunks; ++ch) {
        const int c0 = ch * kChunk;
        if (chunks > 1) {  // the registers hold the last chunk only: reload
            load_sel(c0);
#pragma unroll
            for (int q = 0; q < kPer; ++q) j[q] = (s[q] >= 0 && s[q] < n) ? t2s[s[q]] : -1;
        }
        uint32_t missing = 0;
#pragma unroll
        for (int q = 0; q < kPer; ++q)
            if (s[q] >= 0 && s[q] < n && j[q] < 0) missing |= 1u << q;
        uint32_t tot;
        uint32_t rank = found + block_exclusive_scan<kCT>(__popc(missing), scan, &tot);
        FreeWalk walk(wpre, fbs, words, rank < F ? rank : 0u);
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = c0 + kPer * tid + q;
            if (i >= m) break;
            int32_t slot = j[q];
            if (missing & (1u << q)) {
                slot = (rank < F) ? walk.next() : -1;
                if (slot >= 0) {
                    if (rank < static_cast<uint32_t>(C)) {
                        mtok[rank] = s[q];
                        mslot[rank] = slot;
                    }
                    if (lazy) {  // the ghost in the slot leaves the tables
                        const int32_t g = s2t[slot];
                        if (g >= 0 && g < n) t2s[g] = -1;
                    }
                    t2s[s[q]] = slot;
                    s2t[slot] = s[q];
                }
                ++rank;
            } else if (s[q] < 0 || s[q] >= n) {
                slot = -1;
            }
            out[i] = slot;
        }
        found += tot;
    }
    const uint32_t got = min(found, F);
    __syncthreads();  // every walk over fbs is done before its bits change
    take_lowest_free<kCT>(fbs, words, got, wpre);
    __syncthreads();
    // the held early slots (not kept by a selected token) are free again
    for (uint32_t e = tid; e < (hold_early ? E : 0u); e += kCT) {
        const int32_t es = e_slot[e];
        if (es >= 0 && es < C && !((keep[es >> 5] >> (es & 31)) & 1u)) atomicOr(&fbs[es >> 5], 1u << (es & 31));
    }
    __syncthreads();
    for (int w = tid; w < words; w += kCT) fb[w] = fbs[w];
    if (tid == 0) {
        c.miss_cnt[b] = static_cast<int32_t>(got);
        c.early_cnt[b] = static_cast<int32_t>(E);
        if (stats && got) atomicAdd(stats + ECHO_STAT_MISSES, got);
        if (stats && E) atomicAdd(stats + ECHO_STAT_EARLY, E);
        if (stats && s_early_used) atomicAdd(stats + ECHO_STAT_EARLY_USED, s_early_used);
        if (stats && s_revived) atomicAdd(stats + ECHO_STAT_REVIVED, s_revived);
        uint32_t flags = s_flags;
        if (found > F) flags |= ECHO_ST_NOSLOT;
        if (flags) set_status(status, static_cast<int>(flags));
    }
}

constexpr int kRecallThreads = 512;
constexpr int kRecallBlocks = 24;
constexpr int kRows = 2;        // rows per warp in flight (4 measured: the host reads queue up and every
                                // kernel of the step slowed about tenfold)
constexpr int kStage = 4096;    // early (token, slot) pairs staged in shared memory per round

// One warp copies kRows rows (those with ok[r]) of `chunks` 16-byte pieces.
__device__ __forceinline__ void copy_rows(const int4* const (&src)[kRows], int4* const (&dst)[kRows],
                                          const bool (&ok)[kRows], int chunks, int lane) {
    for (int c0 = 0; c0 < chunks; c0 += 96) {
        int4 v[kRows][3];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int c = c0 + lane + 32 * j;
                v[r][j] = (ok[r] && c < chunks) ? __ldcs(src[r] + c) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int c = c0 + lane + 32 * j;
                if (ok[r] && c < chunks) dst[r][c] = v[r][j];
            }
    }
}

// Rows of all requests form one list (request b's rows at pre[b] .. pre[b+1]);
// warp w of the grid copies rows w*2, w*2+1, then strides by the grid's warps.
__global__ void __launch_bounds__(kRecallThreads)
    recall_kernel(int B, const int64_t* __restrict__ tok_off, const int64_t* __restrict__ tok_end, int64_t n_tokens,
                  int C,
                  const int32_t* __restrict__ tok_list, const int32_t* __restrict__ slot_list,
                  const int32_t* __restrict__ cnt, const uint8_t* host, uint8_t* __restrict__ dev, int64_t row_bytes,
                  int32_t* status) {
    extern __shared__ int32_t pre[];  // [B + 1]
    __shared__ uint32_t scan[kRecallThreads / 32 + 1];
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    pdl_wait();  // the lists and counts come from the cache step (when launched as its dependent)
    uint32_t run = 0;
    for (int b0 = 0; b0 < B; b0 += kRecallThreads) {
        const int b = b0 + static_cast<int>(threadIdx.x);
        const uint32_t v = (b < B) ? static_cast<uint32_t>(min(max(cnt[b], 0), C)) : 0u;
        uint32_t tot;
        const uint32_t ex = block_exclusive_scan<kRecallThreads>(v, scan, &tot);
        if (b < B) pre[b] = static_cast<int32_t>(run + ex);
        run += tot;
    }
    if (threadIdx.x == 0) pre[B] = static_cast<int32_t>(run);
    __syncthreads();
    const int total = static_cast<int>(run);
    const int chunks = static_cast<int>(row_bytes / 16);
    for (int i0 = (blockIdx.x * warps + (threadIdx.x >> 5)) * kRows; i0 < total;
         i0 += gridDim.x * warps * kRows) {
        const int4* src[kRows];
        int4* dst[kRows];
        bool ok[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int i = i0 + r;
            ok[r] = false;
            src[r] = nullptr;
            dst[r] = nullptr;
            if (i < total) {
                int lo = 0, hi = B - 1;  // request of row i: largest b with pre[b] <= i
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (pre[mid] <= i)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                const int b = lo;
                int64_t base, n;
                const bool range_ok = request_range(tok_off, tok_end, n_tokens, b, &base, &n);
                const int64_t e = static_cast<int64_t>(b) * C + (i - pre[b]);
                const int32_t tok = tok_list[e];
                const int32_t slot = slot_list[e];
                if (range_ok && tok >= 0 && tok < n && slot >= 0 && slot < C) {
                    ok[r] = true;
                    src[r] = reinterpret_cast<const int4*>(host + (base + tok) * row_bytes);
                    dst[r] = reinterpret_cast<int4*>(dev + (static_cast<int64_t>(b) * C + slot) * row_bytes);
                } else if (lane == 0) {
                    set_status(status, ECHO_ST_BADDATA);
                }
            }
        }
        copy_rows(src, dst, ok, chunks, lane);
    }
}

// The early fetch: G = gridDim.x / B blocks per request (at least one; blocks
// beyond a multiple of G idle).  Every block of a request computes the early
// set from the above-threshold words and the free-bit snapshot (the tables
// are not touched), stages (token, slot) pairs in shared memory, and copies
// the staged rows whose index is g (mod G), g its place in the request's group.
__global__ void __launch_bounds__(kRecallThreads)
    early_fetch_kernel(int B, const int64_t* __restrict__ tok_off, const int64_t* __restrict__ tok_end, int64_t n_tokens,
                       const uint32_t* __restrict__ above, int cap, const uint32_t* __restrict__ snap, int C,
                       int32_t* __restrict__ early_tok, int32_t* __restrict__ early_slot, const uint8_t* host,
                       uint8_t* __restrict__ dev, int64_t row_bytes, int32_t* status) {
    extern __shared__ uint32_t esm[];  // wpre [words + 1], fbs [words], stage tokens, stage slots
    __shared__ uint32_t scan[kRecallThreads / 32 + 1];
    const int words = C / 32;
    uint32_t* wpre = esm;
    uint32_t* fbs = wpre + words + 1;
    int32_t* stok = reinterpret_cast<int32_t*>(fbs + words);
    int32_t* sslot = stok + kStage;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = kRecallThreads / 32;
    const int G = max(1, static_cast<int>(gridDim.x) / B);
    const int groups = static_cast<int>(gridDim.x) / G;
    const int g = static_cast<int>(blockIdx.x) % G;
    const int chunks = static_cast<int>(row_bytes / 16);
    // the request's rows come from the caller, not the score kernel: read them
    // before waiting for it
    int b = static_cast<int>(blockIdx.x) / G;
    int64_t base = 0, n = 0;
    bool range_ok = b < B && request_range(tok_off, tok_end, n_tokens, b, &base, &n);
    pdl_wait();  // the above-threshold words and the snapshot come from the score kernel
    for (; b < B && static_cast<int>(blockIdx.x) < groups * G; b += groups) {
        if (b != static_cast<int>(blockIdx.x) / G) range_ok = request_range(tok_off, tok_end, n_tokens, b, &base, &n);
        if (!range_ok) {
            if (threadIdx.x == 0) set_status(status, ECHO_ST_BADDATA);
            continue;
        }
        if (n == 0 || cap == 0) continue;
        const uint32_t* ab = above + 4 * (base / 128 + b);
        const int nw = static_cast<int>((n + 31) >> 5);
        const uint32_t tail_mask = (n & 31) ? (1u << (n & 31)) - 1u : ~0u;
        uint32_t v[kEarlyWordsFetch];
        early_words<kEarlyWordsFetch>(ab, nw, tail_mask, kEarlyWordsFetch * threadIdx.x, v);
        const uint32_t F = free_prefix<kRecallThreads>(snap + static_cast<int64_t>(b) * words, words, scan, wpre, fbs);
        const uint32_t limit = (cap < 0) ? F : min(F, static_cast<uint32_t>(cap));
        for (uint32_t r_lo = 0; r_lo < limit; r_lo += kStage) {
            if (r_lo > 0) early_words<kEarlyWordsFetch>(ab, nw, tail_mask, kEarlyWordsFetch * threadIdx.x, v);
            const uint32_t r_hi = min(limit, r_lo + kStage);
            const uint32_t found = early_assign<kRecallThreads, kEarlyWordsFetch>(
                ab, nw, tail_mask, limit, r_lo, r_hi, wpre, fbs, words, scan, v, [&](uint32_t r, int tok, int slot) {
                    stok[r - r_lo] = tok;
                    sslot[r - r_lo] = slot;
                });
            const uint32_t E = min(found, limit);
            __syncthreads();
            const int staged = static_cast<int>(min(E, r_hi) - min(E, r_lo));
            if (g == 0) {  // the first block of the request's group writes the early lists
                int32_t* et = early_tok + static_cast<int64_t>(b) * C + r_lo;
                int32_t* es = early_slot + static_cast<int64_t>(b) * C + r_lo;
                for (int i = static_cast<int>(threadIdx.x); i < staged; i += kRecallThreads) {
                    et[i] = stok[i];
                    es[i] = sslot[i];
                }
            }
            const int share = staged > g ? (staged - g + G - 1) / G : 0;
            for (int k0 = warp * kRows; k0 < share; k0 += kWarps * kRows) {
                const int4* src[kRows];
                int4* dst[kRows];
                bool ok[kRows];
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    const int k = k0 + r;
                    ok[r] = false;
                    src[r] = nullptr;
                    dst[r] = nullptr;
                    if (k < share) {
                        const int i = g + G * k;
                        const int32_t tok = stok[i], slot = sslot[i];
                        if (tok >= 0 && tok < n && slot >= 0 && slot < C) {
                            ok[r] = true;
                            src[r] = reinterpret_cast<const int4*>(host + (base + tok) * row_bytes);
                            dst[r] = reinterpret_cast<int4*>(dev + (static_cast<int64_t>(b) * C + slot) * row_bytes);
                        } else if (lane == 0) {
                            set_status(status, ECHO_ST_BADDATA);
                        }
                    }
                }
                copy_rows(src, dst, ok, chunks, lane);
            }
            __syncthreads();  // the stage is reused by the next round / request
            if (found < r_hi) break;  // every marked token was counted
        }
    }
}

// Cross-layer seed of the early set: one block per request marks, in the
// above-threshold word layout the score kernel writes (the request's words
// from 4 * (floor(first row / 128) + b); bit j of word w = request-local token
// 32 w + j), the tokens the previous layer selected that are not resident in
// this layer, and snapshots this layer's free bits -- the two inputs the early
// fetch, the cached top-k and the cache step read.
constexpr int kSeedThreads = 256;
__global__ void __launch_bounds__(kSeedThreads)
    seed_kernel(const int64_t* __restrict__ tok_off, const int64_t* __restrict__ tok_end, int64_t n_tokens,
                const int32_t* __restrict__ prev_sel, int m, uint32_t* __restrict__ above,
                const int32_t* __restrict__ tok2slot, const uint32_t* __restrict__ freebits,
                uint32_t* __restrict__ free_snap, int C, int32_t* status) {
    const int b = blockIdx.x, tid = threadIdx.x;
    int64_t base, n;
    if (!request_range(tok_off, tok_end, n_tokens, b, &base, &n) && tid == 0) set_status(status, ECHO_ST_BADDATA);
    uint32_t* ab = above + 4 * (base / 128 + b);
    const int nw = static_cast<int>((n + 31) >> 5);
    for (int w = tid; w < nw; w += kSeedThreads) ab[w] = 0u;
    const int words = C / 32;
    for (int w = tid; w < words; w += kSeedThreads)
        free_snap[static_cast<int64_t>(b) * words + w] = freebits[static_cast<int64_t>(b) * words + w];
    __syncthreads();
    const int32_t* ps = prev_sel + static_cast<int64_t>(b) * m;
    for (int i = tid; i < m; i += kSeedThreads) {
        const int32_t t = ps[i];
        if (t >= 0 && t < n && tok2slot[base + t] < 0) atomicOr(ab + (t >> 5), 1u << (t & 31));
    }
}

}  // namespace

cudaError_t launch_recall(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, int C, const int32_t* tok_list,
                          const int32_t* slot_list, const int32_t* cnt, const void* host_kv, void* dev_kv,
                          int64_t row_bytes, int32_t* status, cudaStream_t s, bool programmatic) {
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    // A few large blocks: the host link, not the SMs, bounds the copy (24 x 16
    // warps x 2 rows keep ~0.9 MB of host reads in flight).  Loads that wait on
    // the host link slow every other kernel that shares an SM with them, so the
    // copy stays on few SMs, and a block this size (512 threads x ~50 registers)
    // cannot share an SM with a 1024-thread top-k CTA, which then runs elsewhere.
    int blocks = kRecallBlocks < sms / 2 ? kRecallBlocks : sms / 2;
    if (blocks < 1) blocks = 1;
    const size_t smem = (static_cast<size_t>(B) + 1) * sizeof(int32_t);
    cudaError_t e = prefer_max_shared(recall_kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(recall_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // programmatic: the blocks may be scheduled while the kernel before them on
    // `s` runs (the cache step lets them at its start); they wait for it first
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kRecallThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, recall_kernel, B, tok_off, tok_end, n_tokens, C, tok_list, slot_list, cnt,
                              static_cast<const uint8_t*>(host_kv), static_cast<uint8_t*>(dev_kv), row_bytes,
                              status);
}

}  // namespace echo

namespace echo {

int enqueue_cache_step(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, const int32_t* sel,
                       int m,
                       const uint32_t* above, int early_cap, const echo_cache* cache, int32_t* sel_slot,
                       int32_t* status, uint32_t* stats, cudaStream_t stream, cudaStream_t copy_stream,
                       bool resolved, bool hold_early, bool lazy) {
    // lazy reuse walks the early set (every early token enters the tables)
    const bool lookup = cache->C <= kLookupMaxSlots && !lazy;
    if (lazy && (resolved || hold_early)) return ECHO_EUNSUPPORTED;
    if (resolved && !lookup) return ECHO_EUNSUPPORTED;
    const size_t smem =
        (lookup ? cache_lookup_smem_words(cache->C, kAWC) : cache_step_smem_words(cache->C)) * sizeof(uint32_t);
    auto lookup_kernel = resolved ? cache_step_lookup_kernel<true> : cache_step_lookup_kernel<false>;
    if (lookup) {
        ECHO_CUDA_OK(prefer_max_shared(lookup_kernel));
        ECHO_CUDA_OK(cudaFuncSetAttribute(lookup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(smem)));
    } else {
        ECHO_CUDA_OK(prefer_max_shared(cache_step_kernel));
        ECHO_CUDA_OK(cudaFuncSetAttribute(cache_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(smem)));
    }
    // Programmatic dependent launch: once the kernel before it on `stream`
    // lets dependents start (top-k does at its start), the look-up form reads
    // the cache's own tables and takes the free-slot prefix while that kernel
    // still runs; it waits (griddepcontrol.wait) before anything else.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(lookup ? kLT : kCT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const CacheArgs ca = cache_args(*cache);
    if (lookup) {
        ECHO_CUDA_OK(cudaLaunchKernelEx(&cfg, lookup_kernel, tok_off, tok_end, n_tokens, sel, m, resolved ? nullptr : above,
                                        early_cap, ca, sel_slot, status, stats, hold_early));
    } else {
        ECHO_CUDA_OK(cudaLaunchKernelEx(&cfg, cache_step_kernel, tok_off, tok_end, n_tokens, sel, m, above, early_cap, ca,
                                        sel_slot, status, stats, hold_early, lazy));
    }
    const int rc = stream_wait(copy_stream, stream);
    if (rc) return rc;
    ECHO_CUDA_OK(launch_recall(B, tok_off, tok_end, n_tokens, cache->C, cache->miss_tok, cache->miss_slot, cache->miss_cnt,
                               cache->host_kv, cache->dev_kv, cache->row_bytes, status, copy_stream,
                               copy_stream == stream));
    return ECHO_OK;
}

int check_cache_step_args(int B, int64_t n_tokens, const int32_t* sel, int m, const echo_cache* cache,
                          const int32_t* sel_slot) {
    if (B <= 0 || n_tokens < 0 || m < 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (m > 0 && (!sel || !sel_slot)) return ECHO_EINVAL;
    if (n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    const int rc = check_cache(cache, B, m);
    if (rc) return rc;
    if (cache->C > kMaxSlots) return ECHO_EUNSUPPORTED;
    return ECHO_OK;
}

}  // namespace echo

extern "C" int echo_cache_step(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                               const int32_t* sel, int m,
                               const uint32_t* above, int early_cap, const echo_cache* cache, int32_t* sel_slot,
                               int32_t* status, uint32_t* stats, echo_stream_t stream, echo_stream_t copy_stream,
                               int flags) {
    using namespace echo;
    if (!tok_off || !status || (flags & ~(ECHO_CACHE_HOLD_EARLY | ECHO_CACHE_LAZY))) return ECHO_EINVAL;
    if ((flags & ECHO_CACHE_HOLD_EARLY) && (flags & ECHO_CACHE_LAZY)) return ECHO_EINVAL;
    const int rc = check_cache_step_args(B, n_tokens, sel, m, cache, sel_slot);
    if (rc) return rc;
    return enqueue_cache_step(B, tok_off, tok_end, n_tokens, sel, m, above, early_cap, cache, sel_slot, status, stats, stream,
                              copy_stream, false, (flags & ECHO_CACHE_HOLD_EARLY) != 0, (flags & ECHO_CACHE_LAZY) != 0);
}

extern "C" int echo_cache_step_resolved(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                                        const int32_t* sel, int m,
                                        const echo_cache* cache, int32_t* sel_slot, int32_t* status, uint32_t* stats,
                                        echo_stream_t stream, echo_stream_t copy_stream, int flags) {
    using namespace echo;
    if (!tok_off || !status || (flags & ~ECHO_CACHE_HOLD_EARLY)) return ECHO_EINVAL;
    const int rc = check_cache_step_args(B, n_tokens, sel, m, cache, sel_slot);
    if (rc) return rc;
    if (cache->C > kLookupMaxSlots) return ECHO_EUNSUPPORTED;
    return enqueue_cache_step(B, tok_off, tok_end, n_tokens, sel, m, nullptr, 0, cache, sel_slot, status, stats, stream,
                              copy_stream, true, (flags & ECHO_CACHE_HOLD_EARLY) != 0, false);
}

extern "C" int echo_early_fetch(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                                const uint32_t* above,
                                int early_cap, const echo_cache* cache, int32_t* status, echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || n_tokens < 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !above || !status) return ECHO_EINVAL;
    if (n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    int rc = check_cache(cache, B, 0);
    if (rc) return rc;
    if (!cache->free_snap) return ECHO_EINVAL;
    if (cache->C > kMaxSlots) return ECHO_EUNSUPPORTED;
    if (n_tokens == 0 || early_cap == 0) return ECHO_OK;
    const int sms = sm_count();
    if (sms <= 0) return ECHO_ECUDA;
    int blocks = kRecallBlocks < sms / 2 ? kRecallBlocks : sms / 2;
    if (blocks < 1) blocks = 1;
    const size_t smem = (2 * static_cast<size_t>(cache->C / 32) + 1 + 2 * kStage) * sizeof(uint32_t);
    ECHO_CUDA_OK(prefer_max_shared(early_fetch_kernel));
    ECHO_CUDA_OK(cudaFuncSetAttribute(early_fetch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
    // Programmatic dependent launch: the blocks are scheduled as the score
    // kernel's CTAs retire and wait (griddepcontrol.wait) for its results.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kRecallThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ECHO_CUDA_OK(cudaLaunchKernelEx(&cfg, early_fetch_kernel, B, tok_off, tok_end, n_tokens, above, early_cap,
                                    static_cast<const uint32_t*>(cache->free_snap), static_cast<int>(cache->C),
                                    cache->early_tok, cache->early_slot,
                                    static_cast<const uint8_t*>(cache->host_kv), static_cast<uint8_t*>(cache->dev_kv),
                                    cache->row_bytes, status));
    return ECHO_OK;
}

extern "C" int echo_seed_early(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                               const int32_t* prev_sel, int m, uint32_t* above, const echo_cache* cache,
                               int32_t* status, echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || n_tokens < 0 || m < 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !prev_sel || !above || !status) return ECHO_EINVAL;
    const int rc = check_cache(cache, B, 0);
    if (rc) return rc;
    if (!cache->free_snap) return ECHO_EINVAL;
    if (n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    seed_kernel<<<B, kSeedThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        tok_off, tok_end, n_tokens, prev_sel, m, above, cache->tok2slot, cache->freebits, cache->free_snap, cache->C,
        status);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}
