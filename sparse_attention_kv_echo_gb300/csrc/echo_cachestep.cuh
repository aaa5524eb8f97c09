// echo_cachestep.cuh -- the GPU-cache step of one request, block-wide, in the
// look-up form.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2,
// panel "One layer, one step: free -> allocate -> recall": the early set
// (panel "Decode: fetch above a predicted threshold") is resident, unselected
// slots are freed, misses take the lowest free slots.
//
// The early fetch already copied the early set's rows and wrote its lists, so
// only the selected tokens among it matter here: a selected token s that is
// not resident is early iff its above-threshold bit is set and its rank r
// among the marked tokens (a prefix of popcounts over the above words) is
// below the early limit; its slot is then the r-th free slot of the step's
// starting free bits.  The early set is never walked: one scan over the above
// words, one over the free bits, O(1) work per selected token.
//
// Resolved form: top-k already looked up every selected token's slot
// (resident or early, -1 for a miss; echo_topk_select_cached) and the early
// set's size; the step reads those instead of the above words and the tables,
// and does the rest.
//
// Order of the parts: prologue_issue() and prologue_finish() read only the
// cache's own tables (slot owners, free bits: the free-slot prefix and the
// early limit), so a kernel may run them before it waits for the kernel that
// writes the selection; then load_selection() and load_above() (one round of
// loads), load_slots() (the selected tokens' slots, a second round),
// above_finish() (the rank prefix over the above words, while the slots are
// in flight) and finish().
#pragma once

#include "echo_common.cuh"
#include "echo_slots.cuh"

namespace echo {

constexpr int kCsPer = 4;   // selection entries per thread per chunk

// Shared memory in 32-bit words: keep [words] | wpre [words + 1] | fbs [words]
// | held [words] | aw [awc] | apre [awc + 1].
__host__ __device__ constexpr size_t cache_lookup_smem_words(int C, int awc) {
    return 4 * static_cast<size_t>(C / 32) + 1 + 2 * static_cast<size_t>(awc) + 1;
}

template <int NT, int AWC, bool kResolved>
struct CacheStepLookup {
    static constexpr bool resolved = kResolved;  // each form is its own kernel: less code to fetch
    // arguments
    CacheArgs c;
    const int32_t* sl;        // this request's selection [m]
    int m;
    int32_t* out;             // its sel_slot [m]
    const uint32_t* ab;       // its above-threshold words (early only)
    int early_cap;
    int32_t* status;
    uint32_t* stats;
    // request
    int b, words, nw, chunks;
    int64_t base, n;
    bool early, pre, range_ok;
    uint32_t tail_mask;
    int32_t *t2s, *s2t, *mtok, *mslot;
    uint32_t* fb;
    // shared memory
    uint32_t *keep, *wpre, *fbs, *held, *aw, *apre, *scan;
    const int32_t* pre_slot;  // resolved form: the selection's slots as top-k looked them up
    bool hold;                // the unselected early tokens' slots are held until the misses are placed
    int32_t E_pre;            // resolved form: the early set's size
    uint32_t *s_flags, *s_used;
    // registers
    static constexpr int kPreW = 4096 / NT;                  // 32-slot words per warp held in registers
    static constexpr int kAwPre = (NT >= 1024) ? 1 : 1024 / NT;  // above words per thread in the first round
    int32_t s[kCsPer], j[kCsPer], own[kPreW];
    int64_t triv_n;           // >= 0: the selection is tokens 0 .. triv_n - 1 (not read from memory)
    int32_t after0;
    uint32_t pf_fb, pf_aw[kAwPre];
    uint32_t limit, A, F0;

    // smem: cache_lookup_smem_words(C, AWC) words; scan: 40 words; flags: 2 words.
    __device__ void init(const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, int b_, const int32_t* sel, int m_,
                         int32_t* sel_slot, const uint32_t* above, int cap, const CacheArgs& args, int32_t* st,
                         uint32_t* sts, uint32_t* smem, uint32_t* scan_, uint32_t* flags,
                         bool hold_early) {
        c = args;
        b = b_;
        m = m_;
        status = st;
        stats = sts;
        early_cap = cap;
        int64_t lo, hi;
        range_ok = seg_bounds(tok_off, tok_end, n_tokens, b, &lo, &hi);
        base = lo;
        n = hi - lo;
        words = c.C / 32;
        t2s = c.tok2slot + base;
        s2t = c.slot2tok + static_cast<int64_t>(b) * c.C;
        fb = c.freebits + static_cast<int64_t>(b) * words;
        mtok = c.miss_tok + static_cast<int64_t>(b) * c.C;
        mslot = c.miss_slot + static_cast<int64_t>(b) * c.C;
        sl = sel + static_cast<int64_t>(b) * m;
        out = sel_slot + static_cast<int64_t>(b) * m;
        chunks = (m + NT * kCsPer - 1) / (NT * kCsPer);
        pre_slot = resolved ? sel_slot + static_cast<int64_t>(b) * m : nullptr;
        hold = hold_early;
        E_pre = 0;
        early = !resolved && above != nullptr && early_cap != 0 && n > 0;
        ab = early ? above + 4 * (base / 128 + b) : nullptr;
        nw = early ? static_cast<int>((n + 31) >> 5) : 0;
        tail_mask = (n & 31) ? (1u << (n & 31)) - 1u : ~0u;
        pre = words <= kPreW * (NT / 32);
        keep = smem;
        wpre = keep + words;
        fbs = wpre + words + 1;
        held = fbs + words;
        aw = held + words;
        apre = aw + AWC;
        scan = scan_;
        s_flags = flags;
        s_used = flags + 1;
        limit = 0;
        A = 0;
        F0 = 0;
        triv_n = -1;
    }

    __device__ __forceinline__ uint32_t above_word(int w) const {
        const uint32_t x = __ldcg(ab + w);
        return (w == nw - 1) ? (x & tail_mask) : x;
    }

    __device__ __forceinline__ int32_t sel_at(int i) const {
        if (i >= m) return -1;
        if (triv_n >= 0) return (i < triv_n) ? i : -1;
        return sl[i];
    }

    __device__ __forceinline__ void load_sel(int c0) {
#pragma unroll
        for (int q = 0; q < kCsPer; ++q) s[q] = sel_at(c0 + kCsPer * static_cast<int>(threadIdx.x) + q);
    }

    // The selection's first chunk and the entry after it (first in the first
    // round of loads), then (one chunk) the slots of the selected tokens as
    // the step found them: two dependent rounds, issued before the prologue's
    // scans so that those hide them.
    __device__ void load_selection() {
        load_sel(0);
        after0 = sel_at(kCsPer * static_cast<int>(threadIdx.x) + kCsPer);
        if constexpr (kResolved) {  // the slots top-k looked up, loaded with the selection
#pragma unroll
            for (int q = 0; q < kCsPer; ++q) {
                const int i = kCsPer * static_cast<int>(threadIdx.x) + q;
                j[q] = (i < m) ? pre_slot[i] : -1;
            }
            E_pre = c.early_cnt[b];
        }
    }
    __device__ void load_slots() {
        if (!kResolved && chunks == 1) {
#pragma unroll
            for (int q = 0; q < kCsPer; ++q) j[q] = (s[q] >= 0 && s[q] < n) ? t2s[s[q]] : -1;
        }
    }

    // Prefix of the popcounts of aw[0, len) on top of A (each thread sums `per`
    // consecutive words; one block scan).
    __device__ void above_prefix(int len) {
        const int tid = static_cast<int>(threadIdx.x);
        const int per = (len + NT - 1) / NT;
        uint32_t local = 0;
        for (int i = 0; i < per; ++i) {
            const int w = tid * per + i;
            if (w < len) local += __popc(aw[w]);
        }
        uint32_t tot;
        uint32_t run = A + block_exclusive_scan<NT>(local, scan, &tot);
        for (int i = 0; i < per; ++i) {
            const int w = tid * per + i;
            if (w < len) {
                apre[w] = run;
                run += __popc(aw[w]);
            }
        }
        A += tot;
    }

    // Part 1a: issue the table loads, one word of each table per thread,
    // into registers.
    __device__ void prologue_issue() {
        const int tid = static_cast<int>(threadIdx.x), lane = tid & 31, warp = tid >> 5;
#pragma unroll
        for (int r = 0; r < kPreW; ++r) {
            const int w = warp + r * (NT / 32);
            own[r] = (pre && w < words) ? s2t[w * 32 + lane] : -1;
        }
        pf_fb = (tid < words) ? fb[tid] : 0u;
    }

    // Part 1b: the rest of the free bits into shared memory, then the
    // starting free-slot prefix and the early limit.
    __device__ void prologue_finish() {
        const int tid = static_cast<int>(threadIdx.x);
        for (int w = tid; w < words; w += NT) {
            fbs[w] = (w == tid) ? pf_fb : fb[w];
            keep[w] = 0u;
        }
        if (tid == 0) {
            *s_flags = range_ok ? 0u : static_cast<uint32_t>(ECHO_ST_BADDATA);
            *s_used = 0;
        }
        __syncthreads();
        if (early || resolved) {
            F0 = free_prefix<NT>(fbs, words, scan, wpre, fbs);
            limit = (early_cap < 0) ? F0 : min(F0, static_cast<uint32_t>(early_cap));
        }
    }

    // The first chunk of above words, one per thread, into registers.
    __device__ void load_above() {
#pragma unroll
        for (int i = 0; i < kAwPre; ++i) {
            const int w = static_cast<int>(threadIdx.x) + i * NT;
            pf_aw[i] = (w < min(nw, AWC)) ? above_word(w) : 0u;
        }
    }

    // The first chunk of above words into shared memory and its rank prefix.
    __device__ void above_finish() {
        const int tid = static_cast<int>(threadIdx.x);
        if (early) {
            const int lim = min(nw, AWC);
#pragma unroll
            for (int i = 0; i < kAwPre; ++i)
                if (tid + i * NT < lim) aw[tid + i * NT] = pf_aw[i];
            for (int w = tid + kAwPre * NT; w < lim; w += NT) aw[w] = above_word(w);
            __syncthreads();
            above_prefix(min(nw, AWC));
        }
        __syncthreads();
    }

    // A selected token s with slot jv (-1: not resident): its early slot if it
    // is in the early set and its word lies in the chunk [k0, k0 + AWC).
    __device__ __forceinline__ int32_t lookup(int32_t sv, int32_t jv, int k0, uint32_t* used) {
        if (sv < 0 || sv >= n || jv >= 0) return jv;
        const int w = sv >> 5;
        if (w < k0 || w >= k0 + AWC) return jv;
        const uint32_t word = aw[w - k0];
        const int bit = sv & 31;
        if (!((word >> bit) & 1u)) return jv;
        const uint32_t r = apre[w - k0] + __popc(word & ((1u << bit) - 1u));
        if (r >= limit) return jv;
        FreeWalk walk(wpre, fbs, words, r);
        const int slot = walk.next();
        if (slot < 0) {
            set_status(status, ECHO_ST_BADDATA);
            return jv;
        }
        t2s[sv] = slot;
        s2t[slot] = sv;
        ++*used;
        return slot;
    }

    // Part 2: everything else; every part above has run.
    __device__ void finish() {
        const int tid = static_cast<int>(threadIdx.x), lane = tid & 31, warp = tid >> 5;
        constexpr int kChunk = NT * kCsPer;
        const int C = c.C;
        // the selected tokens of the early set take their slots
        uint32_t used = 0;
        for (int k0 = 0; !kResolved && k0 < nw; k0 += AWC) {
            if (k0 > 0) {
                const int len = min(AWC, nw - k0);
                __syncthreads();  // the previous chunk's look-ups are done
                for (int w = tid; w < len; w += NT) aw[w] = above_word(k0 + w);
                __syncthreads();
                above_prefix(len);
                __syncthreads();
            }
            if (chunks == 1) {
#pragma unroll
                for (int q = 0; q < kCsPer; ++q) j[q] = lookup(s[q], j[q], k0, &used);
            } else {
                for (int ch = 0; ch < chunks; ++ch) {
                    load_sel(ch * kChunk);
#pragma unroll
                    for (int q = 0; q < kCsPer; ++q)
                        lookup(s[q], (s[q] >= 0 && s[q] < n) ? t2s[s[q]] : -1, k0, &used);
                }
            }
        }
        const uint32_t E = resolved ? min(static_cast<uint32_t>(max(E_pre, 0)), F0) : min(A, limit);
        if (used) atomicAdd(s_used, used);
        // the early set's slots (the lowest E free slots at the start) leave the free
        // bits (held: the early set's slots); the selected early tokens keep theirs,
        // the others are free again before the misses are placed, or, holding, after
        // (their early copies may still be in flight)
        for (int w = tid; w < words; w += NT) held[w] = fbs[w];
        __syncthreads();  // every look-up walk over fbs is done before its bits change
        take_lowest_free<NT>(fbs, words, E, wpre);
        __syncthreads();
        for (int w = tid; w < words; w += NT) held[w] &= ~fbs[w];
        __syncthreads();

        // 1a. slots that hold a selected token are kept; the selection must be
        // ascending with -1 padding last
        for (int ch = 0; ch < chunks; ++ch) {
            const int c0 = ch * kChunk;
            int32_t after = after0;
            if (chunks > 1) {
                load_sel(c0);
                after = sel_at(c0 + kCsPer * tid + kCsPer);
            }
            uint32_t flags = 0;
#pragma unroll
            for (int q = 0; q < kCsPer; ++q) {
                const int32_t nxt = (q + 1 < kCsPer) ? s[q + 1] : after;
                if (s[q] >= 0 && s[q] < n) {
                    if (nxt >= 0 && nxt <= s[q]) flags |= ECHO_ST_BADDATA;
                    if (chunks > 1) j[q] = t2s[s[q]];  // the early look-ups above already wrote theirs
                } else {
                    j[q] = -1;
                    if (s[q] >= 0 || nxt >= 0) flags |= ECHO_ST_BADDATA;
                }
            }
            if (flags) atomicOr(s_flags, flags);
#pragma unroll
            for (int q = 0; q < kCsPer; ++q)
                if (j[q] >= 0 && j[q] < C) atomicOr(&keep[j[q] >> 5], 1u << (j[q] & 31));
        }
        __syncthreads();

        // 1b. every other slot occupied at the start of the step is freed (bytes
        // stay, nothing is written back), one warp per 32-slot word
        auto free_word = [&](int w, int32_t st) {
            const int slot = w * 32 + lane;
            const bool kept = (keep[w] >> lane) & 1u;
            const bool freeing = st >= 0 && !kept;
            if (freeing) {
                s2t[slot] = -1;
                if (st < n) t2s[st] = -1;
            }
            const unsigned fm = __ballot_sync(0xffffffffu, freeing);
            if (lane == 0) fbs[w] |= fm;
        };
        if (pre) {
#pragma unroll
            for (int r = 0; r < kPreW; ++r) {
                const int w = warp + r * (NT / 32);
                if (w < words) free_word(w, own[r]);
            }
        } else {
            // only the slots that held a resident token at the start (free bit clear in fb, which
            // this step writes at its end only) and are not kept: their owners' loads go together
            for (int w = tid; w < words; w += NT) {
                uint32_t occ = ~__ldcg(fb + w) & ~keep[w];
                if (!occ) continue;
                fbs[w] |= occ;
                while (occ) {
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
        __syncthreads();

        if (!hold) {  // the unselected early tokens' slots are free for the misses
            for (int w = tid; w < words; w += NT) {
                fbs[w] |= held[w] & ~keep[w];
                held[w] = 0u;
            }
            __syncthreads();
        }

        // 2. free-slot prefix over the new free-bit words
        const uint32_t F = free_prefix<NT>(fbs, words, scan, wpre, fbs);

        // 3. the misses, in ascending token order, take the lowest free slots; the
        // slot of every selected entry is written on the way
        uint32_t found = 0;
        for (int ch = 0; ch < chunks; ++ch) {
            const int c0 = ch * kChunk;
            if (chunks > 1) {  // the registers hold the last chunk only: reload
                load_sel(c0);
#pragma unroll
                for (int q = 0; q < kCsPer; ++q) j[q] = (s[q] >= 0 && s[q] < n) ? t2s[s[q]] : -1;
            }
            uint32_t missing = 0;
#pragma unroll
            for (int q = 0; q < kCsPer; ++q)
                if (s[q] >= 0 && s[q] < n && j[q] < 0) missing |= 1u << q;
            uint32_t tot;
            uint32_t rank = found + block_exclusive_scan<NT>(__popc(missing), scan, &tot);
            FreeWalk walk(wpre, fbs, words, rank < F ? rank : 0u);
#pragma unroll
            for (int q = 0; q < kCsPer; ++q) {
                const int i = c0 + kCsPer * tid + q;
                if (i >= m) break;
                int32_t slot = j[q];
                if (missing & (1u << q)) {
                    slot = (rank < F) ? walk.next() : -1;
                    if (slot >= 0) {
                        if (rank < static_cast<uint32_t>(C)) {
                            mtok[rank] = s[q];
                            mslot[rank] = slot;
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
        take_lowest_free<NT>(fbs, words, got, wpre);
        __syncthreads();
        for (int w = tid; w < words; w += NT) fb[w] = fbs[w] | (held[w] & ~keep[w]);
        if (tid == 0) {
            c.miss_cnt[b] = static_cast<int32_t>(got);
            if (stats && got) atomicAdd(stats + ECHO_STAT_MISSES, got);
            if constexpr (!kResolved) {  // (the resolved form's top-k counted the early set)
                c.early_cnt[b] = static_cast<int32_t>(E);
                if (stats && E) atomicAdd(stats + ECHO_STAT_EARLY, E);
                if (stats && *s_used) atomicAdd(stats + ECHO_STAT_EARLY_USED, *s_used);
            }
            uint32_t flags = *s_flags;
            if (found > F) flags |= ECHO_ST_NOSLOT;
            if (flags) set_status(status, static_cast<int>(flags));
        }
    }
};

}  // namespace echo
