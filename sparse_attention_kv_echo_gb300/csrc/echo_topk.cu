// echo_topk.cu -- exact top-k per request and the EMA threshold update.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2
// "The top-k dependency": selection is an exact top-k; the predicted
// threshold is an EMA (alpha = 0.5) of the previous step's k-th score; the
// real kernel bins scores by the top 8 bits of each score shifted by the
// predicted threshold (panel "Prefill: one-round histogram").
//
// One thread-block cluster of kCS CTAs (1024 threads each) per request; CTA r
// of the cluster owns the r-th contiguous slice of the request's tokens and
// reads its scores from global memory once, into shared memory (slices of up
// to kSliceMax tokens).
//   1. boundary bin: from the 256-bin histogram of the shifted scores (made by
//      the score kernel, or rebuilt here), the bin b* where the count from the
//      top reaches k.  Shifting is monotone, so every token in a bin above b*
//      outranks every token at or below it.
//   2. every CTA counts its slice's tokens above b* and lists its tokens of
//      b* (order key, index) in its own shared memory; one cluster barrier
//      publishes the counts and the lists.
//   3. every CTA gathers the whole boundary bin over distributed shared
//      memory and runs the same radix select on it: K*, the key of the k-th
//      score, then ~index among keys equal to K* for the lower-index tie rule.
//      Redundant selection replaces a broadcast barrier.  When the bin does
//      not fit, the selects run as passes over the scores in global memory.
//   4. a CTA's place in the output is the count of selected tokens in the
//      slices before it (their counts above b*, plus their boundary-bin
//      entries at or above the cut), so one ordered pass per slice writes the
//      indices in ascending order with block-wide scans, with no further
//      exchange.
// A good prediction puts the k-th score near 0 after the shift, where the
// exponent bins are narrow, so the boundary bin holds few tokens.
//
// The cached form (echo_topk_select_cached) also looks up, for every selected
// token, the slot the GPU cache gives it at the start of the step's cache
// step: its resident slot, or, for a token of the early set (above-threshold,
// not resident, rank below the early limit), the rank-th free slot, which it
// enters into the tables; -1 marks a miss.  Each CTA stages its slice's slot
// entries and above-threshold words with the scores, the request's free bits
// and their prefix, and exchanges its above-threshold count at the selection's
// cluster barrier, so the look-up needs no further exchange.
#include <cooperative_groups.h>

#include "echo_common.cuh"
#include "echo_internal.h"
#include "echo_radix.cuh"
#include "echo_slots.cuh"

namespace cg = cooperative_groups;

namespace echo {
namespace {

using namespace radix;

constexpr int kCS = 8;            // CTAs per request (one cluster)
constexpr int kCandMax = 6144;    // boundary-bin entries of a request a CTA gathers
constexpr int kCandLocal = 2048;  // boundary-bin entries of one slice
constexpr int kFbWordsMax = 1024; // free-bit words of a request the cached form stages (C <= 32768)
constexpr int kSliceMax = 16384;  // scores of its slice a CTA keeps in shared memory

struct TopkShared {
    uint32_t hist[256];
    uint32_t hist_acc[256];        // leader: cluster-wide rebuild of the histogram
    uint32_t scan[40];
    uint32_t cand_key[kCandMax];   // the request's boundary bin, slices in rank order
    uint32_t cand_idx[kCandMax];
    uint32_t loc_key[kCandLocal];  // this slice's boundary-bin entries
    uint32_t loc_idx[kCandLocal];
    uint32_t r_above[kCS];         // per slice: tokens above b*
    uint32_t r_cnt[kCS];           // per slice: boundary-bin entries
    uint32_t r_ex[kCS];            // per slice: the caller's count exchanged with them
    uint32_t cnt;                  // this slice: boundary-bin entries
    uint32_t n_above;              // this slice: tokens above b*
    uint32_t ex;                   // this slice: the caller's count
    uint32_t red[3];               // radix select: min, max and count of the elements
    uint32_t taken[2];             // boundary-bin entries taken: before this slice, in all
    uint32_t digit;
    uint32_t above;
    uint32_t minkey;
    uint32_t flag;
};

__host__ __device__ constexpr size_t topk_cache_offset() { return (sizeof(TopkShared) + 15) / 16 * 16; }
constexpr size_t kTopkSmem = topk_cache_offset() + sizeof(float) * kSliceMax;
// cached form, after the scores: slot entries of the slice [kSliceMax] | free bits
// [kFbWordsMax] | their prefix [kFbWordsMax + 1] | above words of the slice [kSliceMax/32 + 2]
constexpr size_t kAwSlice = kSliceMax / 32 + 2;
constexpr size_t kTopkCachedSmem =
    kTopkSmem + sizeof(int32_t) * kSliceMax + sizeof(uint32_t) * (2 * kFbWordsMax + 1 + kAwSlice);
static_assert(kTopkCachedSmem <= 227u * 1024u, "top-k shared memory");

// Split cluster barrier: arrive says this CTA is done reading the others'
// shared memory; wait (before exit) lets no CTA leave while another may still
// read its shared memory.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Segments: decode requests (CSR tok_off over the scores) or prefill rows
// (W > 0: row b holds row0 + b + 1 scores starting at b * W).  In prefill the
// threshold is one scalar for every row and is not updated here.
struct TopkSegs {
    const int64_t* tok_off;
    const int64_t* tok_end;  // optional current ends (growing contexts)
    int64_t n_tokens;
    int64_t row0;
    int64_t W;
};

// The 256-bin histogram of the request's shifted scores summed over the
// cluster's slices (out of line: only when the one given does not describe
// the scores or none is given).
__device__ __noinline__ void rebuild_hist(cg::cluster_group& cluster, TopkShared& sh, TopkShared& lsh, bool leader,
                                          const float* xs, int64_t s_lo, int64_t s_hi, float shift) {
    const int tid = threadIdx.x;
    if (leader)
        for (int i = tid; i < 256; i += kTT) sh.hist_acc[i] = 0u;
    for (int i = tid; i < 256; i += kTT) sh.hist[i] = 0u;
    cluster.sync();
    for (int64_t s0 = s_lo; s0 < s_hi; s0 += kTT) {
        const int64_t s = s0 + tid;
        const bool v = s < s_hi;
        const uint32_t bin = v ? shifted_bin(xs[s - s_lo], shift) : 256u;
        const unsigned grp = __match_any_sync(0xffffffffu, bin);
        if (v && (tid & 31) == __ffs(grp) - 1) atomicAdd(&sh.hist[bin], __popc(grp));
    }
    __syncthreads();
    for (int i = tid; i < 256; i += kTT)
        if (sh.hist[i]) atomicAdd(&lsh.hist_acc[i], sh.hist[i]);
    cluster.sync();
    for (int i = tid; i < 256; i += kTT) sh.hist[i] = lsh.hist_acc[i];
}

// Outcome of the cluster-wide selection for the calling CTA's slice.
struct SliceSel {
    uint32_t bstar, K, idx_cut;
    uint32_t offset;     // selected tokens of the slices before this one
    uint32_t total;      // selected tokens of the request
    uint32_t ex_before;  // the exchanged counts of the slices before this one
    uint32_t ex_all;     // the exchanged counts of every slice
};

// Steps 1-4 of the selection of a request with n > k, block-wide in every CTA
// of its cluster.  xs: the slice's scores (xs[i] = token s_lo + i; shared or
// global memory), sc: the request's scores.  ex_mine: a count the caller
// exchanges with the slices' counts (0 when it has none).  Ends with the split
// barrier's arrive; the caller waits on it before it exits.
__device__ SliceSel cluster_select(cg::cluster_group& cluster, TopkShared& sh, TopkShared& lsh, int rank, bool leader,
                                   const float* xs, const float* sc, int64_t s_lo, int64_t s_hi, int64_t n, int k,
                                   float shift, bool have, uint32_t hist_mine, uint32_t ex_mine, int32_t* status,
                                   uint32_t* stats) {
    const int tid = threadIdx.x;
    // ---- 1-2. boundary bin; each slice lists its boundary-bin tokens in its own shared memory
    uint32_t bstar = 0, above = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        if (have) {
            if (tid < 256) sh.hist[tid] = hist_mine;
        } else {
            rebuild_hist(cluster, sh, lsh, leader, xs, s_lo, s_hi, shift);
        }
        __syncthreads();
        if (tid < 32) find_digit(sh.hist, static_cast<uint32_t>(k), &sh.digit, &sh.above);
        if (tid == 0) {
            sh.cnt = 0;
            sh.n_above = 0;
            sh.ex = ex_mine;
        }
        __syncthreads();
        bstar = sh.digit;
        above = sh.above;
        const uint32_t eq_total = sh.hist[bstar];
        uint32_t my_above = 0;
        for (int64_t s0 = s_lo; s0 < s_hi; s0 += kTT) {
            const int64_t s = s0 + tid;
            const bool v = s < s_hi;
            const float x = v ? xs[s - s_lo] : 0.f;
            const uint32_t bin = shifted_bin(x, shift);
            my_above += v && bin > bstar;
            const bool in = v && bin == bstar;
            const unsigned m = __ballot_sync(0xffffffffu, in);
            if (m) {
                const int first = __ffs(m) - 1;
                uint32_t base = 0;
                if ((tid & 31) == first) base = atomicAdd(&sh.cnt, static_cast<uint32_t>(__popc(m)));
                base = __shfl_sync(0xffffffffu, base, first);
                const uint32_t pos = base + __popc(m & ((1u << (tid & 31)) - 1u));
                if (in && pos < kCandLocal) {
                    sh.loc_key[pos] = order_key(x);
                    sh.loc_idx[pos] = static_cast<uint32_t>(s);
                }
            }
        }
        my_above = __reduce_add_sync(0xffffffffu, my_above);
        if ((tid & 31) == 0 && my_above) atomicAdd(&sh.n_above, my_above);
        cluster.sync();  // every slice's counts and list are complete
        if (tid < kCS) {
            sh.r_above[tid] = *cluster.map_shared_rank(&sh.n_above, tid);
            sh.r_cnt[tid] = *cluster.map_shared_rank(&sh.cnt, tid);
            sh.r_ex[tid] = *cluster.map_shared_rank(&sh.ex, tid);
        }
        __syncthreads();
        uint32_t sum_above = 0, sum_cnt = 0;
        for (int r = 0; r < kCS; ++r) {
            sum_above += sh.r_above[r];
            sum_cnt += sh.r_cnt[r];
        }
        if (sum_above == above && sum_cnt == eq_total) break;
        // The histogram given does not describe these scores: rebuild it here.
        if (leader && tid == 0) set_status(status, ECHO_ST_BADDATA);
        have = false;
        cluster.sync();  // every slice has read the counts before they are reset
    }

    // ---- 3. the boundary bin gathered (slices in rank order), K* and the index cut
    uint32_t above_before = 0, pre = 0, total_cnt = 0, above_all = 0, ex_before = 0, ex_all = 0;
    bool fits = true;
    for (int r = 0; r < kCS; ++r) {
        const uint32_t a = sh.r_above[r], c = sh.r_cnt[r], e = sh.r_ex[r];
        if (r < rank) {
            above_before += a;
            pre += c;
            ex_before += e;
        }
        above_all += a;
        total_cnt += c;
        ex_all += e;
        fits = fits && c <= static_cast<uint32_t>(kCandLocal);
    }
    fits = fits && total_cnt <= static_cast<uint32_t>(kCandMax);
    if (fits) {
        for (uint32_t g0 = 0; g0 < total_cnt; g0 += 2 * kTT) {
            uint32_t kv[2] = {0u, 0u}, iv[2] = {0u, 0u};
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t g = g0 + j * kTT + tid;
                if (g < total_cnt) {
                    int r = 0;
                    uint32_t base = 0;
                    while (r < kCS - 1 && g >= base + sh.r_cnt[r]) base += sh.r_cnt[r++];
                    kv[j] = *cluster.map_shared_rank(&sh.loc_key[g - base], r);
                    iv[j] = *cluster.map_shared_rank(&sh.loc_idx[g - base], r);
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t g = g0 + j * kTT + tid;
                if (g < total_cnt) {
                    sh.cand_key[g] = kv[j];
                    sh.cand_idx[g] = iv[j];
                }
            }
        }
    }
    if (tid == 0) {
        sh.taken[0] = 0;
        sh.taken[1] = 0;
    }
    cluster_arrive_release();  // done reading the other slices' shared memory
    __syncthreads();
    if (leader && tid == 0 && stats) {
        atomicMax(stats + ECHO_STAT_BOUNDARY_MAX, total_cnt);
        if (!fits) atomicAdd(stats + ECHO_STAT_TOPK_FALLBACK, 1u);
    }
    const uint32_t need = static_cast<uint32_t>(k) - above;  // >= 1
    uint32_t rem = 0, eqn = 0, K = 0, idx_cut = 0xFFFFFFFFu;
    if (fits) {
        SmemCands src{sh.cand_key, sh.cand_idx, total_cnt, false, 0};
        K = radix_select(src, need, sh, &rem, &eqn);
        if (rem < eqn) {
            SmemCands src2{sh.cand_key, sh.cand_idx, total_cnt, true, K};
            uint32_t r2, e2;
            idx_cut = ~radix_select(src2, rem, sh, &r2, &e2);
        }
    } else {
        K = global_select(sc, n, shift, bstar, need, sh, &idx_cut);
    }

    // ---- 4. this slice's place: the selected tokens of the slices before it
    uint32_t t_before = 0, t_all = 0;
    if (fits) {
        for (uint32_t i = tid; i < total_cnt; i += kTT) {
            const uint32_t key = sh.cand_key[i];
            const bool t = key > K || (key == K && sh.cand_idx[i] <= idx_cut);
            t_all += t;
            t_before += t && i < pre;
        }
    } else {
        const int64_t lim = leader ? n : s_lo;
        for (int64_t s = tid; s < lim; s += kTT) {
            const float x = sc[s];
            if (shifted_bin(x, shift) != bstar) continue;
            const uint32_t key = order_key(x);
            const bool t = key > K || (key == K && static_cast<uint32_t>(s) <= idx_cut);
            t_all += t;
            t_before += t && s < s_lo;
        }
    }
    t_before = __reduce_add_sync(0xffffffffu, t_before);
    t_all = __reduce_add_sync(0xffffffffu, t_all);
    if ((tid & 31) == 0) {
        if (t_before) atomicAdd(&sh.taken[0], t_before);
        if (t_all) atomicAdd(&sh.taken[1], t_all);
    }
    __syncthreads();
    SliceSel r;
    r.bstar = bstar;
    r.K = K;
    r.idx_cut = idx_cut;
    r.offset = above_before + sh.taken[0];
    r.total = above_all + sh.taken[1];
    r.ex_before = ex_before;
    r.ex_all = ex_all;
    return r;
}

__global__ void __cluster_dims__(kCS, 1, 1) __launch_bounds__(kTT, 1)
    topk_kernel(TopkSegs segs, const float* __restrict__ scores, int k, const uint32_t* __restrict__ hist,
                float* theta_hat, float alpha, int32_t* __restrict__ sel, float* kth_out, int32_t* status,
                uint32_t* stats) {
    pdl_launch_dependents();  // a programmatic dependent (the cache step) may start its table prologue
    extern __shared__ uint8_t smem_raw[];
    TopkShared& sh = *reinterpret_cast<TopkShared*>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const bool leader = rank == 0;
    TopkShared& lsh = *cluster.map_shared_rank(&sh, 0);     // the leader's shared memory
    const int b = blockIdx.x / kCS, tid = threadIdx.x;
    const bool prefill = segs.W > 0;
    int64_t lo, n;
    if (prefill) {
        lo = static_cast<int64_t>(b) * segs.W;
        n = segs.row0 + b + 1;
        if (n > segs.W) {
            if (leader && tid == 0) set_status(status, ECHO_ST_BADDATA);
            n = 0;
        }
    } else {
        int64_t hi;
        if (!seg_bounds(segs.tok_off, segs.tok_end, segs.n_tokens, b, &lo, &hi) && leader && tid == 0)
            set_status(status, ECHO_ST_BADDATA);
        n = hi - lo;
    }
    const float* sc = scores + (n > 0 ? lo : 0);
    int32_t* out = sel + static_cast<int64_t>(b) * k;
    float* const theta_upd = prefill ? nullptr : theta_hat;   // prefill: one scalar, updated per block
    const float th_old = theta_hat ? theta_hat[prefill ? 0 : b] : __int_as_float(0x7f800000);
    const float shift = isfinite(th_old) ? th_old : 0.f;

    // ---- trivial requests: the leader alone, no cluster traffic
    if (n == 0) {
        if (!leader) return;
        for (int i = tid; i < k; i += kTT) out[i] = -1;
        if (tid == 0) kth_out[b] = __int_as_float(0xff800000);
        return;
    }
    if (n <= k) {
        if (!leader) return;
        if (tid == 0) {
            sh.minkey = 0xFFFFFFFFu;
            sh.flag = 0;
        }
        __syncthreads();
        uint32_t mk = 0xFFFFFFFFu;
        bool nan = false;
        for (int64_t s = tid; s < n; s += kTT) {
            const float x = sc[s];
            nan |= isnan(x);
            mk = min(mk, order_key(x));
        }
        for (int i = tid; i < k; i += kTT) out[i] = (i < n) ? i : -1;
        atomicMin(&sh.minkey, mk);
        if (nan) sh.flag = 1;
        __syncthreads();
        if (tid == 0) {
            if (sh.flag) set_status(status, ECHO_ST_NAN);
            const float kth = key_to_float(sh.minkey);
            kth_out[b] = kth;
            if (theta_upd) theta_upd[b] = ema_update(th_old, kth, alpha);
        }
        return;
    }

    // this CTA's slice of the request; its scores are staged in shared memory
    // when they fit (xs[i] is the score of token s_lo + i), the histogram row
    // is fetched alongside
    const int64_t s_lo = n * rank / kCS, s_hi = n * (rank + 1) / kCS;
    const int64_t len = s_hi - s_lo;
    const uint32_t hist_mine = (hist && tid < 256) ? hist[static_cast<int64_t>(b) * 256 + tid] : 0u;
    float* const cache = reinterpret_cast<float*>(smem_raw + topk_cache_offset());
    const bool cached = len <= kSliceMax;
    if (cached) {
        for (int64_t i0 = 0; i0 < len; i0 += 4 * kTT) {
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t i = i0 + j * kTT + tid;
                v[j] = i < len ? sc[s_lo + i] : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t i = i0 + j * kTT + tid;
                if (i < len) cache[i] = v[j];
            }
        }
    }
    const float* const xs = cached ? cache : sc + s_lo;

    const SliceSel ss = cluster_select(cluster, sh, lsh, rank, leader, xs, sc, s_lo, s_hi, n, k, shift,
                                       hist != nullptr, hist_mine, 0u, status, stats);

    // ---- 5. ordered write of the slice's selected indices
    uint32_t written = ss.offset;
    bool nan = false;
    for (int64_t c0 = s_lo; c0 < s_hi; c0 += 4 * kTT) {
        const int64_t s0 = c0 + 4 * tid;
        uint32_t f = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t s = s0 + j;
            if (s < s_hi) {
                const float x = xs[s - s_lo];
                nan |= isnan(x);
                if (takes(x, shift, ss.bstar, ss.K, ss.idx_cut, s)) f |= 1u << j;
            }
        }
        uint32_t tot;
        uint32_t pos = written + block_exclusive_scan<kTT>(__popc(f), sh.scan, &tot);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (f & (1u << j)) {
                if (pos < static_cast<uint32_t>(k)) out[pos] = static_cast<int32_t>(s0 + j);
                ++pos;
            }
        written += tot;
    }
    if (leader) {
        for (int i = static_cast<int>(ss.total) + tid; i < k; i += kTT) out[i] = -1;
        if (tid == 0) {
            if (ss.total != static_cast<uint32_t>(k)) set_status(status, ECHO_ST_BADDATA);
            const float kth = key_to_float(ss.K);
            kth_out[b] = kth;
            if (theta_upd) theta_upd[b] = ema_update(th_old, kth, alpha);
        }
    }
    if (__any_sync(0xffffffffu, nan) && (tid & 31) == 0) set_status(status, ECHO_ST_NAN);
    cluster_wait_acquire();  // no CTA leaves while another may still read its shared memory
}

// The GPU cache as the cached form sees it.
struct TopkCache {
    const uint32_t* above;     // above-threshold words (echo_index_scores layout); null: no early set
    int early_cap;             // < 0: no cap but the free slots
    int32_t* tok2slot;         // [n_tokens] request-local slots; the early entries are written here
    int32_t* slot2tok;         // [B*C]
    const uint32_t* freebits;  // [B*C/32] free bits at the step's start
    int32_t* early_cnt;        // [B] out: the early set's size
    int32_t* sel_slot;         // [B*k] out: slot of each selected entry (-1: a miss, padding)
    int C;
};

__global__ void __cluster_dims__(kCS, 1, 1) __launch_bounds__(kTT, 1)
    topk_cached_kernel(TopkSegs segs, const float* __restrict__ scores, int k, const uint32_t* __restrict__ hist,
                       float* theta_hat, float alpha, int32_t* __restrict__ sel, float* kth_out, TopkCache tc,
                       int32_t* status, uint32_t* stats) {
    pdl_launch_dependents();  // a programmatic dependent (the cache step) may start its table prologue
    extern __shared__ uint8_t smem_raw[];
    TopkShared& sh = *reinterpret_cast<TopkShared*>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const bool leader = rank == 0;
    TopkShared& lsh = *cluster.map_shared_rank(&sh, 0);
    const int b = blockIdx.x / kCS, tid = threadIdx.x;
    int64_t lo, n;
    {
        int64_t hi;
        if (!seg_bounds(segs.tok_off, segs.tok_end, segs.n_tokens, b, &lo, &hi) && leader && tid == 0)
            set_status(status, ECHO_ST_BADDATA);
        n = hi - lo;
    }
    const float* sc = scores + lo;
    int32_t* out = sel + static_cast<int64_t>(b) * k;
    int32_t* out_slot = tc.sel_slot + static_cast<int64_t>(b) * k;
    const float th_old = theta_hat ? theta_hat[b] : __int_as_float(0x7f800000);
    const float shift = isfinite(th_old) ? th_old : 0.f;
    const int words = tc.C / 32;
    int32_t* t2s = tc.tok2slot + lo;
    int32_t* s2t = tc.slot2tok + static_cast<int64_t>(b) * tc.C;
    const uint32_t* ab = tc.above ? tc.above + 4 * (lo / 128 + b) : nullptr;

    // this CTA's slice: scores and slot entries staged in shared memory when the
    // slice fits, with the request's free bits and the slice's above words
    const int64_t s_lo = n * rank / kCS, s_hi = n * (rank + 1) / kCS;
    const int64_t len = s_hi - s_lo;
    const uint32_t hist_mine = (hist && tid < 256) ? hist[static_cast<int64_t>(b) * 256 + tid] : 0u;
    const uint32_t fb_mine = (tid < words) ? tc.freebits[static_cast<int64_t>(b) * words + tid] : 0u;
    float* const cache = reinterpret_cast<float*>(smem_raw + topk_cache_offset());
    int32_t* const tcache = reinterpret_cast<int32_t*>(smem_raw + kTopkSmem);
    uint32_t* const fbs = reinterpret_cast<uint32_t*>(tcache + kSliceMax);
    uint32_t* const wpre = fbs + kFbWordsMax;
    uint32_t* const aw = wpre + kFbWordsMax + 1;
    const bool cached = len <= kSliceMax;
    if (tid == 0) sh.red[0] = 0u;
    if (cached) {
        for (int64_t i0 = 0; i0 < len; i0 += 4 * kTT) {
            float v[4];
            int32_t t[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t i = i0 + j * kTT + tid;
                v[j] = i < len ? sc[s_lo + i] : 0.f;
                t[j] = i < len ? t2s[s_lo + i] : -1;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t i = i0 + j * kTT + tid;
                if (i < len) {
                    cache[i] = v[j];
                    tcache[i] = t[j];
                }
            }
        }
    }
    const float* const xs = cached ? cache : sc + s_lo;
    // above word w of the request with the bits of tokens outside the slice cleared
    const int64_t w_lo = s_lo >> 5;
    const int nwa = len > 0 ? static_cast<int>(((s_hi - 1) >> 5) - w_lo + 1) : 0;
    auto above_word = [&](int64_t w) -> uint32_t {
        uint32_t x = __ldcg(ab + w);
        const int64_t t0 = w * 32;
        if (t0 < s_lo) x &= ~0u << static_cast<int>(s_lo - t0);
        if (t0 + 32 > s_hi) x &= (1u << static_cast<int>(s_hi - t0)) - 1u;
        return x;
    };
    if (ab && cached)
        for (int i = tid; i < nwa; i += kTT) aw[i] = above_word(w_lo + i);
    __syncthreads();
    // the free-slot prefix of the start free bits, this slice's above-threshold count
    uint32_t F0;
    {
        uint32_t tot;
        const uint32_t ex = block_exclusive_scan<kTT>(static_cast<uint32_t>(__popc(fb_mine)), sh.scan, &tot);
        if (tid < words) {
            fbs[tid] = fb_mine;
            wpre[tid] = ex;
        }
        if (tid == 0) wpre[words] = tot;
        F0 = tot;
    }
    if (ab) {
        uint32_t mine = 0;
        for (int i = tid; i < nwa; i += kTT) mine += __popc(cached ? aw[i] : above_word(w_lo + i));
        mine = __reduce_add_sync(0xffffffffu, mine);
        if ((tid & 31) == 0 && mine) atomicAdd(&sh.red[0], mine);
    }
    __syncthreads();
    const uint32_t a_cnt = sh.red[0];
    const uint32_t limit = ab ? ((tc.early_cap < 0) ? F0 : min(F0, static_cast<uint32_t>(tc.early_cap))) : 0u;
    auto above_bit = [&](int64_t s) -> uint32_t {
        const uint32_t x = cached ? aw[(s >> 5) - w_lo] : above_word(s >> 5);
        return (x >> (s & 31)) & 1u;
    };

    // ---- selection; every token when n <= k
    const bool all = n <= k;
    SliceSel ss;
    if (!all) {
        ss = cluster_select(cluster, sh, lsh, rank, leader, xs, sc, s_lo, s_hi, n, k, shift, hist != nullptr,
                            hist_mine, a_cnt, status, stats);
    } else {
        // the slices exchange their above counts and their smallest keys (the k-th score)
        uint32_t mk = 0xFFFFFFFFu;
        for (int64_t s = s_lo + tid; s < s_hi; s += kTT) mk = min(mk, order_key(xs[s - s_lo]));
        mk = __reduce_min_sync(0xffffffffu, mk);
        if (tid == 0) {
            sh.ex = a_cnt;
            sh.minkey = 0xFFFFFFFFu;
        }
        __syncthreads();
        if ((tid & 31) == 0) atomicMin(&sh.minkey, mk);
        cluster.sync();
        if (tid < kCS) {
            sh.r_ex[tid] = *cluster.map_shared_rank(&sh.ex, tid);
            sh.r_cnt[tid] = *cluster.map_shared_rank(&sh.minkey, tid);
        }
        __syncthreads();
        ss.bstar = 0;
        ss.K = 0xFFFFFFFFu;
        ss.idx_cut = 0;
        ss.offset = static_cast<uint32_t>(s_lo);
        ss.total = static_cast<uint32_t>(n);
        ss.ex_before = 0;
        ss.ex_all = 0;
        for (int r = 0; r < kCS; ++r) {
            const uint32_t e = sh.r_ex[r];
            if (r < rank) ss.ex_before += e;
            ss.ex_all += e;
            ss.K = min(ss.K, sh.r_cnt[r]);
        }
        cluster_arrive_release();  // done reading the other slices' shared memory
    }
    const uint32_t E = min(ss.ex_all, limit);

    // ---- 5. ordered write of the slice's selected indices and their slots: the
    // resident slot, or for a token of the early set the rank-th free slot at the
    // step's start (entered into the tables here), else -1 (a miss)
    uint32_t written = ss.offset, abase = ss.ex_before, used = 0;
    bool nan = false, bad = false;
    for (int64_t c0 = s_lo; c0 < s_hi; c0 += 4 * kTT) {
        const int64_t s0 = c0 + 4 * tid;
        uint32_t f = 0, a = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t s = s0 + j;
            if (s < s_hi) {
                const float x = xs[s - s_lo];
                nan |= isnan(x);
                if (all || takes(x, shift, ss.bstar, ss.K, ss.idx_cut, s)) f |= 1u << j;
                if (ab && above_bit(s)) a |= 1u << j;
            }
        }
        uint32_t tot;
        const uint32_t ex =
            block_exclusive_scan<kTT>(static_cast<uint32_t>(__popc(f)) | (static_cast<uint32_t>(__popc(a)) << 16),
                                      sh.scan, &tot);
        uint32_t pos = written + (ex & 0xFFFFu);
        const uint32_t ar = abase + (ex >> 16);
        // slots as the step found them; e: the taken tokens of the early set (the
        // thread's above tokens have consecutive ranks, so one walk serves them all)
        int32_t sl[4];
        uint32_t e = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t s = s0 + j;
            sl[j] = (f & (1u << j)) ? (cached ? tcache[s - s_lo] : t2s[s]) : -1;
            if ((f & (1u << j)) && sl[j] < 0 && (a & (1u << j)) && ar + __popc(a & ((1u << j) - 1u)) < limit)
                e |= 1u << j;
        }
        if (e) {
            const int j0 = __ffs(e) - 1;
            uint32_t wr = ar + __popc(a & ((1u << j0) - 1u));
            FreeWalk walk(wpre, fbs, words, wr);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (a & (1u << j)) {
                    const uint32_t r = ar + __popc(a & ((1u << j) - 1u));
                    if (!(e & (1u << j)) || r < wr) continue;
                    while (wr < r) {  // the free slots of the thread's unselected above tokens
                        walk.next();
                        ++wr;
                    }
                    const int slot = walk.next();
                    ++wr;
                    const int64_t s = s0 + j;
                    if (slot >= 0) {
                        sl[j] = slot;
                        t2s[s] = slot;
                        s2t[slot] = static_cast<int32_t>(s);
                        ++used;
                    } else {
                        bad = true;
                    }
                }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (f & (1u << j)) {
                if (pos < static_cast<uint32_t>(k)) {
                    out[pos] = static_cast<int32_t>(s0 + j);
                    out_slot[pos] = sl[j];
                }
                ++pos;
            }
        written += tot & 0xFFFFu;
        abase += tot >> 16;
    }
    if (leader) {
        for (int i = static_cast<int>(ss.total) + tid; i < k; i += kTT) {
            out[i] = -1;
            out_slot[i] = -1;
        }
        if (tid == 0) {
            const uint32_t want = all ? static_cast<uint32_t>(n) : static_cast<uint32_t>(k);
            if (ss.total != want) set_status(status, ECHO_ST_BADDATA);
            if (n == 0) {
                kth_out[b] = __int_as_float(0xff800000);
            } else {
                const float kth = key_to_float(ss.K);
                kth_out[b] = kth;
                if (theta_hat) theta_hat[b] = ema_update(th_old, kth, alpha);
            }
            tc.early_cnt[b] = static_cast<int32_t>(E);
            if (stats && E) atomicAdd(stats + ECHO_STAT_EARLY, E);
        }
    }
    used = __reduce_add_sync(0xffffffffu, used);
    if ((tid & 31) == 0 && used && stats) atomicAdd(stats + ECHO_STAT_EARLY_USED, used);
    if (__any_sync(0xffffffffu, nan) && (tid & 31) == 0) set_status(status, ECHO_ST_NAN);
    if (__any_sync(0xffffffffu, bad) && (tid & 31) == 0) set_status(status, ECHO_ST_BADDATA);
    cluster_wait_acquire();  // no CTA leaves while another may still read its shared memory
}

}  // namespace
}  // namespace echo

namespace echo {

int launch_topk(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, int64_t row0, int64_t W, const float* scores, int k,
                const uint32_t* hist, float* theta_hat, float alpha, int32_t* sel_idx, float* kth, int32_t* status,
                uint32_t* stats, cudaStream_t stream) {
    const size_t smem = kTopkSmem;
    ECHO_CUDA_OK(prefer_max_shared(topk_kernel));
    ECHO_CUDA_OK(cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
    if (W > 0)  // prefill rows: one block per row, each row's scores read once
        return launch_select_rows(B, row0, W, scores, k, hist, theta_hat, sel_idx, kth, status, stats, stream);
    TopkSegs segs{tok_off, tok_end, n_tokens, row0, W};
    topk_kernel<<<B * kCS, kTT, smem, stream>>>(segs, scores, k, hist, theta_hat, alpha, sel_idx, kth, status, stats);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}

}  // namespace echo

extern "C" int echo_topk_select(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                                const float* scores, int k,
                                const uint32_t* hist, float* theta_hat, float alpha, int32_t* sel_idx, float* kth,
                                int32_t* status, uint32_t* stats, echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || n_tokens < 0 || k <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !sel_idx || !kth || !status || (n_tokens > 0 && !scores)) return ECHO_EINVAL;
    if (n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    return launch_topk(B, tok_off, tok_end, n_tokens, 0, 0, scores, k, hist, theta_hat, alpha, sel_idx, kth, status, stats,
                       stream);
}

namespace echo {

int launch_topk_cached(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, const float* scores, int k,
                       const uint32_t* hist, float* theta_hat, float alpha, int32_t* sel_idx, float* kth,
                       const uint32_t* above, int early_cap, const echo_cache* cache, int32_t* sel_slot,
                       int32_t* status, uint32_t* stats, cudaStream_t stream) {
    const size_t smem = kTopkCachedSmem;
    ECHO_CUDA_OK(prefer_max_shared(topk_cached_kernel));
    ECHO_CUDA_OK(cudaFuncSetAttribute(topk_cached_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
    TopkSegs segs{tok_off, tok_end, n_tokens, 0, 0};
    TopkCache tc{above, early_cap, cache->tok2slot, cache->slot2tok, cache->freebits, cache->early_cnt, sel_slot,
                 static_cast<int>(cache->C)};
    topk_cached_kernel<<<B * kCS, kTT, smem, stream>>>(segs, scores, k, hist, theta_hat, alpha, sel_idx, kth, tc,
                                                       status, stats);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}

}  // namespace echo

extern "C" int echo_topk_select_cached(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                                       const float* scores, int k,
                                       const uint32_t* hist, float* theta_hat, float alpha, int32_t* sel_idx,
                                       float* kth, const uint32_t* above, int early_cap, const echo_cache* cache,
                                       int32_t* sel_slot, int32_t* status, uint32_t* stats, echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || n_tokens < 0 || k <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !sel_idx || !kth || !status || !sel_slot || (n_tokens > 0 && !scores)) return ECHO_EINVAL;
    if (n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    const int rc = check_cache(cache, B, k);
    if (rc) return rc;
    if (cache->C / 32 > kFbWordsMax) return ECHO_EUNSUPPORTED;
    return launch_topk_cached(B, tok_off, tok_end, n_tokens, scores, k, hist, theta_hat, alpha, sel_idx, kth, above, early_cap,
                              cache, sel_slot, status, stats, static_cast<cudaStream_t>(stream));
}
