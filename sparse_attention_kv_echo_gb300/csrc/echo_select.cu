// echo_select.cu -- decode top-k from candidate lists, one thread block per request.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2
// "The top-k dependency": the selection is an exact top-k of the scores, the
// predicted threshold an EMA (alpha = 0.5) of the previous step's k-th score,
// and the one-round histogram bins the threshold-shifted scores by their top
// 8 bits (panel "Prefill: one-round histogram").
//
// The score kernel appends, per request, every token whose score key reaches
// the request's cut to a candidate list.  A list that holds at least k tokens
// holds the whole top-k (the k-th score is then at or above the cut), so the
// block selects among the list alone: the list into shared memory, the k-th
// key and the index cut by radix select, the selected tokens marked in a
// bitmap of the request's tokens, and one ordered pass over the bitmap words
// writes the indices in ascending order.  Otherwise (no list yet, too few or
// too many entries) it selects from all the scores: the boundary bin b* from
// the histogram, one pass that writes the bitmap words of the tokens above b*
// (one ballot per 32 tokens) and gathers b*'s entries into shared memory, the
// cut inside b* by radix select, and the same ordered pass.  A b* too large
// for shared memory gets a second round of 256 bins over the next 8 bits of
// its shifted keys (one counting pass, one gather pass of the sub-bin that
// holds the k-th token); only a sub-bin that still does not fit (thousands of
// equal scores) is selected by radix passes over the scores.  Every pass over
// the scores keeps 8 loads per thread in flight.
//
// The cached form also gives every selected token the slot it holds at the
// start of the cache step: its resident slot, or, for a token of the early set
// (above the prediction, not resident, rank among the marked tokens below the
// early limit), the rank-th free slot of the step's starting free bits, which
// it enters into the tables.  The ordered pass walks the above-threshold words
// beside the bitmap: a thread's marked tokens have consecutive ranks, so one
// walk over the free bits serves all of them.
//
// The next step's cut is the key of rank 4k of this step: exactly, when the
// step selected from all its scores (from the gathered bin, or by radix
// passes over the bin that holds that rank); a list that holds between 3k and
// 6k tokens keeps its cut, a longer one is cut at its rank-4k key, a shorter
// one is lowered to a histogram bin edge with at most 12288 tokens above it.
// The cut only decides which path the next step takes.
#include "echo_common.cuh"
#include "echo_internal.h"
#include "echo_radix.cuh"
#include "echo_slots.cuh"

namespace echo {
namespace {

using namespace radix;

constexpr int kSelCap = 16384;                 // list entries / boundary-bin entries in shared memory
constexpr int64_t kWinTokens = 1 << 19;        // tokens per bitmap window (64 KB)
constexpr int kWinWords = static_cast<int>(kWinTokens / 32);
constexpr int kFbMax = 1024;                   // free-bit words of a request (C <= 32768)
constexpr uint32_t kNoCut = 0xFFFFFFFFu;
constexpr uint32_t kCutRank = 4;               // next cut: the key of rank 4k ...
constexpr uint32_t kCutLow = 3, kCutHigh = 6;  // ... recomputed when a list leaves [3k, 6k] entries
constexpr uint32_t kCutMaxAbove = 12288;       // histogram rule: tokens above the cut at most

struct SelShared {
    uint32_t hist[256];
    uint32_t red[3];
    uint32_t digit, above;
    uint32_t digit2, above2;   // the bin of the next cut's rank
    uint32_t scan[40];
    uint32_t cnt;       // boundary-bin entries seen
    uint32_t n_above;   // tokens above the boundary bin
    uint32_t flag;      // the list is inconsistent with the request
    uint32_t nan;
    uint32_t minkey;
    uint32_t used;      // early tokens entered into the tables
    uint32_t cut;       // the next step's cut (warp 0 of cut_from_hist)
};

constexpr size_t kHead = (sizeof(SelShared) + 15) / 16 * 16;
// SelShared | key [kSelCap] | idx [kSelCap] | bitmap [kWinWords] | fbs [kFbMax] | wpre [kFbMax + 1]
constexpr size_t kSelSmem = kHead + 4 * (2 * static_cast<size_t>(kSelCap) + kWinWords + 2 * kFbMax + 1);
static_assert(kSelSmem <= 227u * 1024u, "select shared memory");

struct SelArgs {
    const int64_t* tok_off;
    const int64_t* tok_end;
    int64_t n_tokens;
    const float* scores;
    int k;
    const uint32_t* hist;
    float* theta_hat;
    float alpha;
    int32_t* sel;
    float* kth;
    // candidate lists (c_key null: none)
    const uint32_t* c_key;
    const int32_t* c_idx;
    const int32_t* c_cnt;
    uint32_t* c_cut;
    int c_cap;
    // cached form (sel_slot null: plain top-k)
    const uint32_t* above;
    int early_cap;
    int32_t* tok2slot;
    int32_t* slot2tok;
    const uint32_t* freebits;
    int32_t* early_cnt;
    int32_t* sel_slot;
    int C;
    int32_t* status;
    uint32_t* stats;
    // prefill rows (W > 0): row b at position row0 + b selects among scores[b * W + s],
    // s <= row0 + b, its histogram shifted by the block's one threshold theta_hat[0],
    // which the block's own EMA (not this kernel) updates
    int64_t row0;
    int64_t W;
};

// Warp 0: the key of the lower edge of the lowest histogram bin d with at most
// kCutMaxAbove tokens in bins >= d, moved back from the shifted scores (shift
// added) -- a cut that leaves at most about that many candidates.
__device__ uint32_t cut_from_hist(const uint32_t* h, float shift) {
    const int lane = threadIdx.x & 31;
    uint32_t c[8];
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        c[j] = h[8 * lane + j];
        sum += c[j];
    }
    uint32_t suf = sum;  // inclusive suffix over lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += y;
    }
    uint32_t acc = suf - sum;  // tokens in the bins above this lane's
    int d = 256;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
        acc += c[j];
        if (acc <= kCutMaxAbove) d = 8 * lane + j;
    }
    d = __reduce_min_sync(0xffffffffu, d);
    if (d <= 0) return 0u;  // every token
    if (d > 255) d = 255;
    return order_key(__fadd_rn(shift, key_to_float(static_cast<uint32_t>(d) << 24)));
}

// Appends the tokens of a warp for which `in` holds to the shared-memory list
// (order key of the score, index) while it has room; returns how many were in.
__device__ __forceinline__ uint32_t warp_gather(bool in, float x, int64_t s, uint32_t* cnt, uint32_t* ckey,
                                                uint32_t* cidx) {
    const int lane = threadIdx.x & 31;
    const unsigned m = __ballot_sync(0xffffffffu, in);
    if (m) {
        const int first = __ffs(m) - 1;
        uint32_t base = 0;
        if (lane == first) base = atomicAdd(cnt, static_cast<uint32_t>(__popc(m)));
        base = __shfl_sync(0xffffffffu, base, first);
        const uint32_t pos = base + __popc(m & ((1u << lane) - 1u));
        if (in && pos < static_cast<uint32_t>(kSelCap)) {
            ckey[pos] = order_key(x);
            cidx[pos] = static_cast<uint32_t>(s);
        }
    }
    return static_cast<uint32_t>(__popc(m));
}

__global__ void __launch_bounds__(kTT, 1) select_kernel(const SelArgs a) {
    pdl_launch_dependents();  // a programmatic dependent (the cache step) may start its table prologue
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SelShared& sh = *reinterpret_cast<SelShared*>(smem_raw);
    uint32_t* const ckey = reinterpret_cast<uint32_t*>(smem_raw + kHead);
    uint32_t* const cidx = ckey + kSelCap;
    uint32_t* const bm = cidx + kSelCap;
    uint32_t* const fbs = bm + kWinWords;
    uint32_t* const wpre = fbs + kFbMax;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    const bool rows = a.W > 0;
    int64_t lo, hi;
    bool range_ok;
    if (rows) {
        lo = static_cast<int64_t>(b) * a.W;
        hi = lo + a.row0 + b + 1;
        range_ok = a.row0 + b + 1 <= a.W;
        if (!range_ok) hi = lo;
    } else {
        range_ok = seg_bounds(a.tok_off, a.tok_end, a.n_tokens, b, &lo, &hi);
    }
    const int64_t n = hi - lo;
    const float* sc = a.scores + lo;
    const uint32_t k = static_cast<uint32_t>(a.k);
    int32_t* out = a.sel + static_cast<int64_t>(b) * a.k;
    const bool cached = a.sel_slot != nullptr;
    int32_t* out_slot = cached ? a.sel_slot + static_cast<int64_t>(b) * a.k : nullptr;
    const float th_old = a.theta_hat ? a.theta_hat[rows ? 0 : b] : __int_as_float(0x7f800000);
    const float shift = isfinite(th_old) ? th_old : 0.f;
    const int words = cached ? a.C / 32 : 0;
    int32_t* t2s = cached ? a.tok2slot + lo : nullptr;
    int32_t* s2t = cached ? a.slot2tok + static_cast<int64_t>(b) * a.C : nullptr;
    const uint32_t* ab = (cached && a.above && n > 0) ? a.above + 4 * (lo / 128 + b) : nullptr;
    if (tid == 0) {
        sh.flag = range_ok ? 0u : 1u;
        sh.nan = 0;
        sh.cnt = 0;
        sh.n_above = 0;
        sh.minkey = 0xFFFFFFFFu;
        sh.used = 0;
        sh.cut = kNoCut;
        if (!range_ok) set_status(a.status, ECHO_ST_BADDATA);
    }
    // the request's free bits and their prefix at the step's start (cached form)
    uint32_t limit = 0;
    if (cached) {
        const uint32_t F0 = free_prefix<kTT>(a.freebits + static_cast<int64_t>(b) * words, words, sh.scan, wpre, fbs);
        limit = ab ? ((a.early_cap < 0) ? F0 : min(F0, static_cast<uint32_t>(a.early_cap))) : 0u;
    }
    __syncthreads();

    if (n == 0) {
        for (int i = tid; i < a.k; i += kTT) {
            out[i] = -1;
            if (out_slot) out_slot[i] = -1;
        }
        if (tid == 0) {
            a.kth[b] = __int_as_float(0xff800000);
            if (cached) a.early_cnt[b] = 0;
            if (a.c_cut) a.c_cut[b] = kNoCut;
        }
        return;
    }

    enum { kAll, kList, kScan };
    int mode = kScan;
    uint32_t K = 0, idx_cut = 0xFFFFFFFFu, ncand = 0;
    bool marked = false;   // the bitmap (single window) already holds the tokens above b*
    const bool single = n <= kWinTokens;
    const uint32_t cut_in = a.c_key ? a.c_cut[b] : kNoCut;
    const uint32_t rc = static_cast<uint32_t>(min(static_cast<int64_t>(kCutRank) * k, n));   // next cut's rank
    if (n <= static_cast<int64_t>(k)) {
        mode = kAll;
    } else if (cut_in != kNoCut) {
        const int32_t cc = a.c_cnt[b];
        if (cc >= static_cast<int32_t>(k) && cc <= min(a.c_cap, kSelCap)) {
            ncand = static_cast<uint32_t>(cc);
            const uint32_t* gk = a.c_key + static_cast<int64_t>(b) * a.c_cap;
            const int32_t* gi = a.c_idx + static_cast<int64_t>(b) * a.c_cap;
            bool bad = false;
            constexpr int U = 4;   // entries per thread in flight
            for (uint32_t i0 = 0; i0 < ncand; i0 += kTT * U) {
                uint32_t kv[U];
                int32_t iv[U];
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    const uint32_t i = i0 + j * kTT + tid;
                    kv[j] = i < ncand ? __ldcg(gk + i) : 0u;
                    iv[j] = i < ncand ? __ldcg(gi + i) : 0;
                }
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    const uint32_t i = i0 + j * kTT + tid;
                    if (i < ncand) {
                        bad |= iv[j] < 0 || iv[j] >= n || kv[j] < cut_in;
                        ckey[i] = kv[j];
                        cidx[i] = static_cast<uint32_t>(iv[j]);
                    }
                }
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&sh.flag, 2u);
            __syncthreads();
            mode = (sh.flag & 2u) ? kScan : kList;
            if (mode == kScan && tid == 0) set_status(a.status, ECHO_ST_BADDATA);
        }
    }

    if (mode == kAll) {
        // every token: the k-th score is the smallest
        uint32_t mk = 0xFFFFFFFFu;
        bool nan = false;
        scan_scores(sc, n, [&](float x, int64_t, bool ok) {
            if (ok) {
                nan |= isnan(x);
                mk = min(mk, order_key(x));
            }
        });
        mk = __reduce_min_sync(0xffffffffu, mk);
        if (lane == 0) atomicMin(&sh.minkey, mk);
        if (nan) sh.nan = 1;
        __syncthreads();
        K = sh.minkey;
    } else if (mode == kList) {
        uint32_t rem, eq;
        K = radix_select(SmemCands{ckey, cidx, ncand, false, 0u}, k, sh, &rem, &eq);
        if (rem < eq) {
            uint32_t r2, e2;
            idx_cut = ~radix_select(SmemCands{ckey, cidx, ncand, true, K}, rem, sh, &r2, &e2);
        }
        // the next cut: unchanged while the list holds between 3k and 6k tokens; a longer list
        // is cut at its rank-4k key; a shorter one is lowered by the histogram when that leaves
        // more tokens above it
        if (ncand > kCutHigh * k) {
            uint32_t r3, e3;
            const uint32_t c = radix_select(SmemCands{ckey, cidx, ncand, false, 0u}, rc, sh, &r3, &e3);
            if (tid == 0) sh.cut = c;
        } else if (ncand < kCutLow * k && a.hist) {
            if (tid < 256) sh.hist[tid] = a.hist[static_cast<int64_t>(b) * 256 + tid];
            __syncthreads();
            if (tid < 32) {
                const uint32_t c = cut_from_hist(sh.hist, shift);
                if (tid == 0) sh.cut = min(c, cut_in);
            }
        } else if (tid == 0) {
            sh.cut = cut_in;
        }
    } else {
        // ---- from all the scores: boundary bin, the tokens above it, its entries
        bool have = a.hist != nullptr;
        uint32_t bstar = 0, above = 0, d_rc = 0, above_rc = 0;
        for (int attempt = 0; attempt < 2; ++attempt) {
            if (have) {
                if (tid < 256) sh.hist[tid] = a.hist[static_cast<int64_t>(b) * 256 + tid];
            } else {
                if (tid < 256) sh.hist[tid] = 0u;
                __syncthreads();
                scan_scores(sc, n, [&](float x, int64_t, bool ok) {
                    const uint32_t d = ok ? shifted_bin(x, shift) : 0x100u;
                    const unsigned peers = __match_any_sync(0xffffffffu, d);
                    if (ok && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[d], static_cast<uint32_t>(__popc(peers)));
                });
            }
            __syncthreads();
            if (tid < 32) {
                find_digit(sh.hist, k, &sh.digit, &sh.above);
                find_digit(sh.hist, rc, &sh.digit2, &sh.above2);   // the bin of the next cut's rank
            }
            if (tid == 0) {
                sh.cnt = 0;
                sh.n_above = 0;
            }
            __syncthreads();
            bstar = sh.digit;
            above = sh.above;
            d_rc = sh.digit2;
            above_rc = sh.above2;
            const uint32_t eq_total = sh.hist[bstar];
            uint32_t my_above = 0;
            bool nan = false;
            scan_scores(sc, n, [&](float x, int64_t s, bool ok) {
                nan |= ok && isnan(x);
                const uint32_t bin = shifted_bin(x, shift);
                const bool up = ok && bin > bstar;
                const unsigned um = __ballot_sync(0xffffffffu, up);
                my_above += up ? 1u : 0u;
                if (single && lane == 0 && s < n) bm[s >> 5] = um;
                warp_gather(ok && bin == bstar, x, s, &sh.cnt, ckey, cidx);
            });
            my_above = __reduce_add_sync(0xffffffffu, my_above);
            if (lane == 0 && my_above) atomicAdd(&sh.n_above, my_above);
            if (nan) sh.nan = 1;
            __syncthreads();
            if (sh.n_above == above && sh.cnt == eq_total) break;
            // the histogram given does not describe these scores: count them here
            if (tid == 0) set_status(a.status, ECHO_ST_BADDATA);
            have = false;
            __syncthreads();  // every thread has read the counts before they are reset
        }
        ncand = sh.cnt;
        const uint32_t bin_cnt = ncand;
        const bool fits = ncand <= static_cast<uint32_t>(kSelCap);
        const uint32_t need = k - above;  // >= 1
        bool deep = false;                // selected by passes over the scores
        if (fits) {
            uint32_t rem, eq;
            K = radix_select(SmemCands{ckey, cidx, ncand, false, 0u}, need, sh, &rem, &eq);
            if (rem < eq) {
                uint32_t r2, e2;
                idx_cut = ~radix_select(SmemCands{ckey, cidx, ncand, true, K}, rem, sh, &r2, &e2);
            }
        } else {
            // the bin does not fit: a second round of 256 bins over the next 8 bits of its
            // shifted keys, then the sub-bin that holds the need-th token is gathered
            __syncthreads();
            if (tid < 256) sh.hist[tid] = 0u;
            if (tid == 0) sh.cnt = 0;
            __syncthreads();
            scan_scores(sc, n, [&](float x, int64_t, bool ok) {
                const uint32_t sk = shifted_key(x, shift);
                const bool in = ok && (sk >> 24) == bstar;
                const uint32_t d = in ? ((sk >> 16) & 255u) : 0x100u;
                const unsigned peers = __match_any_sync(0xffffffffu, d);
                if (in && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[d], static_cast<uint32_t>(__popc(peers)));
            });
            __syncthreads();
            if (tid < 32) find_digit(sh.hist, need, &sh.digit, &sh.above);
            __syncthreads();
            const uint32_t sub = (bstar << 8) | sh.digit;
            const uint32_t need2 = need - sh.above;
            scan_scores(sc, n, [&](float x, int64_t s, bool ok) {
                warp_gather(ok && (shifted_key(x, shift) >> 16) == sub, x, s, &sh.cnt, ckey, cidx);
            });
            __syncthreads();
            const uint32_t n2 = sh.cnt;
            if (n2 <= static_cast<uint32_t>(kSelCap)) {
                uint32_t rem, eq;
                K = radix_select(SmemCands{ckey, cidx, n2, false, 0u}, need2, sh, &rem, &eq);
                if (rem < eq) {
                    uint32_t r2, e2;
                    idx_cut = ~radix_select(SmemCands{ckey, cidx, n2, true, K}, rem, sh, &r2, &e2);
                }
            } else {
                deep = true;   // (many equal scores) radix passes over the sub-bin's scores
                K = scan_select(sc, n, shift, sub, 16, need2, sh, &idx_cut);
            }
            ncand = 0;   // the gathered entries are not the boundary bin: mark from the scores
        }
        if (tid == 0 && a.stats) {
            atomicMax(a.stats + ECHO_STAT_BOUNDARY_MAX, bin_cnt);
            if (deep) atomicAdd(a.stats + ECHO_STAT_TOPK_FALLBACK, 1u);
            if (cut_in != kNoCut) atomicAdd(a.stats + ECHO_STAT_CAND_MISS, 1u);
        }
        // the next cut: the key of rank 4k, exactly (in the gathered bin, or by radix passes
        // over the scores of the bin that holds it)
        if (a.c_cut) {
            uint32_t c;
            if (fits && d_rc == bstar) {
                uint32_t r3, e3;
                c = radix_select(SmemCands{ckey, cidx, ncand, false, 0u}, rc - above, sh, &r3, &e3);
            } else {
                c = scan_select(sc, n, shift, d_rc, 8, rc - above_rc, sh, static_cast<uint32_t*>(nullptr));
            }
            if (tid == 0) sh.cut = c;
        }
        marked = single && fits;
    }
    __syncthreads();

    // ---- ordered write, one bitmap window (2^19 tokens) at a time
    uint32_t run_sel = 0, run_ab = 0, used = 0;
    bool bad = false;
    for (int64_t w0 = 0; w0 < n; w0 += kWinTokens) {
        const int64_t wn = min(kWinTokens, n - w0);
        const int Ww = static_cast<int>((wn + 31) >> 5);
        // the window's selected tokens into the bitmap
        if (mode == kAll) {
            for (int w = tid; w < Ww; w += kTT) {
                const int64_t t0 = w0 + 32 * static_cast<int64_t>(w);
                bm[w] = (n - t0 >= 32) ? 0xFFFFFFFFu : ((1u << (n - t0)) - 1u);
            }
        } else if (mode == kList || marked) {
            if (mode == kList)
                for (int w = tid; w < Ww; w += kTT) bm[w] = 0u;
            __syncthreads();
            for (uint32_t i = tid; i < ncand; i += kTT) {
                const uint32_t key = ckey[i], s = cidx[i];
                if (static_cast<int64_t>(s) < w0 || static_cast<int64_t>(s) >= w0 + wn) continue;
                if (key > K || (key == K && s <= idx_cut)) {
                    const uint32_t r = static_cast<uint32_t>(s - w0);
                    atomicOr(&bm[r >> 5], 1u << (r & 31));
                }
            }
        } else {
            // from the scores: selected <=> key > K, or key == K and index <= the cut
            scan_scores(sc + w0, wn, [&](float x, int64_t s, bool ok) {
                bool t = false;
                if (ok) {
                    const uint32_t key = order_key(x);
                    t = key > K || (key == K && static_cast<uint32_t>(w0 + s) <= idx_cut);
                }
                const unsigned m = __ballot_sync(0xffffffffu, t);
                if (lane == 0 && s < wn) bm[s >> 5] = m;
            });
        }
        __syncthreads();
        // this thread's words [wa, wb): counts, then the block's prefixes
        const int cw = (Ww + kTT - 1) / kTT;
        const int wa = min(tid * cw, Ww), wb = min(wa + cw, Ww);
        const int64_t aw0 = w0 >> 5;
        uint32_t cs = 0, ca = 0;
        for (int w = wa; w < wb; ++w) {
            cs += __popc(bm[w]);
            if (ab) ca += __popc(__ldcg(ab + aw0 + w));
        }
        uint32_t ts, ta = 0;
        uint32_t pos = run_sel + block_exclusive_scan<kTT>(cs, sh.scan, &ts);
        uint32_t ar = run_ab;
        if (ab) ar += block_exclusive_scan<kTT>(ca, sh.scan, &ta);
        FreeWalk walk;
        bool walking = false;
        uint32_t wr = 0;   // rank of the free slot the walk gives next
        for (int w = wa; w < wb; ++w) {
            const uint32_t sm = bm[w];
            const uint32_t am = ab ? __ldcg(ab + aw0 + w) : 0u;
            uint32_t all = sm | am;
            while (all) {
                const int j = __ffs(all) - 1;
                all &= all - 1;
                const int64_t s = w0 + 32 * static_cast<int64_t>(w) + j;
                const bool is_sel = (sm >> j) & 1u;
                int32_t slot = -1;
                if (cached && is_sel) slot = t2s[s];
                if ((am >> j) & 1u) {
                    const uint32_t r = ar++;
                    if (is_sel && slot < 0 && r < limit) {
                        // the token is in the early set: the rank-th free slot
                        if (!walking) {
                            walk.init(wpre, fbs, words, r);
                            walking = true;
                            wr = r;
                        }
                        while (wr < r) {
                            walk.next();
                            ++wr;
                        }
                        const int fs = walk.next();
                        ++wr;
                        if (fs >= 0) {
                            slot = fs;
                            t2s[s] = fs;
                            s2t[fs] = static_cast<int32_t>(s);
                            ++used;
                        } else {
                            bad = true;
                        }
                    }
                }
                if (is_sel) {
                    if (pos < k) {
                        out[pos] = static_cast<int32_t>(s);
                        if (out_slot) out_slot[pos] = slot;
                    }
                    ++pos;
                }
            }
        }
        run_sel += ts;
        run_ab += ta;
        __syncthreads();  // the bitmap is rebuilt for the next window
    }
    for (uint32_t i = min(run_sel, k) + tid; i < k; i += kTT) {
        out[i] = -1;
        if (out_slot) out_slot[i] = -1;
    }
    used = __reduce_add_sync(0xffffffffu, used);
    if (lane == 0 && used) atomicAdd(&sh.used, used);
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&sh.flag, 4u);
    __syncthreads();
    if (tid == 0) {
        const uint32_t want = (mode == kAll) ? static_cast<uint32_t>(n) : k;
        int st = 0;
        if (run_sel != want || (sh.flag & 4u)) st |= ECHO_ST_BADDATA;
        if (sh.nan) st |= ECHO_ST_NAN;
        if (st) set_status(a.status, st);
        const float kth = key_to_float(K);
        a.kth[b] = kth;
        if (a.theta_hat && !rows) a.theta_hat[b] = ema_update(th_old, kth, a.alpha);
        if (a.c_cut) a.c_cut[b] = (mode == kAll) ? kNoCut : sh.cut;
        if (cached) {
            const uint32_t E = ab ? min(run_ab, limit) : 0u;
            a.early_cnt[b] = static_cast<int32_t>(E);
            if (a.stats && E) atomicAdd(a.stats + ECHO_STAT_EARLY, E);
            if (a.stats && sh.used) atomicAdd(a.stats + ECHO_STAT_EARLY_USED, sh.used);
        }
    }
}

}  // namespace

int launch_select_rows(int R, int64_t row0, int64_t W, const float* scores, int k, const uint32_t* hist,
                       float* theta_hat, int32_t* sel_idx, float* kth, int32_t* status, uint32_t* stats,
                       cudaStream_t stream) {
    SelArgs a{};
    a.scores = scores;
    a.k = k;
    a.hist = hist;
    a.theta_hat = theta_hat;
    a.sel = sel_idx;
    a.kth = kth;
    a.status = status;
    a.stats = stats;
    a.early_cap = 0;
    a.row0 = row0;
    a.W = W;
    ECHO_CUDA_OK(prefer_max_shared(select_kernel));
    ECHO_CUDA_OK(cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kSelSmem)));
    select_kernel<<<R, kTT, kSelSmem, stream>>>(a);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}

}  // namespace echo

extern "C" int echo_topk_select_cands(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                                      const float* scores, int k, const uint32_t* hist, float* theta_hat, float alpha,
                                      const echo_cands* cands, int32_t* sel_idx, float* kth, const uint32_t* above,
                                      int early_cap, const echo_cache* cache, int32_t* sel_slot, int32_t* status,
                                      uint32_t* stats, echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || n_tokens < 0 || k <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !sel_idx || !kth || !status || (n_tokens > 0 && !scores)) return ECHO_EINVAL;
    if (n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    if (cands && (!cands->key || !cands->idx || !cands->cnt || !cands->cut || cands->cap <= 0)) return ECHO_EINVAL;
    if (cache) {
        if (!sel_slot) return ECHO_EINVAL;
        const int rc = check_cache(cache, B, k);
        if (rc) return rc;
        if (cache->C / 32 > kFbMax) return ECHO_EUNSUPPORTED;
    }
    SelArgs a{tok_off, tok_end, n_tokens, scores, k, hist, theta_hat, alpha, sel_idx, kth,
              cands ? cands->key : nullptr, cands ? cands->idx : nullptr, cands ? cands->cnt : nullptr,
              cands ? cands->cut : nullptr, cands ? cands->cap : 0,
              cache ? above : nullptr, early_cap, cache ? cache->tok2slot : nullptr,
              cache ? cache->slot2tok : nullptr, cache ? cache->freebits : nullptr,
              cache ? cache->early_cnt : nullptr, cache ? sel_slot : nullptr, cache ? cache->C : 0, status, stats};
    ECHO_CUDA_OK(prefer_max_shared(select_kernel));
    ECHO_CUDA_OK(cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kSelSmem)));
    select_kernel<<<B, kTT, kSelSmem, static_cast<cudaStream_t>(stream)>>>(a);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}
