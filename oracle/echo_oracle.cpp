/*
 * echo_oracle.cpp -- plain CPU oracle for the ECHO per-layer decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the bench's CPU
 * baseline leg are the only code that loads this library.  The CUDA library
 * never includes, links or calls it, and it shares no header, helper, table or
 * constant with the CUDA sources.  It is written for a reader who checks it
 * against the sources below by eye: every step is the definition, in fp64
 * where the step is arithmetic, with no blocking, fusion or reordering.
 *
 * Sources (page title, then section):
 *   [EXPL] "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs"
 *          (interactive explainer page), section 2 "The top-k dependency",
 *          sub-panels "Five fixed-size integer tensors on the GPU",
 *          "One layer, one step: free -> allocate -> recall",
 *          "Decode: fetch above a predicted threshold",
 *          "Prefill: one-round histogram".
 *   [AE]   "OSDI'26 Artifact Evaluation for ECHO: Efficient KV Cache Offloading
 *          with Lossless Prefetching for Serving Native Sparse Attention LLMs",
 *          sections "Download the model" (DeepSeek-V3.2) and "Baselines under
 *          evaluation" (bounded GPU cache NSA_DEV_CACHE_SIZE).
 *   [OCP]  OCP 8-bit Floating Point Specification (OFP8), format E4M3.
 *   [IDX]  The DeepSeek-V3.2 lightning-indexer score this library computes:
 *          I[s] = sum_h w[h] * ReLU(q[h] . k[s]), 64 heads x 128 dims, FP8
 *          keys with one fp32 scale per token.
 *
 * Readings where the sources are silent are marked READING and listed with
 * their reasons in the design notes of the repository.
 *
 * Return codes of the int-valued functions: 0 ok, 1 bad argument, 2 capacity
 * (k > C or cache full), 3 NaN/Inf met.
 *
 * Build: g++ -O2 -std=c++17 -shared -fPIC -ffp-contract=off -pthread.
 * -ffp-contract=off matters: the fp32 EMA below must round every product
 * and sum separately, as written.
 */
#include <algorithm>
#include <cmath>
#include <limits>
#include <cstdint>
#include <cstring>
#include <map>
#include <set>
#include <thread>
#include <vector>

namespace {

constexpr int ORC_OK = 0;
constexpr int ORC_EINVAL = 1;
constexpr int ORC_ECAPACITY = 2;
constexpr int ORC_ENAN = 3;

// ---------------------------------------------------------------------------
// [OCP] E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
// Exponent field 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there is
// no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448.
// ---------------------------------------------------------------------------
double e4m3_value(uint8_t code) {
    const int sign = code >> 7;
    const int e = (code >> 3) & 0xF;
    const int m = code & 0x7;
    if (e == 15 && m == 7) return std::nan("");
    double mag;
    if (e == 0)
        mag = std::ldexp(m / 8.0, -6);
    else
        mag = std::ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

// Round-to-nearest-even onto the E4M3 grid, saturating to +-448 (the
// behaviour of a "satfinite" conversion).  Plain search: the positive codes
// 0..126 are in ascending order of value, so a binary search finds the two
// neighbours of |x|; the nearer wins, and an exact tie goes to the even code
// (the code whose mantissa LSB is 0).
uint8_t e4m3_round(double x) {
    if (std::isnan(x)) return 0x7F;
    const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
    const double a = std::fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    int lo = 0, hi = 126;  // invariant: value(lo) <= a
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (e4m3_value((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    const double vlo = e4m3_value((uint8_t)lo);
    if (vlo == a) return sign | (uint8_t)lo;
    const double vhi = e4m3_value((uint8_t)(lo + 1));
    const double dlo = a - vlo, dhi = vhi - a;
    int c;
    if (dlo < dhi)
        c = lo;
    else if (dhi < dlo)
        c = lo + 1;
    else
        c = (lo % 2 == 0) ? lo : lo + 1;
    return sign | (uint8_t)c;
}

bool finite_f(float x) { return std::isfinite(x); }

uint32_t f32_bits(float x) {
    uint32_t u;
    std::memcpy(&u, &x, 4);
    return u;
}

float bits_f32(uint32_t u) {
    float x;
    std::memcpy(&x, &u, 4);
    return x;
}

// A key on which unsigned comparison orders floats: larger float, larger key.
// -0 is first made +0 so that the two zeros compare equal (READING: the pages
// do not say how signed zeros rank; they are equal scores).
uint32_t order_key(float x) {
    if (x == 0.0f) x = 0.0f;
    const uint32_t u = f32_bits(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// Query quantisation (READING; the sources say only that the score GEMM runs
// in FP8): one power-of-two scale per (request, head), the smallest 2^e with
// amax <= 448 * 2^e, with e held at or above -126 so that 2^e is a normal
// float; amax == 0 gives scale 1.  Dividing by a power of two is exact, so
// q / scale is rounded once, onto the E4M3 grid, without saturating.
// ---------------------------------------------------------------------------
int q_scale_exponent(float amax) {
    if (amax == 0.0f) return 0;
    int e = -126;
    while ((double)amax > std::ldexp(448.0, e)) ++e;
    return e;
}

// ---------------------------------------------------------------------------
// Exact top-k of one score vector [EXPL "guarantees an exact top-k"]:
// stable sort of indices by score, descending, so equal scores keep the lower
// index first; take min(k, n); report them in ascending index order
// (READING: the output order is not stated), padded with -1.
// kth = the score of the k-th element of the sorted order, or of the last
// selected one when n < k (READING).  -INFINITY when n == 0.
// ---------------------------------------------------------------------------
int topk_one(const float* scores, int64_t n, int k, int32_t* idx, float* kth) {
    std::vector<int32_t> order((size_t)n);
    for (int64_t i = 0; i < n; ++i) {
        if (std::isnan(scores[i])) return ORC_ENAN;
        order[(size_t)i] = (int32_t)i;
    }
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
        return order_key(scores[a]) > order_key(scores[b]);
    });
    const int64_t take = std::min<int64_t>(k, n);
    std::vector<int32_t> chosen(order.begin(), order.begin() + take);
    std::sort(chosen.begin(), chosen.end());
    for (int i = 0; i < k; ++i) idx[i] = (i < take) ? chosen[(size_t)i] : -1;
    if (take == 0) {
        *kth = -INFINITY;
    } else {
        float v = scores[order[(size_t)(take - 1)]];
        if (v == 0.0f) v = 0.0f;
        *kth = v;
    }
    return ORC_OK;
}

// [EXPL "Decode: fetch above a predicted threshold"]: the predicted threshold
// is an EMA, weight alpha = 0.5, of the previous step's k-th score.
// theta_next = alpha * kth + (1 - alpha) * theta, each operation rounded in
// fp32.  READING: the first step has no prediction (theta = +inf, so nothing
// is fetched early) and the first k-th score replaces it instead of being
// averaged with +inf.  A request with no tokens (kth = -inf) keeps theta.
float ema(float theta, float kth, float alpha) {
    if (std::isinf(kth) && kth < 0) return theta;
    if (std::isinf(theta)) return kth;
    const float one_minus = 1.0f - alpha;
    const float a = alpha * kth;
    const float b = one_minus * theta;
    return a + b;
}

// ---------------------------------------------------------------------------
// One segment's GPU cache, held as the ordered containers the definition
// talks about: a token -> slot map and the set of free slots.
// ---------------------------------------------------------------------------
struct Cache {
    std::map<int32_t, int32_t> resident;  // token -> slot
    std::set<int32_t> free_slots;         // ascending
};

Cache load_cache(int64_t n, int C, const int32_t* tok2slot, const int32_t* slot2tok) {
    Cache c;
    for (int64_t s = 0; s < n; ++s)
        if (tok2slot[s] >= 0) c.resident[(int32_t)s] = tok2slot[s];
    for (int j = 0; j < C; ++j)
        if (slot2tok[j] < 0) c.free_slots.insert(j);
    return c;
}

void store_cache(const Cache& c, int64_t n, int C, int32_t* tok2slot, int32_t* slot2tok) {
    for (int64_t s = 0; s < n; ++s) tok2slot[s] = -1;
    for (int j = 0; j < C; ++j) slot2tok[j] = -1;
    for (const auto& kv : c.resident) {
        tok2slot[kv.first] = kv.second;
        slot2tok[kv.second] = kv.first;
    }
}

// Slot tables must be mutual inverses; anything else is a bad argument.
bool cache_consistent(int64_t n, int C, const int32_t* tok2slot, const int32_t* slot2tok) {
    for (int64_t s = 0; s < n; ++s) {
        const int32_t j = tok2slot[s];
        if (j < -1 || j >= C) return false;
        if (j >= 0 && slot2tok[j] != s) return false;
    }
    for (int j = 0; j < C; ++j) {
        const int32_t s = slot2tok[j];
        if (s < -1 || s >= n) return false;
        if (s >= 0 && tok2slot[s] != j) return false;
    }
    return true;
}

}  // namespace

extern "C" {

// ---- [OCP] E4M3 codec -----------------------------------------------------
double orc_e4m3_decode(uint8_t code) { return e4m3_value(code); }
uint8_t orc_e4m3_encode(double x) { return e4m3_round(x); }

void orc_e4m3_encode_f32(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_round((double)x[i]);
}

uint32_t orc_order_key(float x) { return order_key(x); }

// ---- query quantisation (READING above) -----------------------------------
// q [B,H,D] f32, w [B,H] f32 -> q8 [B,H,D] E4M3 bytes, qscale [B,H] f32 (the
// power of two), wfold [B,H] f32 = w * qscale rounded in fp32 (what a scaled
// kernel multiplies by; the oracle's score below does not use it).
int orc_quantize_q(const float* q, const float* w, int B, int H, int D, uint8_t* q8,
                   float* qscale, float* wfold) {
    if (B < 0 || H <= 0 || D <= 0) return ORC_EINVAL;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const float* row = q + ((int64_t)b * H + h) * D;
            float amax = 0.0f;
            for (int d = 0; d < D; ++d) {
                if (!finite_f(row[d])) return ORC_ENAN;
                amax = std::max(amax, std::fabs(row[d]));
            }
            if (!finite_f(w[(int64_t)b * H + h])) return ORC_ENAN;
            const int e = q_scale_exponent(amax);
            const double scale = std::ldexp(1.0, e);
            for (int d = 0; d < D; ++d)
                q8[((int64_t)b * H + h) * D + d] = e4m3_round((double)row[d] / scale);
            qscale[(int64_t)b * H + h] = (float)scale;
            wfold[(int64_t)b * H + h] = (float)((double)w[(int64_t)b * H + h] * scale);
        }
    return ORC_OK;
}

// ---- [IDX] indexer score, fp64, direct form ------------------------------
// out[s] = sum_h w[h] * max(0, sum_d (dec(q8[h,d]) * qscale[h]) * (dec(k8[s,d]) * ks[s]))
// absb[s] = sum_h |w[h]| * sum_d |dec(q8[h,d]) * qscale[h] * dec(k8[s,d]) * ks[s]|,
// the size of the terms, which bounds the rounding a reordered sum may make.
// Tokens are the rows tok[0..n) of k8 [*,D] and ks; tok == NULL means 0..n-1.
void orc_scores(const uint8_t* q8, const float* qscale, const float* w, int H, int D,
                const uint8_t* k8, const float* ks, const int64_t* tok, int64_t n,
                double* out, double* absb) {
    std::vector<double> qv((size_t)H * D);
    for (int h = 0; h < H; ++h)
        for (int d = 0; d < D; ++d)
            qv[(size_t)h * D + d] = e4m3_value(q8[(int64_t)h * D + d]) * (double)qscale[h];
    std::vector<double> kv((size_t)D);
    for (int64_t i = 0; i < n; ++i) {
        const int64_t s = tok ? tok[i] : i;
        for (int d = 0; d < D; ++d) kv[(size_t)d] = e4m3_value(k8[s * D + d]) * (double)ks[s];
        double total = 0.0, bound = 0.0;
        for (int h = 0; h < H; ++h) {
            double dot = 0.0, dabs = 0.0;
            for (int d = 0; d < D; ++d) {
                const double p = qv[(size_t)h * D + d] * kv[(size_t)d];
                dot += p;
                dabs += std::fabs(p);
            }
            total += (double)w[h] * std::max(0.0, dot);
            bound += std::fabs((double)w[h]) * dabs;
        }
        out[i] = total;
        if (absb) absb[i] = bound;
    }
}

// ---- [EXPL "Prefill: one-round histogram"] --------------------------------
// 256 bins over the top 8 bits of each score shifted by the predicted
// threshold: bin = order_key(fp32(score - shift)) >> 24, one fp32 subtraction
// rounded to nearest.  shift is the threshold when it is finite, else 0
// (READING: with no prediction yet the scores are binned unshifted).
void orc_hist256(const float* scores, int64_t n, float theta, uint32_t* hist) {
    const float shift = std::isfinite(theta) ? theta : 0.0f;
    for (int i = 0; i < 256; ++i) hist[i] = 0;
    for (int64_t s = 0; s < n; ++s) {
        float x = scores[s];
        if (x == 0.0f) x = 0.0f;
        const float d = x - shift;
        hist[order_key(d) >> 24] += 1;
    }
}

// ---- exact top-k ----------------------------------------------------------
int orc_topk(const float* scores, int64_t n, int k, int32_t* idx, float* kth) {
    if (n < 0 || k <= 0) return ORC_EINVAL;
    return topk_one(scores, n, k, idx, kth);
}

float orc_ema(float theta, float kth, float alpha) { return ema(theta, kth, alpha); }

// ---- [EXPL "Decode: fetch above a predicted threshold"] -------------------
// Before top-k is known, tokens that score strictly above the predicted
// threshold and are not resident are fetched early (READING: strict ">").
// They are taken in ascending token order, at most min(cap, F) of them, F the
// number of free slots when the step starts (READING: the page's early-fetch
// cap value did not survive; cap < 0 means "no cap beyond F").  They get the
// lowest free slots, in ascending order, and become resident at once.
// Outputs: early_tok / early_slot [count], *count.
int orc_early_fetch(int64_t n, int C, const float* scores, float theta, int cap,
                    int32_t* tok2slot, int32_t* slot2tok, int32_t* early_tok,
                    int32_t* early_slot, int32_t* count) {
    if (!cache_consistent(n, C, tok2slot, slot2tok)) return ORC_EINVAL;
    Cache c = load_cache(n, C, tok2slot, slot2tok);
    const int64_t F = (int64_t)c.free_slots.size();
    const int64_t limit = (cap < 0) ? F : std::min<int64_t>(cap, F);
    int32_t got = 0;
    for (int64_t s = 0; s < n && got < limit; ++s) {
        if (!(scores[s] > theta)) continue;
        if (c.resident.count((int32_t)s)) continue;
        const int32_t slot = *c.free_slots.begin();
        c.free_slots.erase(c.free_slots.begin());
        c.resident[(int32_t)s] = slot;
        early_tok[got] = (int32_t)s;
        early_slot[got] = slot;
        ++got;
    }
    *count = got;
    store_cache(c, n, C, tok2slot, slot2tok);
    return ORC_OK;
}

// ---- cross-layer early fetch ----------------------------------------------
// Page "ECHO Guide: KV Offloading for Native Sparse Attention", section "Intra-Query
// Prefetching: Layer-to-Layer Pipeline": the tokens that layer l selects are
// mostly selected by layers l+1 and l+2 too, so the ones not yet resident for
// layer l+1 are fetched as soon as layer l's selection is known.  READING: the
// early set of layer l+1 is then layer l's selection (prev_sel [m], -1
// padded, entries >= n ignored) minus layer l+1's residents, taken exactly as
// the threshold early fetch takes its marked tokens: ascending token order,
// at most min(cap, F) (F = free slots of layer l+1 at that moment), lowest
// free slots ascending, resident at once.  Outputs as orc_early_fetch.
int orc_early_from_selection(int64_t n, int C, const int32_t* prev_sel, int m, int cap, int32_t* tok2slot,
                             int32_t* slot2tok, int32_t* early_tok, int32_t* early_slot, int32_t* count) {
    if (!cache_consistent(n, C, tok2slot, slot2tok) || m < 0) return ORC_EINVAL;
    std::set<int32_t> marked;
    for (int i = 0; i < m; ++i)
        if (prev_sel[i] >= 0 && prev_sel[i] < n) marked.insert(prev_sel[i]);
    Cache c = load_cache(n, C, tok2slot, slot2tok);
    const int64_t F = (int64_t)c.free_slots.size();
    const int64_t limit = (cap < 0) ? F : std::min<int64_t>(cap, F);
    int32_t got = 0;
    for (int32_t s : marked) {  // ascending
        if (got >= limit) break;
        if (c.resident.count(s)) continue;
        const int32_t slot = *c.free_slots.begin();
        c.free_slots.erase(c.free_slots.begin());
        c.resident[s] = slot;
        early_tok[got] = s;
        early_slot[got] = slot;
        ++got;
    }
    *count = got;
    store_cache(c, n, C, tok2slot, slot2tok);
    return ORC_OK;
}

// ---- [EXPL "One layer, one step: free -> allocate -> recall"] -------------
// sel [m] is the step's selection in ascending token order, -1 padded.
// early_tok [n_early] are the tokens this step's early fetch made resident
// (orc_early_fetch's output; may be NULL when n_early = 0).
// 1. Free every resident token that is not selected: both table entries go
//    to -1; the KV bytes stay where they are and nothing is written back to
//    the host, which holds every token.  With hold_early, the slot of an
//    early token of this step is held until step 2 is done (a variant, not
//    the contract reading: the early copy into that slot may still be in
//    flight during the step, so no miss of the same step is placed there;
//    the slot is free again for the next step).  Without it the early tokens
//    are residents like any other.
// 2. The selected tokens that are not resident are the misses; in ascending
//    token order each takes the lowest free slot, in ascending order.
// 3. The held slots are free.
// 4. sel_slot[i] = slot of sel[i] (-1 for padding).
// Outputs: miss_tok / miss_slot [*nmiss], *nfreed (held slots included).
// Capacity: selected tokens plus held slots must not exceed C (return 2,
// state untouched).
int orc_cache_step(int64_t n, int C, int32_t* tok2slot, int32_t* slot2tok, const int32_t* sel,
                   int m, const int32_t* early_tok, int32_t n_early, int hold_early, int32_t* sel_slot,
                   int32_t* miss_tok, int32_t* miss_slot, int32_t* nmiss, int32_t* nfreed) {
    if (!cache_consistent(n, C, tok2slot, slot2tok)) return ORC_EINVAL;
    if (n_early < 0 || (n_early > 0 && !early_tok)) return ORC_EINVAL;
    std::set<int32_t> selected;
    for (int i = 0; i < m; ++i) {
        if (sel[i] < 0) continue;
        if (sel[i] >= n) return ORC_EINVAL;
        selected.insert(sel[i]);
    }
    std::set<int32_t> early;
    if (hold_early) early.insert(early_tok, early_tok + n_early);
    int64_t held_count = 0;
    for (int32_t e : early)
        if (!selected.count(e)) ++held_count;
    if ((int64_t)selected.size() + held_count > C) return ORC_ECAPACITY;
    Cache c = load_cache(n, C, tok2slot, slot2tok);
    // 1. free (early slots held)
    int32_t freed = 0;
    std::vector<int32_t> held;
    for (auto it = c.resident.begin(); it != c.resident.end();) {
        if (!selected.count(it->first)) {
            if (early.count(it->first))
                held.push_back(it->second);
            else
                c.free_slots.insert(it->second);
            it = c.resident.erase(it);
            ++freed;
        } else {
            ++it;
        }
    }
    // 2. allocate, misses in ascending token order (std::set is ordered)
    int32_t got = 0;
    for (int32_t s : selected) {
        if (c.resident.count(s)) continue;
        const int32_t slot = *c.free_slots.begin();
        c.free_slots.erase(c.free_slots.begin());
        c.resident[s] = slot;
        miss_tok[got] = s;
        miss_slot[got] = slot;
        ++got;
    }
    // 3. the held slots are free again
    for (int32_t slot : held) c.free_slots.insert(slot);
    // 3. slot of every selected entry
    for (int i = 0; i < m; ++i) sel_slot[i] = (sel[i] < 0) ? -1 : c.resident.at(sel[i]);
    *nmiss = got;
    *nfreed = freed;
    store_cache(c, n, C, tok2slot, slot2tok);
    return ORC_OK;
}

}  // extern "C"

namespace {

// ---- lazy-reuse eviction (a variant of the cache step) ---------------------
// READING of the alternative to "resident == selected after every step"
// (freed slots keep their token until overwritten): a slot freed at a step keeps its bytes and both table entries until
// the slot is handed to another token.  Its token is then a ghost: present in
// the cache, not resident.  A selected ghost is a hit: it is resident in its
// slot again, with no copy.  Handing a slot to a token drops the ghost in it.
// Slots are handed out as in the contract: lowest free slot first.
// State: tok2slot / slot2tok are mutual inverses over the present tokens
// (resident or ghost); free_[j] = 1 when slot j holds no resident token (a
// ghost's slot is free).
struct LazyCache {
    std::map<int32_t, int32_t> present;  // token -> slot
    std::map<int32_t, int32_t> owner;    // slot -> token
    std::set<int32_t> free_slots;        // ascending
};

LazyCache load_lazy(int64_t n, int C, const int32_t* tok2slot, const int32_t* slot2tok, const uint8_t* free_) {
    LazyCache c;
    for (int64_t s = 0; s < n; ++s)
        if (tok2slot[s] >= 0) c.present[(int32_t)s] = tok2slot[s];
    for (int j = 0; j < C; ++j) {
        if (slot2tok[j] >= 0) c.owner[j] = slot2tok[j];
        if (free_[j]) c.free_slots.insert(j);
    }
    return c;
}

void store_lazy(const LazyCache& c, int64_t n, int C, int32_t* tok2slot, int32_t* slot2tok, uint8_t* free_) {
    for (int64_t s = 0; s < n; ++s) tok2slot[s] = -1;
    for (int j = 0; j < C; ++j) {
        slot2tok[j] = -1;
        free_[j] = 0;
    }
    for (const auto& kv : c.present) tok2slot[kv.first] = kv.second;
    for (const auto& kv : c.owner) slot2tok[kv.first] = kv.second;
    for (int32_t j : c.free_slots) free_[j] = 1;
}

// Hands slot j to token t: the ghost in j (if any) leaves the cache.
void lazy_take(LazyCache& c, int32_t j, int32_t t) {
    const auto o = c.owner.find(j);
    if (o != c.owner.end()) c.present.erase(o->second);
    c.owner[j] = t;
    c.present[t] = j;
    c.free_slots.erase(j);
}

}  // namespace

extern "C" {

// The early set under lazy reuse: tokens scoring strictly above theta that are
// not present (a ghost's bytes are already in the cache), ascending, at most
// min(cap, F) of them (F = free slots at the start, ghost slots included),
// with the lowest free slots ascending.  Only reports the pairs; the cache
// step takes them.
int orc_lazy_early(int64_t n, int C, const float* scores, float theta, int cap, const int32_t* tok2slot,
                   const int32_t* slot2tok, const uint8_t* free_, int32_t* early_tok, int32_t* early_slot,
                   int32_t* count) {
    if (!cache_consistent(n, C, tok2slot, slot2tok)) return ORC_EINVAL;
    const LazyCache c = load_lazy(n, C, tok2slot, slot2tok, free_);
    const int64_t F = (int64_t)c.free_slots.size();
    const int64_t limit = (cap < 0) ? F : std::min<int64_t>(cap, F);
    auto next = c.free_slots.begin();
    int32_t got = 0;
    for (int64_t s = 0; s < n && got < limit; ++s) {
        if (!(scores[s] > theta)) continue;
        if (c.present.count((int32_t)s)) continue;
        early_tok[got] = (int32_t)s;
        early_slot[got] = *next++;
        ++got;
    }
    *count = got;
    return ORC_OK;
}

// The cache step under lazy reuse.  sel [m] ascending, -1 padded; the early
// pairs as orc_lazy_early gave them.
//   0. each early token takes its slot (dropping the ghost there), resident.
//   1. every resident token that is not selected becomes a ghost (its slot
//      free, both table entries kept).
//   2. every selected token still present is resident (a ghost is revived in
//      its slot: its slot is no longer free).
//   3. the misses (selected, not present), ascending, take the lowest free
//      slots ascending, dropping the ghosts there.
//   4. sel_slot[i] = slot of sel[i] (-1 for padding).
// Outputs: miss_tok / miss_slot [*nmiss]; *nrevived = ghosts revived in step 2.
// Capacity: the selection must fit C (return 2, state untouched).
int orc_lazy_cache_step(int64_t n, int C, int32_t* tok2slot, int32_t* slot2tok, uint8_t* free_, const int32_t* sel,
                        int m, const int32_t* early_tok, const int32_t* early_slot, int32_t n_early,
                        int32_t* sel_slot, int32_t* miss_tok, int32_t* miss_slot, int32_t* nmiss,
                        int32_t* nrevived) {
    if (!cache_consistent(n, C, tok2slot, slot2tok)) return ORC_EINVAL;
    if (n_early < 0 || (n_early > 0 && (!early_tok || !early_slot))) return ORC_EINVAL;
    std::set<int32_t> selected;
    for (int i = 0; i < m; ++i) {
        if (sel[i] < 0) continue;
        if (sel[i] >= n) return ORC_EINVAL;
        selected.insert(sel[i]);
    }
    if ((int64_t)selected.size() > C) return ORC_ECAPACITY;
    LazyCache c = load_lazy(n, C, tok2slot, slot2tok, free_);
    for (int i = 0; i < n_early; ++i) {
        if (!c.free_slots.count(early_slot[i]) || c.present.count(early_tok[i])) return ORC_EINVAL;
        lazy_take(c, early_slot[i], early_tok[i]);
    }
    // 1. resident and unselected -> ghost
    for (const auto& kv : c.present)
        if (!c.free_slots.count(kv.second) && !selected.count(kv.first)) c.free_slots.insert(kv.second);
    // 2. selected and present -> resident
    int32_t revived = 0;
    for (int32_t t : selected) {
        const auto it = c.present.find(t);
        if (it == c.present.end()) continue;
        if (c.free_slots.erase(it->second)) ++revived;
    }
    // 3. the misses take the lowest free slots
    int32_t got = 0;
    for (int32_t t : selected) {
        if (c.present.count(t)) continue;
        const int32_t j = *c.free_slots.begin();
        lazy_take(c, j, t);
        miss_tok[got] = t;
        miss_slot[got] = j;
        ++got;
    }
    for (int i = 0; i < m; ++i) sel_slot[i] = (sel[i] < 0) ? -1 : c.present.at(sel[i]);
    *nmiss = got;
    *nrevived = revived;
    store_lazy(c, n, C, tok2slot, slot2tok, free_);
    return ORC_OK;
}

// ---- recall: the device copy of a row is the host row, byte for byte ------
void orc_recall(const uint8_t* host_rows, int64_t row_bytes, const int32_t* tok,
                const int32_t* slot, int32_t count, uint8_t* dev_rows) {
    for (int32_t i = 0; i < count; ++i)
        std::memcpy(dev_rows + (int64_t)slot[i] * row_bytes, host_rows + (int64_t)tok[i] * row_bytes,
                    (size_t)row_bytes);
}

// ---- append: one new token per request ------------------------------------
// EXPL section 2 ("One layer, one step"): the host holds every token, which is
// why eviction needs no write-back; the pages give no append mechanics.
// READING: request b's rows live in its region [tok_off[b], tok_off[b+1]) and
// tok_end[b] is its current end.  For each request with pos = tok_end[b]:
//   - no room (pos == tok_off[b+1]): nothing changes, full[b] = 1;
//   - the indexer key [IDX, FP8 keys with one fp32 scale per token]:
//     amax = max_d |k[d]|, ks = amax / 448 rounded in fp32, and
//     k8[d] = E4M3 round-to-nearest-even (saturating) of k[d] / ks rounded in
//     fp32 (both divisions in the precision the GPU takes them, since they
//     decide integer codes); amax = 0 gives ks = 0 and all-zero codes;
//   - the KV row goes to host row pos;
//   - the lowest free slot of the request, if any, takes the token (tok2slot,
//     slot2tok) and its device row gets the KV row; with none free the token
//     is host-only and will be recalled when selected;
//   - tok_end[b] = pos + 1.
// A non-finite key component returns 3 with nothing changed.
int orc_append_tokens(int B, const int64_t* tok_off, int64_t* tok_end, const float* k_new, int D,
                      const uint8_t* kv_new, int64_t row_bytes, uint8_t* k8, float* ks, uint8_t* host_rows, int C,
                      int32_t* tok2slot, int32_t* slot2tok, uint8_t* dev_rows, int32_t* full) {
    if (B < 0 || D <= 0 || C < 0 || row_bytes <= 0) return ORC_EINVAL;
    for (int b = 0; b < B; ++b) {
        if (tok_off[b] < 0 || tok_off[b + 1] < tok_off[b]) return ORC_EINVAL;
        if (tok_end[b] < tok_off[b] || tok_end[b] > tok_off[b + 1]) return ORC_EINVAL;
        for (int d = 0; d < D; ++d)
            if (!finite_f(k_new[(int64_t)b * D + d])) return ORC_ENAN;
    }
    for (int b = 0; b < B; ++b) {
        full[b] = 0;
        const int64_t pos = tok_end[b];
        if (pos == tok_off[b + 1]) {
            full[b] = 1;
            continue;
        }
        const float* k = k_new + (int64_t)b * D;
        float amax = 0.0f;
        for (int d = 0; d < D; ++d) amax = std::max(amax, std::fabs(k[d]));
        const float scale = amax / 448.0f;
        ks[pos] = scale;
        for (int d = 0; d < D; ++d) {
            if (amax == 0.0f) {
                k8[pos * D + d] = 0;
            } else {
                const float x = k[d] / scale;
                k8[pos * D + d] = e4m3_round((double)x);
            }
        }
        std::memcpy(host_rows + pos * row_bytes, kv_new + (int64_t)b * row_bytes, (size_t)row_bytes);
        for (int slot = 0; slot < C; ++slot) {
            if (slot2tok[(int64_t)b * C + slot] != -1) continue;
            slot2tok[(int64_t)b * C + slot] = (int32_t)(pos - tok_off[b]);
            tok2slot[pos] = slot;
            std::memcpy(dev_rows + ((int64_t)b * C + slot) * row_bytes, kv_new + (int64_t)b * row_bytes,
                        (size_t)row_bytes);
            break;
        }
        tok_end[b] = pos + 1;
    }
    return ORC_OK;
}

// ---- sparse MLA decode attention over the selected slots ------------------
// The consumer of the cache (EXPL section 2 names the sparse
// attention over the k selected tokens but gives no formula).  READING: MLA
// in its absorbed form, one latent KV row of 576 bf16 per token (512 latent
// + 64 rotary dims) shared by every query head; for head h over the valid
// slots t (slot >= 0):
//   s_t = scale * sum_{d<576} q[h,d] * kv[slot_t, d]
//   out[h, :] = sum_t softmax(s)_t * kv[slot_t, 0:512],  lse[h] = log sum_t exp(s_t)
// in fp64 (bf16 values are exact in fp64); no valid slot: out = 0,
// lse = -inf.  mass[h, d] = sum_t softmax(s)_t * |kv[slot_t, d]| (may be
// NULL) sizes the rounding a reordered or lower-precision sum may make.
double orc_bf16_value(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

int orc_mla_decode(const uint16_t* q, int H, const uint16_t* kv, int64_t rows, const int32_t* slots, int k,
                   double scale, double* out, double* lse, double* mass) {
    const int DQK = 576, DV = 512;
    if (H <= 0 || k < 0 || rows < 0) return ORC_EINVAL;
    for (int i = 0; i < k; ++i)
        if (slots[i] >= rows) return ORC_EINVAL;
    std::vector<double> sc((size_t)k);
    for (int h = 0; h < H; ++h) {
        double mx = -std::numeric_limits<double>::infinity();
        for (int i = 0; i < k; ++i) {
            if (slots[i] < 0) continue;
            double acc = 0.0;
            for (int d = 0; d < DQK; ++d)
                acc += orc_bf16_value(q[(int64_t)h * DQK + d]) * orc_bf16_value(kv[(int64_t)slots[i] * DQK + d]);
            sc[(size_t)i] = scale * acc;
            mx = std::max(mx, sc[(size_t)i]);
        }
        double* o = out + (int64_t)h * DV;
        double* ms = mass ? mass + (int64_t)h * DV : nullptr;
        for (int d = 0; d < DV; ++d) {
            o[d] = 0.0;
            if (ms) ms[d] = 0.0;
        }
        if (!(mx > -std::numeric_limits<double>::infinity())) {
            lse[h] = -std::numeric_limits<double>::infinity();
            continue;
        }
        double sum = 0.0;
        for (int i = 0; i < k; ++i)
            if (slots[i] >= 0) sum += std::exp(sc[(size_t)i] - mx);
        for (int i = 0; i < k; ++i) {
            if (slots[i] < 0) continue;
            const double p = std::exp(sc[(size_t)i] - mx) / sum;
            for (int d = 0; d < DV; ++d) {
                const double v = orc_bf16_value(kv[(int64_t)slots[i] * DQK + d]);
                o[d] += p * v;
                if (ms) ms[d] += p * std::fabs(v);
            }
        }
        lse[h] = mx + std::log(sum);
    }
    return ORC_OK;
}

// ---- [EXPL "Prefill: one-round histogram"] chunked-prefill block ----------
// Rows r = 0..R-1 of one query block sit at absolute positions p = row0 + r
// and see the causal prefix [0, p] (READING: the row's own token included).
// scores [R, W] (row stride W >= row0 + R) are the per-row scores; only
// entries [0, p] of row r are read.  Per row: exact top-k over [0, p]
// (everything when p + 1 <= k), ascending, -1 padded into sel [R, k], kth[r].
// hist [R, 256] (optional) is the per-row histogram of the shifted scores.
// union_mask [row0 + R] is set to 1 for every token selected by some row.
int orc_prefill_rows(const float* scores, int64_t W, int R, int64_t row0, int k, float theta,
                     int32_t* sel, float* kth, uint32_t* hist, uint8_t* union_mask) {
    if (R < 0 || row0 < 0 || k <= 0 || W < row0 + R) return ORC_EINVAL;
    std::memset(union_mask, 0, (size_t)(row0 + R));
    for (int r = 0; r < R; ++r) {
        const int64_t p = row0 + r;
        const float* row = scores + (int64_t)r * W;
        const int rc = topk_one(row, p + 1, k, sel + (int64_t)r * k, kth + r);
        if (rc) return rc;
        if (hist) orc_hist256(row, p + 1, theta, hist + (int64_t)r * 256);
        for (int i = 0; i < k; ++i)
            if (sel[(int64_t)r * k + i] >= 0) union_mask[sel[(int64_t)r * k + i]] = 1;
    }
    return ORC_OK;
}

// The early-set cap of the held-slot variant of a decode step with selection
// width k: C - k on top of the caller's cap (cap < 0: no cap of its own), so
// that selected tokens plus held slots stay within C.
int orc_early_cap_for(int cap, int C, int k) {
    const int room = C - k;
    return (cap < 0 || cap > room) ? room : cap;
}

// ---- one whole decode step of one layer, for the CPU baseline ------------
// Everything the GPU path does for B requests of one layer, in order, with
// the oracle's own fp64 scores rounded to fp32 feeding selection:
// quantise q, score, early fetch above theta (if predictor), exact top-k,
// EMA, cache step, recall of early and late misses.  Requests are split over
// nthreads std::threads.  State arrays are updated in place.
// tok_off [B+1]; q [B,H,D]; w [B,H]; k8 [tok_off[B], D]; ks; theta [B];
// tok2slot [tok_off[B]] (request-local slot); slot2tok [B*C] (request-local
// token); host_rows [tok_off[B], row_bytes]; dev_rows [B*C, row_bytes];
// sel_idx / sel_slot [B,k]; kth [B]; nmiss [B]; scores_out [tok_off[B]] or NULL.
int orc_decode_step(int B, const int64_t* tok_off, const float* q, const float* w, int H, int D,
                    const uint8_t* k8, const float* ks, int k, float alpha, int predictor, int cap,
                    float* theta, int C, int32_t* tok2slot, int32_t* slot2tok,
                    const uint8_t* host_rows, int64_t row_bytes, uint8_t* dev_rows,
                    int32_t* sel_idx, int32_t* sel_slot, float* kth, int32_t* nmiss,
                    float* scores_out, int nthreads) {
    if (B <= 0 || H <= 0 || D <= 0 || k <= 0 || k > C) return B <= 0 ? ORC_EINVAL : ORC_ECAPACITY;
    std::vector<int> rcs((size_t)B, ORC_OK);
    auto one = [&](int b) {
        const int64_t off = tok_off[b];
        const int64_t n = tok_off[b + 1] - off;
        std::vector<uint8_t> q8((size_t)H * D);
        std::vector<float> qs((size_t)H), wf((size_t)H);
        int rc = orc_quantize_q(q + (int64_t)b * H * D, w + (int64_t)b * H, 1, H, D, q8.data(),
                                qs.data(), wf.data());
        if (rc) { rcs[(size_t)b] = rc; return; }
        std::vector<double> sd((size_t)n);
        orc_scores(q8.data(), qs.data(), w + (int64_t)b * H, H, D, k8 + off * D, ks + off, nullptr,
                   n, sd.data(), nullptr);
        std::vector<float> sf((size_t)n);
        for (int64_t s = 0; s < n; ++s) sf[(size_t)s] = (float)sd[(size_t)s];
        if (scores_out) std::memcpy(scores_out + off, sf.data(), (size_t)n * 4);
        int32_t* t2s = tok2slot + off;
        int32_t* s2t = slot2tok + (int64_t)b * C;
        uint8_t* drows = dev_rows + (int64_t)b * C * row_bytes;
        const uint8_t* hrows = host_rows + off * row_bytes;
        std::vector<int32_t> et((size_t)C), es((size_t)C);
        int32_t ne = 0;
        if (predictor) {
            rc = orc_early_fetch(n, C, sf.data(), theta[b], cap, t2s, s2t, et.data(), es.data(), &ne);
            if (rc) { rcs[(size_t)b] = rc; return; }
            orc_recall(hrows, row_bytes, et.data(), es.data(), ne, drows);
        }
        rc = topk_one(sf.data(), n, k, sel_idx + (int64_t)b * k, kth + b);
        if (rc) { rcs[(size_t)b] = rc; return; }
        theta[b] = ema(theta[b], kth[b], alpha);
        std::vector<int32_t> mt((size_t)k), ms((size_t)k);
        int32_t nm = 0, nf = 0;
        rc = orc_cache_step(n, C, t2s, s2t, sel_idx + (int64_t)b * k, k, et.data(), ne, 0,
                            sel_slot + (int64_t)b * k, mt.data(), ms.data(), &nm, &nf);
        if (rc) { rcs[(size_t)b] = rc; return; }
        orc_recall(hrows, row_bytes, mt.data(), ms.data(), nm, drows);
        nmiss[b] = nm;
    };
    const int T = std::max(1, std::min(nthreads, B));
    std::vector<std::thread> pool;
    for (int t = 0; t < T; ++t)
        pool.emplace_back([&, t]() {
            for (int b = t; b < B; b += T) one(b);
        });
    for (auto& th : pool) th.join();
    for (int b = 0; b < B; ++b)
        if (rcs[(size_t)b]) return rcs[(size_t)b];
    return ORC_OK;
}

}  // extern "C"
