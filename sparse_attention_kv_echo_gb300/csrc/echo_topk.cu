// echo_topk.cu -- exact top-k per request and the EMA threshold update.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2
// "The top-k dependency": selection is an exact top-k; the predicted
// threshold is an EMA (alpha = 0.5) of the previous step's k-th score; the
// real kernel bins scores by the top 8 bits of each score shifted by the
// predicted threshold (panel "Prefill: one-round histogram").
//
// One thread-block cluster of kCS CTAs (1024 threads each) per request; CTA r
// of the cluster owns the r-th contiguous slice of the request's tokens.
//   1. boundary bin: from the 256-bin histogram of the shifted scores (made by
//      the score kernel, or rebuilt here), the bin b* where the count from the
//      top reaches k.  Shifting is monotone, so every token in a bin above b*
//      outranks every token at or below it.
//   2. every CTA scans its slice once and appends the tokens of bin b* to the
//      leader CTA's shared memory through distributed shared memory (one
//      atomic per warp); the leader runs a radix select (four 8-bit digits of
//      the order key) for K*, the key of the k-th score, and a second one on
//      ~index to resolve equal keys towards the lower index.  When bin b*
//      does not fit in shared memory the leader runs the same selects as
//      passes over the scores in global memory.
//   3. every CTA counts its selected tokens; a cluster-wide prefix of those
//      counts (read over DSMEM) places each slice, and one ordered pass per
//      slice writes the indices in ascending order with block-wide scans.
// A good prediction puts the k-th score near 0 after the shift, where the
// exponent bins are narrow, so the boundary bin holds few tokens.
#include <cooperative_groups.h>

#include "echo_common.cuh"
#include "echo_internal.h"

namespace cg = cooperative_groups;

namespace echo {
namespace {

constexpr int kTT = 1024;
constexpr int kCS = 8;           // CTAs per request (one cluster)
constexpr int kCandMax = 12288;  // boundary-bin entries the leader keeps in shared memory

struct TopkShared {
    uint32_t hist[256];
    uint32_t hist_acc[256];      // leader: cluster-wide rebuild of the histogram
    uint32_t scan[40];
    uint32_t cand_key[kCandMax];
    uint32_t cand_idx[kCandMax];
    uint32_t cnt;                // leader: boundary-bin entries appended
    uint32_t chk_above;          // leader: tokens above b*, summed over the cluster
    uint32_t chk_eq;             // leader: tokens in b*, summed over the cluster
    uint32_t digit;
    uint32_t above;
    uint32_t minkey;
    uint32_t flag;
    uint32_t K;                  // leader -> all: key of the k-th score
    uint32_t idx_cut;            // leader -> all: last index taken among keys == K
    uint32_t selected;           // this CTA's number of selected tokens
};

// Warp 0: the largest digit d with (count of digits >= d) >= target, and the
// count strictly above d.  target >= 1 and total >= target.
__device__ void find_digit(const uint32_t* h, uint32_t target, uint32_t* out_digit, uint32_t* out_above) {
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
    const uint32_t above_lane = suf - sum;
    const bool hit = above_lane < target && suf >= target;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (m == 0) {
        if (lane == 0) {
            *out_digit = 0;
            *out_above = 0;
        }
        return;
    }
    if (lane == __ffs(m) - 1) {
        uint32_t acc = above_lane;
        int d = 8 * lane;
        for (int j = 7; j >= 0; --j) {
            if (acc + c[j] >= target) {
                d = 8 * lane + j;
                break;
            }
            acc += c[j];
        }
        *out_digit = static_cast<uint32_t>(d);
        *out_above = acc;
    }
}

// Elements seen by a radix select.
struct SmemCands {
    const uint32_t* key;
    const uint32_t* idx;
    uint32_t cnt;
    bool by_index;      // select on ~index among key == eq_key
    uint32_t eq_key;
    template <class F>
    __device__ __forceinline__ void for_each(F f) const {
        for (uint32_t i = threadIdx.x; i < cnt; i += kTT) {
            if (!by_index)
                f(key[i]);
            else if (key[i] == eq_key)
                f(~idx[i]);
        }
    }
};

struct GlobalCands {
    const float* sc;
    int64_t n;
    float shift;
    uint32_t bstar;
    bool by_index;
    uint32_t eq_key;
    template <class F>
    __device__ __forceinline__ void for_each(F f) const {
        for (int64_t s = threadIdx.x; s < n; s += kTT) {
            const float x = sc[s];
            if (shifted_bin(x, shift) != bstar) continue;
            const uint32_t key = order_key(x);
            if (!by_index)
                f(key);
            else if (key == eq_key)
                f(~static_cast<uint32_t>(s));
        }
    }
};

// The r-th largest value (1-based) among the elements (block-wide); *rem = r
// minus the number of elements strictly larger (>= 1), *eq = number equal to it.
template <class Src>
__device__ uint32_t radix_select(const Src& src, uint32_t r, TopkShared& sh, uint32_t* rem, uint32_t* eq) {
    uint32_t prefix = 0, mask = 0;
    uint32_t last_count = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kTT) sh.hist[i] = 0u;
        __syncthreads();
        src.for_each([&](uint32_t v) {
            if ((v & mask) == prefix) atomicAdd(&sh.hist[(v >> shift) & 255u], 1u);
        });
        __syncthreads();
        if (threadIdx.x < 32) find_digit(sh.hist, r, &sh.digit, &sh.above);
        __syncthreads();
        const uint32_t d = sh.digit;
        r -= sh.above;
        last_count = sh.hist[d];
        prefix |= d << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    *rem = r;
    *eq = last_count;
    return prefix;
}

__device__ __forceinline__ float ema_update(float theta, float kth, float alpha) {
    if (isinf(theta)) return kth;
    const float a = __fmul_rn(alpha, kth);
    const float b = __fmul_rn(__fsub_rn(1.0f, alpha), theta);
    return __fadd_rn(a, b);
}

__device__ __forceinline__ bool takes(float x, float shift, uint32_t bstar, uint32_t K, uint32_t cut, int64_t s) {
    const uint32_t bin = shifted_bin(x, shift);
    const uint32_t key = order_key(x);
    return bin > bstar || (bin == bstar && (key > K || (key == K && static_cast<uint32_t>(s) <= cut)));
}

// Segments: decode requests (CSR tok_off over the scores) or prefill rows
// (W > 0: row b holds row0 + b + 1 scores starting at b * W).  In prefill the
// threshold is one scalar for every row and is not updated here.
struct TopkSegs {
    const int64_t* tok_off;
    int64_t n_tokens;
    int64_t row0;
    int64_t W;
};

__global__ void __cluster_dims__(kCS, 1, 1) __launch_bounds__(kTT, 1)
    topk_kernel(TopkSegs segs, const float* __restrict__ scores, int k, const uint32_t* __restrict__ hist,
                float* theta_hat, float alpha, int32_t* __restrict__ sel, float* kth_out, int32_t* status,
                uint32_t* stats) {
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
        lo = segs.tok_off[b];
        const int64_t hi = segs.tok_off[b + 1];
        n = hi - lo;
        if (lo < 0 || hi < lo || hi > segs.n_tokens) {
            if (leader && tid == 0) set_status(status, ECHO_ST_BADDATA);
            n = 0;
        }
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

    // this CTA's slice of the request
    const int64_t s_lo = n * rank / kCS, s_hi = n * (rank + 1) / kCS;

    // ---- 1-2. boundary bin, its tokens gathered in the leader
    bool have = hist != nullptr;
    uint32_t bstar = 0, above = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        if (have) {
            for (int i = tid; i < 256; i += kTT) sh.hist[i] = hist[static_cast<int64_t>(b) * 256 + i];
        } else {
            // rebuild: slice histograms summed into the leader over DSMEM
            if (leader)
                for (int i = tid; i < 256; i += kTT) sh.hist_acc[i] = 0u;
            for (int i = tid; i < 256; i += kTT) sh.hist[i] = 0u;
            cluster.sync();
            for (int64_t s0 = s_lo; s0 < s_hi; s0 += kTT) {
                const int64_t s = s0 + tid;
                const bool v = s < s_hi;
                const uint32_t bin = v ? shifted_bin(sc[s], shift) : 256u;
                const unsigned grp = __match_any_sync(0xffffffffu, bin);
                if (v && (tid & 31) == __ffs(grp) - 1) atomicAdd(&sh.hist[bin], __popc(grp));
            }
            __syncthreads();
            for (int i = tid; i < 256; i += kTT)
                if (sh.hist[i]) atomicAdd(&lsh.hist_acc[i], sh.hist[i]);
            cluster.sync();
            for (int i = tid; i < 256; i += kTT) sh.hist[i] = lsh.hist_acc[i];
        }
        __syncthreads();
        if (tid < 32) find_digit(sh.hist, static_cast<uint32_t>(k), &sh.digit, &sh.above);
        if (leader && tid == 0) {
            sh.cnt = 0;
            sh.chk_above = 0;
            sh.chk_eq = 0;
        }
        __syncthreads();
        bstar = sh.digit;
        above = sh.above;
        const uint32_t eq_total = sh.hist[bstar];
        cluster.sync();  // the leader's counters are reset before anyone appends
        uint32_t my_above = 0, my_eq = 0;
        for (int64_t s0 = s_lo; s0 < s_hi; s0 += kTT) {
            const int64_t s = s0 + tid;
            const bool v = s < s_hi;
            const float x = v ? sc[s] : 0.f;
            const uint32_t bin = shifted_bin(x, shift);
            my_above += v && bin > bstar;
            const bool in = v && bin == bstar;
            my_eq += in;
            const unsigned m = __ballot_sync(0xffffffffu, in);
            if (in) {
                const int leader_lane = __ffs(m) - 1;
                uint32_t basepos = 0;
                if ((tid & 31) == leader_lane) basepos = atomicAdd(&lsh.cnt, __popc(m));
                basepos = __shfl_sync(m, basepos, leader_lane);
                const uint32_t pos = basepos + __popc(m & ((1u << (tid & 31)) - 1u));
                if (pos < kCandMax) {
                    lsh.cand_key[pos] = order_key(x);
                    lsh.cand_idx[pos] = static_cast<uint32_t>(s);
                }
            }
        }
        // warp-reduce the checks before the remote atomics
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            my_above += __shfl_xor_sync(0xffffffffu, my_above, o);
            my_eq += __shfl_xor_sync(0xffffffffu, my_eq, o);
        }
        if ((tid & 31) == 0) {
            if (my_above) atomicAdd(&lsh.chk_above, my_above);
            if (my_eq) atomicAdd(&lsh.chk_eq, my_eq);
        }
        cluster.sync();
        const bool consistent = lsh.chk_above == above && lsh.chk_eq == eq_total;
        cluster.sync();  // everyone has read the leader's checks before they may be reset
        if (consistent) break;
        // The histogram given does not describe these scores: rebuild it here.
        if (leader && tid == 0) set_status(status, ECHO_ST_BADDATA);
        have = false;
    }

    // ---- 3. K*, the key of the k-th score, and the index cut among equal keys (leader)
    if (leader) {
        const uint32_t need = static_cast<uint32_t>(k) - above;  // >= 1
        const uint32_t cnt = sh.cnt;
        if (tid == 0 && stats) {
            atomicMax(stats + ECHO_STAT_BOUNDARY_MAX, cnt);
            if (cnt > kCandMax) atomicAdd(stats + ECHO_STAT_TOPK_FALLBACK, 1u);
        }
        uint32_t rem = 0, eqn = 0, K = 0, idx_cut = 0xFFFFFFFFu;
        if (cnt <= kCandMax) {
            SmemCands src{sh.cand_key, sh.cand_idx, cnt, false, 0};
            K = radix_select(src, need, sh, &rem, &eqn);
            if (rem < eqn) {
                SmemCands src2{sh.cand_key, sh.cand_idx, cnt, true, K};
                uint32_t r2, e2;
                idx_cut = ~radix_select(src2, rem, sh, &r2, &e2);
            }
        } else {
            GlobalCands src{sc, n, shift, bstar, false, 0};
            K = radix_select(src, need, sh, &rem, &eqn);
            if (rem < eqn) {
                GlobalCands src2{sc, n, shift, bstar, true, K};
                uint32_t r2, e2;
                idx_cut = ~radix_select(src2, rem, sh, &r2, &e2);
            }
        }
        if (tid == 0) {
            sh.K = K;
            sh.idx_cut = idx_cut;
        }
    }
    cluster.sync();
    const uint32_t K = lsh.K, idx_cut = lsh.idx_cut;

    // ---- 4. ordered compaction: count, cluster prefix, write
    uint32_t mine = 0;
    bool nan = false;
    for (int64_t s = s_lo + tid; s < s_hi; s += kTT) {
        const float x = sc[s];
        nan |= isnan(x);
        mine += takes(x, shift, bstar, K, idx_cut, s);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
    if (tid == 0) {
        sh.selected = 0;
        sh.flag = 0;
    }
    __syncthreads();
    if ((tid & 31) == 0 && mine) atomicAdd(&sh.selected, mine);
    if (nan) sh.flag = 1;
    cluster.sync();
    uint32_t offset = 0, total = 0;
    for (int r = 0; r < kCS; ++r) {
        const uint32_t c = cluster.map_shared_rank(&sh, r)->selected;
        if (r < rank) offset += c;
        total += c;
    }
    uint32_t written = offset;
    for (int64_t c0 = s_lo; c0 < s_hi; c0 += 4 * kTT) {
        const int64_t s0 = c0 + 4 * tid;
        uint32_t f = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t s = s0 + j;
            if (s < s_hi && takes(sc[s], shift, bstar, K, idx_cut, s)) f |= 1u << j;
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
        for (int i = static_cast<int>(total) + tid; i < k; i += kTT) out[i] = -1;
        if (tid == 0) {
            if (total != static_cast<uint32_t>(k)) set_status(status, ECHO_ST_BADDATA);
            const float kth = key_to_float(K);
            kth_out[b] = kth;
            if (theta_upd) theta_upd[b] = ema_update(th_old, kth, alpha);
        }
    }
    if (tid == 0 && sh.flag) set_status(status, ECHO_ST_NAN);
    cluster.sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace
}  // namespace echo

namespace echo {

int launch_topk(int B, const int64_t* tok_off, int64_t n_tokens, int64_t row0, int64_t W, const float* scores, int k,
                const uint32_t* hist, float* theta_hat, float alpha, int32_t* sel_idx, float* kth, int32_t* status,
                uint32_t* stats, cudaStream_t stream) {
    const size_t smem = sizeof(TopkShared);
    ECHO_CUDA_OK(prefer_max_shared(topk_kernel));
    ECHO_CUDA_OK(cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
    TopkSegs segs{tok_off, n_tokens, row0, W};
    topk_kernel<<<B * kCS, kTT, smem, stream>>>(segs, scores, k, hist, theta_hat, alpha, sel_idx, kth, status, stats);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}

}  // namespace echo

extern "C" int echo_topk_select(int B, const int64_t* tok_off, int64_t n_tokens, const float* scores, int k,
                                const uint32_t* hist, float* theta_hat, float alpha, int32_t* sel_idx, float* kth,
                                int32_t* status, uint32_t* stats, echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || n_tokens < 0 || k <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !sel_idx || !kth || !status || (n_tokens > 0 && !scores)) return ECHO_EINVAL;
    if (n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    return launch_topk(B, tok_off, n_tokens, 0, 0, scores, k, hist, theta_hat, alpha, sel_idx, kth, status, stats,
                       stream);
}
