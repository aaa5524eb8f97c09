// echo_topk.cu -- exact top-k per request and the EMA threshold update.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2
// "The top-k dependency": selection is an exact top-k; the predicted
// threshold is an EMA (alpha = 0.5) of the previous step's k-th score; the
// real kernel bins scores by the top 8 bits of each score shifted by the
// predicted threshold (panel "Prefill: one-round histogram").
//
// One CTA of 1024 threads per request:
//   1. boundary bin: from the 256-bin histogram of the shifted scores (made by
//      the score kernel, or here), the bin b* where the count from the top
//      reaches k.  Shifting is monotone, so every token in a bin above b*
//      outranks every token at or below it.
//   2. one pass collects the tokens of bin b* into shared memory; a radix
//      select (four 8-bit digits of the order key) finds K*, the key of the
//      k-th score, and a second radix select on ~index resolves equal keys
//      towards the lower index.  When bin b* does not fit in shared memory the
//      same selects run as passes over the scores in global memory.
//   3. one ordered pass writes the selected indices in ascending order with
//      block-wide prefix sums; the k-th score updates the EMA.
// A good prediction puts the k-th score near 0 after the shift, where the
// exponent bins are narrow, so the boundary bin holds few tokens.
#include "echo_common.cuh"
#include "echo_internal.h"

namespace echo {
namespace {

constexpr int kTT = 1024;
constexpr int kCandMax = 12288;

struct TopkShared {
    uint32_t hist[256];
    uint32_t scan[40];
    uint32_t cand_key[kCandMax];
    uint32_t cand_idx[kCandMax];
    uint32_t cnt;
    uint32_t digit;
    uint32_t above;
    uint32_t minkey;
    uint32_t flag;
    uint32_t chk_above;
    uint32_t chk_eq;
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

// The r-th largest value (1-based) among the elements; *rem = r minus the
// number of elements strictly larger (>= 1), *eq = number equal to it.
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

__global__ void __launch_bounds__(kTT, 1)
    topk_kernel(const int64_t* __restrict__ tok_off, int64_t n_tokens, const float* __restrict__ scores, int k,
                const uint32_t* __restrict__ hist, float* theta_hat, float alpha, int32_t* __restrict__ sel,
                float* kth_out, int32_t* status, uint32_t* stats) {
    extern __shared__ uint8_t smem_raw[];
    TopkShared& sh = *reinterpret_cast<TopkShared*>(smem_raw);
    const int b = blockIdx.x, tid = threadIdx.x;
    const int64_t lo = tok_off[b], hi = tok_off[b + 1];
    int64_t n = hi - lo;
    if (lo < 0 || hi < lo || hi > n_tokens) {
        if (tid == 0) set_status(status, ECHO_ST_BADDATA);
        n = 0;
    }
    const float* sc = scores + (n > 0 ? lo : 0);
    int32_t* out = sel + static_cast<int64_t>(b) * k;
    const float th_old = theta_hat ? theta_hat[b] : __int_as_float(0x7f800000);
    const float shift = isfinite(th_old) ? th_old : 0.f;

    if (n == 0) {
        for (int i = tid; i < k; i += kTT) out[i] = -1;
        if (tid == 0) kth_out[b] = __int_as_float(0xff800000);
        return;
    }
    if (n <= k) {
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
            if (theta_hat) theta_hat[b] = ema_update(th_old, kth, alpha);
        }
        return;
    }

    // ---- 1. histogram of shifted bins, boundary bin
    bool have = hist != nullptr;
    uint32_t bstar = 0, above = 0, eq_total = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        if (have) {
            for (int i = tid; i < 256; i += kTT) sh.hist[i] = hist[static_cast<int64_t>(b) * 256 + i];
        } else {
            for (int i = tid; i < 256; i += kTT) sh.hist[i] = 0u;
            __syncthreads();
            for (int64_t s0 = 0; s0 < n; s0 += kTT) {
                const int64_t s = s0 + tid;
                const bool v = s < n;
                const uint32_t bin = v ? shifted_bin(sc[s], shift) : 256u;
                const unsigned grp = __match_any_sync(0xffffffffu, bin);
                if (v && (tid & 31) == __ffs(grp) - 1) atomicAdd(&sh.hist[bin], __popc(grp));
            }
        }
        __syncthreads();
        if (tid < 32) find_digit(sh.hist, static_cast<uint32_t>(k), &sh.digit, &sh.above);
        if (tid == 0) {
            sh.cnt = 0;
            sh.chk_above = 0;
            sh.chk_eq = 0;
        }
        __syncthreads();
        bstar = sh.digit;
        above = sh.above;
        eq_total = sh.hist[bstar];
        // ---- 2. collect the boundary bin; count what lies above it
        uint32_t my_above = 0, my_eq = 0;
        for (int64_t s0 = 0; s0 < n; s0 += kTT) {
            const int64_t s = s0 + tid;
            const bool v = s < n;
            const float x = v ? sc[s] : 0.f;
            const uint32_t bin = shifted_bin(x, shift);
            my_above += v && bin > bstar;
            const bool in = v && bin == bstar;
            my_eq += in;
            const unsigned m = __ballot_sync(0xffffffffu, in);
            if (in) {
                const int leader = __ffs(m) - 1;
                uint32_t basepos = 0;
                if ((tid & 31) == leader) basepos = atomicAdd(&sh.cnt, __popc(m));
                basepos = __shfl_sync(m, basepos, leader);
                const uint32_t pos = basepos + __popc(m & ((1u << (tid & 31)) - 1u));
                if (pos < kCandMax) {
                    sh.cand_key[pos] = order_key(x);
                    sh.cand_idx[pos] = static_cast<uint32_t>(s);
                }
            }
        }
        atomicAdd(&sh.chk_above, my_above);
        atomicAdd(&sh.chk_eq, my_eq);
        __syncthreads();
        if (sh.chk_above == above && sh.chk_eq == eq_total) break;
        // The histogram given does not describe these scores: rebuild it here.
        if (tid == 0) set_status(status, ECHO_ST_BADDATA);
        have = false;
        __syncthreads();
    }
    const uint32_t need = static_cast<uint32_t>(k) - above;  // >= 1
    const uint32_t cnt = sh.cnt;
    if (tid == 0 && stats) {
        atomicMax(stats + ECHO_STAT_BOUNDARY_MAX, cnt);
        if (cnt > kCandMax) atomicAdd(stats + ECHO_STAT_TOPK_FALLBACK, 1u);
    }
    __syncthreads();

    // ---- 3. K*, the key of the k-th score, and the index cut among equal keys
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

    // ---- 4. ordered compaction
    if (tid == 0) sh.flag = 0;
    __syncthreads();
    uint32_t written = 0;
    bool nan = false;
    for (int64_t c0 = 0; c0 < n; c0 += 4 * kTT) {
        const int64_t s0 = c0 + 4 * tid;
        uint32_t f = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t s = s0 + j;
            if (s < n) {
                const float x = sc[s];
                nan |= isnan(x);
                const uint32_t bin = shifted_bin(x, shift);
                const uint32_t key = order_key(x);
                const bool take = bin > bstar ||
                                  (bin == bstar && (key > K || (key == K && static_cast<uint32_t>(s) <= idx_cut)));
                f |= static_cast<uint32_t>(take) << j;
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
    if (nan) sh.flag = 1;
    for (int i = static_cast<int>(written) + tid; i < k; i += kTT) out[i] = -1;
    __syncthreads();
    if (tid == 0) {
        if (sh.flag) set_status(status, ECHO_ST_NAN);
        if (written != static_cast<uint32_t>(k)) set_status(status, ECHO_ST_BADDATA);
        const float kth = key_to_float(K);
        kth_out[b] = kth;
        if (theta_hat) theta_hat[b] = ema_update(th_old, kth, alpha);
    }
}

}  // namespace
}  // namespace echo

extern "C" int echo_topk_select(int B, const int64_t* tok_off, int64_t n_tokens, const float* scores, int k,
                                const uint32_t* hist, float* theta_hat, float alpha, int32_t* sel_idx, float* kth,
                                int32_t* status, uint32_t* stats, echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || n_tokens < 0 || k <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !sel_idx || !kth || !status || (n_tokens > 0 && !scores)) return ECHO_EINVAL;
    if (n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    const size_t smem = sizeof(TopkShared);
    ECHO_CUDA_OK(cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
    topk_kernel<<<B, kTT, smem, stream>>>(tok_off, n_tokens, scores, k, hist, theta_hat, alpha, sel_idx, kth, status,
                                          stats);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}
