// echo_radix.cuh -- radix selection shared by the top-k kernels.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2
// "The top-k dependency": selection is an exact top-k; equal scores go to the
// lower token index.  Scores are compared through order_key (an unsigned key
// with the order of the float), so a radix select over the keys finds the
// k-th score exactly; a second select over the inverted indices of the keys
// equal to it finds the index cut.  The EMA threshold update (alpha = 0.5 of
// the previous k-th score, panel "Decode: fetch above a predicted threshold")
// lives here too, so that every top-k kernel applies it the same way.
//
// The selects run block-wide in 1024-thread blocks; the shared scratch is any
// struct with members hist[256], red[3], digit and above (uint32).
#pragma once

#include "echo_common.cuh"

namespace echo {
namespace radix {

constexpr int kTT = 1024;   // threads of every block that runs a select

// Warp 0: the largest digit d with (count of digits >= d) >= target, and the
// count strictly above d.  target >= 1 and total >= target.
__device__ inline void find_digit(const uint32_t* h, uint32_t target, uint32_t* out_digit, uint32_t* out_above) {
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

// Elements seen by a radix select.  for_each(f) calls f(v, ok) on every lane of
// a warp the same number of times, so f may use warp-collective operations;
// ok is false on lanes that hold no element.
struct SmemCands {
    const uint32_t* key;
    const uint32_t* idx;
    uint32_t cnt;
    bool by_index;      // select on ~index among key == eq_key
    uint32_t eq_key;
    template <class F>
    __device__ __forceinline__ void for_each(F f) const {
        for (uint32_t i0 = threadIdx.x & ~31u; i0 < cnt; i0 += kTT) {
            const uint32_t i = i0 + (threadIdx.x & 31u);
            bool ok = i < cnt;
            uint32_t v = 0;
            if (ok) {
                v = key[i];
                if (by_index) {
                    ok = v == eq_key;
                    v = ~idx[i];
                }
            }
            f(v, ok);
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
        for (int64_t s0 = threadIdx.x & ~31; s0 < n; s0 += kTT) {
            const int64_t s = s0 + (threadIdx.x & 31);
            bool ok = s < n;
            uint32_t v = 0;
            if (ok) {
                const float x = sc[s];
                v = order_key(x);
                ok = shifted_bin(x, shift) == bstar;
                if (by_index) {
                    ok = ok && v == eq_key;
                    v = ~static_cast<uint32_t>(s);
                }
            }
            f(v, ok);
        }
    }
};

// The r-th largest value (1-based) among the elements (block-wide); *rem = r
// minus the number of elements strictly larger (>= 1), *eq = number equal to it.
// The leading bits that every element shares are skipped (a boundary bin's
// keys share their sign and most of their exponent), and lanes adding to the
// same digit add once per warp.
template <class Src, class Sh>
__device__ uint32_t radix_select(const Src& src, uint32_t r, Sh& sh, uint32_t* rem, uint32_t* eq) {
    const unsigned lane = threadIdx.x & 31u;
    if (threadIdx.x == 0) {
        sh.red[0] = 0xFFFFFFFFu;
        sh.red[1] = 0u;
        sh.red[2] = 0u;
    }
    __syncthreads();
    src.for_each([&](uint32_t v, bool ok) {
        const unsigned m = __ballot_sync(0xffffffffu, ok);
        if (m == 0) return;
        const uint32_t lo = __reduce_min_sync(0xffffffffu, ok ? v : 0xFFFFFFFFu);
        const uint32_t hi = __reduce_max_sync(0xffffffffu, ok ? v : 0u);
        if (lane == 0) {
            atomicMin(&sh.red[0], lo);
            atomicMax(&sh.red[1], hi);
            atomicAdd(&sh.red[2], static_cast<uint32_t>(__popc(m)));
        }
    });
    __syncthreads();
    const uint32_t vmin = sh.red[0], vmax = sh.red[1], total = sh.red[2];
    if (vmin == vmax) {
        __syncthreads();  // everyone has read red before a later select resets it
        *rem = r;
        *eq = total;
        return vmin;
    }
    int shift = (31 - __clz(vmin ^ vmax)) & ~7;
    uint32_t mask = (shift >= 24) ? 0u : ~((1u << (shift + 8)) - 1u);
    uint32_t prefix = vmin & mask;
    uint32_t last_count = 0;
    for (; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kTT) sh.hist[i] = 0u;
        __syncthreads();
        src.for_each([&](uint32_t v, bool ok) {
            ok = ok && (v & mask) == prefix;
            const uint32_t d = (v >> shift) & 255u;
            const unsigned peers = __match_any_sync(0xffffffffu, ok ? d : 0x100u);
            if (ok && lane == static_cast<unsigned>(__ffs(peers) - 1))
                atomicAdd(&sh.hist[d], static_cast<uint32_t>(__popc(peers)));
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

// K* and the index cut over the scores in global memory, when the boundary
// bin does not fit shared memory (out of line: rare, and kept out of the
// common path's instruction stream).
template <class Sh>
__device__ __noinline__ uint32_t global_select(const float* sc, int64_t n, float shift, uint32_t bstar, uint32_t need,
                                               Sh& sh, uint32_t* idx_cut) {
    uint32_t rem = 0, eqn = 0;
    GlobalCands src{sc, n, shift, bstar, false, 0};
    const uint32_t K = radix_select(src, need, sh, &rem, &eqn);
    *idx_cut = 0xFFFFFFFFu;
    if (rem < eqn) {
        GlobalCands src2{sc, n, shift, bstar, true, K};
        uint32_t r2, e2;
        *idx_cut = ~radix_select(src2, rem, sh, &r2, &e2);
    }
    return K;
}


// The tokens s of [0, n), chunk after chunk of kTT * 8: thread t of the block
// holds tokens c0 + j * kTT + t for j < 8, loaded up front (8 independent loads
// in flight per thread, L2 only: the scores were just written), then calls
// f(x, s, ok) on each in order.  The 32 lanes of a warp hold 32 consecutive
// tokens starting at a multiple of 32, so a ballot over them is one bitmap
// word, and every lane calls f the same number of times (f may be
// warp-collective).
template <class F>
__device__ __forceinline__ void scan_scores(const float* sc, int64_t n, F f) {
    constexpr int U = 8;
    for (int64_t c0 = 0; c0 < n; c0 += static_cast<int64_t>(kTT) * U) {
        float x[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int64_t s = c0 + static_cast<int64_t>(j) * kTT + threadIdx.x;
            x[j] = s < n ? __ldcg(sc + s) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int64_t s = c0 + static_cast<int64_t>(j) * kTT + threadIdx.x;
            f(x[j], s, s < n);
        }
    }
}

// Key of a score shifted by the predicted threshold (its top 8 bits are the
// histogram bin).
__device__ __forceinline__ uint32_t shifted_key(float x, float shift) {
    return order_key(__fsub_rn(__fadd_rn(x, 0.0f), shift));
}

// Elements for a radix select over the scores in global memory: the tokens
// whose shifted key starts with `prefix` (its top pbits bits; pbits 8 or 16),
// as the order keys of their scores (or ~index among keys equal to eq_key).
struct ScoreScan {
    const float* sc;
    int64_t n;
    float shift;
    uint32_t prefix;
    int pbits;
    bool by_index;
    uint32_t eq_key;
    template <class F>
    __device__ __forceinline__ void for_each(F f) const {
        scan_scores(sc, n, [&](float x, int64_t s, bool ok) {
            uint32_t v = 0;
            if (ok) {
                ok = (shifted_key(x, shift) >> (32 - pbits)) == prefix;
                v = order_key(x);
                if (by_index) {
                    ok = ok && v == eq_key;
                    v = ~static_cast<uint32_t>(s);
                }
            }
            f(v, ok);
        });
    }
};

// The need-th largest key among the tokens with that shifted-key prefix, and
// (idx_cut non-null) the index cut among the tokens equal to it.
template <class Sh>
__device__ __noinline__ uint32_t scan_select(const float* sc, int64_t n, float shift, uint32_t prefix, int pbits,
                                             uint32_t need, Sh& sh, uint32_t* idx_cut) {
    uint32_t rem = 0, eqn = 0;
    const uint32_t K = radix_select(ScoreScan{sc, n, shift, prefix, pbits, false, 0u}, need, sh, &rem, &eqn);
    if (idx_cut) {
        *idx_cut = 0xFFFFFFFFu;
        if (rem < eqn) {
            uint32_t r2, e2;
            *idx_cut = ~radix_select(ScoreScan{sc, n, shift, prefix, pbits, true, K}, rem, sh, &r2, &e2);
        }
    }
    return K;
}

}  // namespace radix
}  // namespace echo
