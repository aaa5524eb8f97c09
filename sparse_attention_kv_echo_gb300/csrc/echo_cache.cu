// echo_cache.cu -- the per-layer GPU cache step, early fetch and recall.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2:
//   panel "Five fixed-size integer tensors on the GPU": nothing changes
//     length, so a decode step stays inside one CUDA graph;
//   panel "One layer, one step: free -> allocate -> recall": unselected slots
//     are freed (no write-back: the host holds every token), misses get
//     slots, their rows are recalled from the host pool;
//   panel "Decode: fetch above a predicted threshold": tokens scoring above
//     the predicted threshold are fetched before top-k completes, up to a cap.
//
// Kernels (one CTA of 1024 threads per request for the table work):
//   early_select_kernel  ordered scan of the score kernel's above-threshold bits
//                        (one word per 32 tokens), keeping non-resident tokens
//                        (block prefix sums); the first min(cap, free) of them
//                        take the lowest free slots.
//   cache_step_kernel    marks the slots of selected residents in a shared
//                        bitmap, frees the rest one warp per 32-slot word
//                        (ballot -> free-bit word), compacts the misses in
//                        ascending order, hands them the lowest free slots by a
//                        prefix sum of popcounts over the free-bit words.
//   recall_kernel        one warp per row, 16-byte loads from the pinned host
//                        pool through its device alias (zero-copy over the
//                        host link), 16-byte stores into the device cache.
#include "echo_common.cuh"
#include "echo_internal.h"

namespace echo {
namespace {

constexpr int kCT = 1024;
constexpr int kMaxSlotsSmem = 1 << 19;   // per-slot-word tables in shared memory: 3 x 2^14 words (192 KB)

struct CacheArgs {
    int32_t* tok2slot;
    int32_t* slot2tok;
    uint32_t* freebits;
    int32_t* miss_tok;
    int32_t* miss_slot;
    int32_t* miss_cnt;
    int32_t* early_tok;
    int32_t* early_slot;
    int32_t* early_cnt;
    int32_t C;
};

CacheArgs cache_args(const echo_cache& c) {
    return CacheArgs{c.tok2slot, c.slot2tok, c.freebits, c.miss_tok, c.miss_slot, c.miss_cnt,
                     c.early_tok, c.early_slot, c.early_cnt, c.C};
}

__device__ __forceinline__ bool request_range(const int64_t* tok_off, int64_t n_tokens, int b, int64_t* base,
                                              int64_t* n) {
    const int64_t lo = tok_off[b], hi = tok_off[b + 1];
    if (lo < 0 || hi < lo || hi > n_tokens) {
        *base = 0;
        *n = 0;
        return false;
    }
    *base = lo;
    *n = hi - lo;
    return true;
}

// Give the first M tokens of tok_list the M lowest free slots of one
// request, in ascending order.  Block-wide and parallel over ranks: a prefix
// of the free-slot counts of the bit words (wpre, shared memory) maps rank r to
// its word by binary search and to its bit as the (r - wpre[w])-th set bit.
// wpre: words + 1 entries, fbs: words entries of shared memory.  Returns the
// number assigned.
__device__ uint32_t assign_lowest_free(uint32_t* fb, int words, uint32_t M, const int32_t* tok_list,
                                       int32_t* slot_list, int32_t* t2s, int32_t* s2t, int64_t n, int C,
                                       uint32_t* scan, uint32_t* wpre, uint32_t* fbs, int32_t* status) {
    uint32_t run = 0;
    for (int w0 = 0; w0 < words; w0 += kCT) {
        const int w = w0 + threadIdx.x;
        const uint32_t f = (w < words) ? fb[w] : 0u;
        if (w < words) fbs[w] = f;
        uint32_t tot;
        const uint32_t ex = block_exclusive_scan<kCT>(__popc(f), scan, &tot);
        if (w < words) wpre[w] = run + ex;
        run += tot;
    }
    if (threadIdx.x == 0) wpre[words] = run;
    __syncthreads();
    const uint32_t take = M < run ? M : run;
    for (uint32_t r = threadIdx.x; r < take; r += kCT) {
        int lo = 0, hi = words - 1;   // largest w with wpre[w] <= r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (wpre[mid] <= r)
                lo = mid;
            else
                hi = mid - 1;
        }
        uint32_t f = fbs[lo];
        for (uint32_t i = r - wpre[lo]; i > 0; --i) f &= f - 1;
        const int slot = lo * 32 + (__ffs(f) - 1);
        const int32_t tok = tok_list[r];
        if (tok >= 0 && tok < n && slot < C && t2s[tok] < 0) {
            t2s[tok] = slot;
            s2t[slot] = tok;
            slot_list[r] = slot;
        } else {
            set_status(status, ECHO_ST_BADDATA);
        }
    }
    // the taken slots are the lowest `take` free ones: clear them word by word
    for (int w = threadIdx.x; w < words; w += kCT) {
        if (wpre[w] >= take) continue;
        uint32_t f = fbs[w];
        uint32_t k = take - wpre[w];
        uint32_t taken = 0;
        while (f && k) {
            const uint32_t low = f & (0u - f);
            taken |= low;
            f ^= low;
            --k;
        }
        if (taken) fb[w] = fbs[w] & ~taken;
    }
    if (take < M && threadIdx.x == 0) set_status(status, ECHO_ST_NOSLOT);
    __syncthreads();
    return take;
}

// Tiles of 128 tokens of request b, and the first tile of b in the list of all
// requests' tiles (the order the score kernel writes its above-threshold words in).
__device__ uint32_t first_tile_of(const int64_t* tok_off, int64_t n_tokens, int b, uint32_t* scan) {
    uint32_t part = 0;
    for (int bb = threadIdx.x; bb < b; bb += kCT) {
        const int64_t lo = tok_off[bb], hi = tok_off[bb + 1];
        if (lo >= 0 && hi >= lo && hi <= n_tokens) part += static_cast<uint32_t>((hi - lo + 127) / 128);
    }
    uint32_t total;
    block_exclusive_scan<kCT>(part, scan, &total);
    return total;
}

__global__ void __launch_bounds__(kCT) early_select_kernel(const int64_t* __restrict__ tok_off, int64_t n_tokens,
                                                           const uint32_t* __restrict__ above, int cap, CacheArgs c,
                                                           int32_t* status, uint32_t* stats) {
    __shared__ uint32_t scan[40];
    extern __shared__ uint32_t dyn[];   // wpre [words + 1], fbs [words]
    const int b = blockIdx.x, tid = threadIdx.x;
    int64_t base, n;
    if (!request_range(tok_off, n_tokens, b, &base, &n) && tid == 0) set_status(status, ECHO_ST_BADDATA);
    const int C = c.C, words = C / 32;
    uint32_t* wpre = dyn;
    uint32_t* fbs = dyn + words + 1;
    int32_t* t2s = c.tok2slot + base;
    int32_t* s2t = c.slot2tok + static_cast<int64_t>(b) * C;
    uint32_t* fb = c.freebits + static_cast<int64_t>(b) * words;
    int32_t* etok = c.early_tok + static_cast<int64_t>(b) * C;
    int32_t* eslot = c.early_slot + static_cast<int64_t>(b) * C;
    if (n == 0 || cap == 0) {
        if (tid == 0) c.early_cnt[b] = 0;
        return;
    }
    const uint32_t t0 = first_tile_of(tok_off, n_tokens, b, scan);
    const uint32_t* ab = above + 4 * static_cast<size_t>(t0);
    const int awords = static_cast<int>(4 * ((n + 127) / 128));
    uint32_t F = 0;
    for (int w0 = 0; w0 < words; w0 += kCT) {
        const int w = w0 + tid;
        uint32_t tot;
        block_exclusive_scan<kCT>(w < words ? __popc(fb[w]) : 0u, scan, &tot);
        F += tot;
    }
    const uint32_t limit = (cap < 0) ? F : min(F, static_cast<uint32_t>(cap));
    uint32_t found = 0;
    // word w covers tokens 32*w .. 32*w+31 of the request: ascending word, ascending bit;
    // the marked tokens are the non-resident ones above the threshold
    for (int w0 = 0; w0 < awords && found < limit; w0 += kCT) {
        const int w = w0 + tid;
        uint32_t cand = (w < awords) ? ab[w] : 0u;
        if (w == awords - 1 && (n & 31)) cand &= (1u << (n & 31)) - 1u;   // no token past the request end
        uint32_t tot;
        uint32_t rank = found + block_exclusive_scan<kCT>(__popc(cand), scan, &tot);
        while (cand) {
            const int bit = __ffs(cand) - 1;
            cand &= cand - 1;
            if (rank < limit) etok[rank] = 32 * w + bit;
            ++rank;
        }
        found += tot;
    }
    const uint32_t E = min(found, limit);
    __syncthreads();
    const uint32_t got = assign_lowest_free(fb, words, E, etok, eslot, t2s, s2t, n, C, scan, wpre, fbs, status);
    if (tid == 0) {
        c.early_cnt[b] = static_cast<int32_t>(got);
        if (stats && got) atomicAdd(stats + ECHO_STAT_EARLY, got);
    }
}

__global__ void __launch_bounds__(kCT) cache_step_kernel(const int64_t* __restrict__ tok_off, int64_t n_tokens,
                                                         const int32_t* __restrict__ sel, int m, CacheArgs c,
                                                         int32_t* __restrict__ sel_slot, int32_t* status,
                                                         uint32_t* stats) {
    extern __shared__ uint32_t keep[];  // keep [words]: a selected token lives in the slot; then wpre, fbs
    __shared__ uint32_t scan[40];
    __shared__ uint32_t s_flags;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int64_t base, n;
    if (!request_range(tok_off, n_tokens, b, &base, &n) && tid == 0) set_status(status, ECHO_ST_BADDATA);
    const int C = c.C, words = C / 32;
    int32_t* t2s = c.tok2slot + base;
    int32_t* s2t = c.slot2tok + static_cast<int64_t>(b) * C;
    uint32_t* fb = c.freebits + static_cast<int64_t>(b) * words;
    const int32_t* sl = sel + static_cast<int64_t>(b) * m;
    int32_t* mtok = c.miss_tok + static_cast<int64_t>(b) * C;
    int32_t* mslot = c.miss_slot + static_cast<int64_t>(b) * C;
    uint32_t* wpre = keep + words;
    uint32_t* fbs = wpre + words + 1;

    for (int w = tid; w < words; w += kCT) keep[w] = 0u;
    if (tid == 0) s_flags = 0;
    __syncthreads();
    // 1a. slots that hold a selected token are kept
    for (int i = tid; i < m; i += kCT) {
        const int32_t s = sl[i];
        if (s < 0) continue;
        if (s >= n) {
            atomicOr(&s_flags, static_cast<uint32_t>(ECHO_ST_BADDATA));
            continue;
        }
        const int32_t j = t2s[s];
        if (j >= 0 && j < C) atomicOr(&keep[j >> 5], 1u << (j & 31));
    }
    __syncthreads();
    // 1b. every other occupied slot is freed; bytes stay, nothing is written back
    for (int w = warp; w < words; w += kCT / 32) {
        const int slot = w * 32 + lane;
        const int32_t s = s2t[slot];
        const bool kept = (keep[w] >> lane) & 1u;
        const bool freeing = s >= 0 && !kept;
        if (freeing) {
            s2t[slot] = -1;
            if (s < n) t2s[s] = -1;
        }
        const unsigned fm = __ballot_sync(0xffffffffu, freeing);
        if (lane == 0 && fm) fb[w] |= fm;
    }
    __syncthreads();
    // 2. misses, ascending; the selection must be ascending with -1 padding last
    uint32_t M = 0, early_used = 0;
    for (int c0 = 0; c0 < m; c0 += 4 * kCT) {
        const int i0 = c0 + 4 * tid;
        uint32_t f = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j;
            if (i < m) {
                const int32_t s = sl[i];
                if (s >= 0 && s < n) {
                    if (i + 1 < m && sl[i + 1] >= 0 && sl[i + 1] <= s)
                        atomicOr(&s_flags, static_cast<uint32_t>(ECHO_ST_BADDATA));
                    if (t2s[s] < 0) f |= 1u << j;
                } else if (s >= 0 || (i + 1 < m && sl[i + 1] >= 0)) {
                    atomicOr(&s_flags, static_cast<uint32_t>(ECHO_ST_BADDATA));
                }
            }
        }
        uint32_t tot;
        uint32_t rank = M + block_exclusive_scan<kCT>(__popc(f), scan, &tot);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (f & (1u << j)) {
                if (rank < static_cast<uint32_t>(C)) mtok[rank] = sl[i0 + j];
                ++rank;
            }
        M += tot;
    }
    if (M > static_cast<uint32_t>(C)) M = C;
    // early fetches of this step that the selection kept
    const int ecnt = min(c.early_cnt[b], C);
    for (int i = tid; i < ecnt; i += kCT) {
        const int32_t s = c.early_tok[static_cast<int64_t>(b) * C + i];
        if (s >= 0 && s < n && t2s[s] >= 0) ++early_used;
    }
    __syncthreads();
    // 3. the misses take the lowest free slots
    const uint32_t got = assign_lowest_free(fb, words, M, mtok, mslot, t2s, s2t, n, C, scan, wpre, fbs, status);
    __syncthreads();
    // 4. slot of every selected entry
    for (int i = tid; i < m; i += kCT) {
        const int32_t s = sl[i];
        sel_slot[static_cast<int64_t>(b) * m + i] = (s >= 0 && s < n) ? t2s[s] : -1;
    }
    if (early_used && stats) atomicAdd(stats + ECHO_STAT_EARLY_USED, early_used);
    __syncthreads();
    if (tid == 0) {
        c.miss_cnt[b] = static_cast<int32_t>(got);
        if (stats && got) atomicAdd(stats + ECHO_STAT_MISSES, got);
        if (s_flags) set_status(status, static_cast<int>(s_flags));
    }
}

__global__ void __launch_bounds__(256) recall_kernel(const int64_t* __restrict__ tok_off, int64_t n_tokens, int C,
                                                     const int32_t* __restrict__ tok_list,
                                                     const int32_t* __restrict__ slot_list,
                                                     const int32_t* __restrict__ cnt, const uint8_t* host,
                                                     uint8_t* __restrict__ dev, int64_t row_bytes, int32_t* status) {
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    int64_t base, n;
    if (!request_range(tok_off, n_tokens, b, &base, &n)) return;
    int count = cnt[b];
    if (count > C) count = C;
    const int chunks = static_cast<int>(row_bytes / 16);
    constexpr int kRows = 2;  // rows per warp in flight
    for (int i0 = (blockIdx.x * warps + (threadIdx.x >> 5)) * kRows; i0 < count;
         i0 += gridDim.x * warps * kRows) {
        const int4* src[kRows];
        int4* dst[kRows];
        bool ok[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int i = i0 + r;
            ok[r] = false;
            if (i < count) {
                const int32_t tok = tok_list[static_cast<int64_t>(b) * C + i];
                const int32_t slot = slot_list[static_cast<int64_t>(b) * C + i];
                if (tok >= 0 && tok < n && slot >= 0 && slot < C) {
                    ok[r] = true;
                    src[r] = reinterpret_cast<const int4*>(host + (base + tok) * row_bytes);
                    dst[r] = reinterpret_cast<int4*>(dev + (static_cast<int64_t>(b) * C + slot) * row_bytes);
                } else if (lane == 0) {
                    set_status(status, ECHO_ST_BADDATA);
                }
            }
        }
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
}

}  // namespace

cudaError_t launch_early_select(int B, const int64_t* tok_off, int64_t n_tokens, const uint32_t* above, int cap,
                                const echo_cache& c, int32_t* status, uint32_t* stats, cudaStream_t s) {
    const size_t smem = (2 * static_cast<size_t>(c.C / 32) + 1) * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(early_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    early_select_kernel<<<B, kCT, smem, s>>>(tok_off, n_tokens, above, cap, cache_args(c), status, stats);
    return cudaGetLastError();
}

cudaError_t launch_recall(int B, const int64_t* tok_off, int64_t n_tokens, int C, const int32_t* tok_list,
                          const int32_t* slot_list, const int32_t* cnt, const void* host_kv, void* dev_kv,
                          int64_t row_bytes, int32_t* status, cudaStream_t s) {
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    // About one block per SM in all: the host link, not the SMs, bounds the copy,
    // and a small footprint lets the step's other kernels run alongside.
    int gx = (sms + B - 1) / B;
    const int rows_per_block = 16;
    const int gx_max = (C + rows_per_block - 1) / rows_per_block;
    if (gx > gx_max) gx = gx_max;
    if (gx < 1) gx = 1;
    recall_kernel<<<dim3(gx, B), 256, 0, s>>>(tok_off, n_tokens, C, tok_list, slot_list, cnt,
                                              static_cast<const uint8_t*>(host_kv), static_cast<uint8_t*>(dev_kv),
                                              row_bytes, status);
    return cudaGetLastError();
}

}  // namespace echo

namespace echo {

int enqueue_cache_step(int B, const int64_t* tok_off, int64_t n_tokens, const int32_t* sel, int m,
                       const echo_cache* cache, int32_t* sel_slot, int32_t* status, uint32_t* stats,
                       cudaStream_t stream, cudaStream_t copy_stream) {
    const size_t smem = (3 * static_cast<size_t>(cache->C / 32) + 1) * sizeof(uint32_t);
    ECHO_CUDA_OK(cudaFuncSetAttribute(cache_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
    cache_step_kernel<<<B, kCT, smem, stream>>>(tok_off, n_tokens, sel, m, cache_args(*cache), sel_slot, status,
                                                stats);
    ECHO_CUDA_OK(cudaGetLastError());
    const int rc = stream_wait(copy_stream, stream);
    if (rc) return rc;
    ECHO_CUDA_OK(launch_recall(B, tok_off, n_tokens, cache->C, cache->miss_tok, cache->miss_slot, cache->miss_cnt,
                               cache->host_kv, cache->dev_kv, cache->row_bytes, status, copy_stream));
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
    if (cache->C > kMaxSlotsSmem) return ECHO_EUNSUPPORTED;
    return ECHO_OK;
}

}  // namespace echo

extern "C" int echo_cache_step(int B, const int64_t* tok_off, int64_t n_tokens, const int32_t* sel, int m,
                               const echo_cache* cache, int32_t* sel_slot, int32_t* status, uint32_t* stats,
                               echo_stream_t stream, echo_stream_t copy_stream) {
    using namespace echo;
    if (!tok_off || !status) return ECHO_EINVAL;
    const int rc = check_cache_step_args(B, n_tokens, sel, m, cache, sel_slot);
    if (rc) return rc;
    return enqueue_cache_step(B, tok_off, n_tokens, sel, m, cache, sel_slot, status, stats, stream, copy_stream);
}

extern "C" int echo_early_fetch(int B, const int64_t* tok_off, int64_t n_tokens, const uint32_t* above,
                                int early_cap, const echo_cache* cache, int32_t* status, uint32_t* stats,
                                echo_stream_t stream, echo_stream_t copy_stream) {
    using namespace echo;
    if (B <= 0 || n_tokens < 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !status || (n_tokens > 0 && !above)) return ECHO_EINVAL;
    if (n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    int rc = check_cache(cache, B, 0);
    if (rc) return rc;
    if (cache->C > kMaxSlotsSmem) return ECHO_EUNSUPPORTED;
    ECHO_CUDA_OK(launch_early_select(B, tok_off, n_tokens, above, early_cap, *cache, status, stats, stream));
    rc = stream_wait(copy_stream, stream);
    if (rc) return rc;
    ECHO_CUDA_OK(launch_recall(B, tok_off, n_tokens, cache->C, cache->early_tok, cache->early_slot,
                               cache->early_cnt, cache->host_kv, cache->dev_kv, cache->row_bytes, status,
                               copy_stream));
    return ECHO_OK;
}
