// echo_pool.cu -- a per-worker GPU cache shared by every request of the batch.
//
// "OSDI'26 Artifact Evaluation for ECHO ...", sections "Baselines under
// evaluation" and the decode-server options: ECHO's device cache is one pool
// of NSA_DEV_CACHE_SIZE slots (260 000 by default) per layer for the worker,
// not a fixed slot range per request.  The pool is the cache of one "request"
// that spans every token of the batch (rows [0, n_tokens), token ids global),
// so the step's early fetch, cache step and recall run unchanged on it.  These
// kernels translate between the per-request calls (scores, top-k) and that
// view:
//   pool_above   the early set's marks: the per-request above-threshold words
//                that echo_index_scores wrote (request b's from word
//                4 * (floor(tok_off[b] / 128) + b), bit j of word w = token
//                32 w + j of the request) become global marks (bit j of word w
//                = token 32 w + j of the batch), residents of the pool left
//                out; and the pool's free bits are snapshotted;
//   pool_select  the per-request selections [B, k] (ascending, -1 padded)
//                become one ascending list of global token ids, padding last;
//   pool_slots   the pool step's slots of that list go back to [B, k].
#include "echo_common.cuh"
#include "echo_internal.h"

namespace echo {
namespace {

constexpr int kPT = 256;
constexpr int kPer = 4;  // selection entries per thread of the mapping kernel

__global__ void __launch_bounds__(kPT)
    pool_above_kernel(int B, const int64_t* __restrict__ tok_off, const int64_t* __restrict__ tok_end, int64_t n_tokens,
                      const uint32_t* __restrict__ above_req, const int32_t* __restrict__ tok2slot,
                      const uint32_t* __restrict__ freebits, uint32_t* __restrict__ free_snap, int pool_words,
                      uint32_t* __restrict__ above_pool, int32_t* status) {
    const int b = blockIdx.x, tid = threadIdx.x;
    if (b == 0)
        for (int w = tid; w < pool_words; w += kPT) free_snap[w] = freebits[w];
    int64_t lo, hi;
    if (!seg_bounds(tok_off, tok_end, n_tokens, b, &lo, &hi)) {
        if (tid == 0) set_status(status, ECHO_ST_BADDATA);
        return;
    }
    const uint32_t* ab = above_req + 4 * (lo / 128 + b);
    const int64_t n = hi - lo;
    const int nw = static_cast<int>((n + 31) >> 5);
    for (int w = tid; w < nw; w += kPT) {
        uint32_t bits = ab[w];
        if (w == nw - 1 && (n & 31)) bits &= (1u << (n & 31)) - 1u;
        while (bits) {
            const int j = __ffs(static_cast<int>(bits)) - 1;
            bits &= bits - 1u;
            const int64_t g = lo + 32 * static_cast<int64_t>(w) + j;
            if (tok2slot[g] < 0) atomicOr(above_pool + (g >> 5), 1u << (g & 31));
        }
    }
}

// Request b's valid selection entries (ascending, before the padding): their
// number, and their offset in the batch-wide list (a block-wide scan over the
// requests in one block).
__device__ __forceinline__ void pool_offsets(int B, const int32_t* sel, int k, int32_t* s_off, uint32_t* scan) {
    uint32_t run = 0;
    for (int b0 = 0; b0 < B; b0 += kPT) {
        const int b = b0 + static_cast<int>(threadIdx.x);
        uint32_t c = 0;
        if (b < B) {
            // the entries before the first -1 (top-k pads at the end)
            int lo = 0, hi = k;
            const int32_t* row = sel + static_cast<int64_t>(b) * k;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (row[mid] >= 0)
                    lo = mid + 1;
                else
                    hi = mid;
            }
            c = static_cast<uint32_t>(lo);
        }
        uint32_t tot;
        const uint32_t ex = block_exclusive_scan<kPT>(c, scan, &tot);
        if (b < B) s_off[b] = static_cast<int32_t>(run + ex);
        run += tot;
        __syncthreads();
    }
    if (threadIdx.x == 0) s_off[B] = static_cast<int32_t>(run);
    __syncthreads();
}

// sel [B, k] (request-local) -> sel_pool [B * k] (global, ascending, padding
// last); or, with to_req, slot_pool [B * k] -> sel_slot [B, k].  Every block
// scans the requests' counts (B binary searches), then maps its kPT * kPer
// entries.
__global__ void __launch_bounds__(kPT)
    pool_map_kernel(int B, const int64_t* __restrict__ tok_off, const int32_t* __restrict__ sel, int k, bool to_req,
                    int32_t* __restrict__ pool_list, int32_t* __restrict__ sel_slot) {
    extern __shared__ int32_t s_off[];  // [B + 1]
    __shared__ uint32_t scan[kPT / 32 + 1];
    pool_offsets(B, sel, k, s_off, scan);
    const int64_t total = static_cast<int64_t>(B) * k;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kPT * kPer;
    const int64_t i1 = min(total, i0 + static_cast<int64_t>(kPT) * kPer);
    for (int64_t i = i0 + threadIdx.x; i < i1; i += kPT) {
        const int b = static_cast<int>(i / k), j = static_cast<int>(i - static_cast<int64_t>(b) * k);
        const int cnt = s_off[b + 1] - s_off[b];
        if (!to_req) {
            if (j < cnt) pool_list[s_off[b] + j] = static_cast<int32_t>(tok_off[b] + sel[i]);
            if (i >= s_off[B]) pool_list[i] = -1;
        } else {
            sel_slot[i] = (j < cnt) ? pool_list[s_off[b] + j] : -1;
        }
    }
}

}  // namespace
}  // namespace echo

extern "C" int echo_pool_above(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                               const uint32_t* above_req, const echo_cache* pool, uint32_t* above_pool,
                               int32_t* status, echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || n_tokens <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS || n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    if (!tok_off || !above_req || !above_pool || !status) return ECHO_EINVAL;
    const int rc = check_cache(pool, 1, 0);
    if (rc) return rc;
    if (!pool->free_snap) return ECHO_EINVAL;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t words = 4 * static_cast<size_t>(n_tokens / 128 + 1);  // echo_above_words(1, n_tokens)
    ECHO_CUDA_OK(cudaMemsetAsync(above_pool, 0, words * sizeof(uint32_t), s));
    pool_above_kernel<<<B, kPT, 0, s>>>(B, tok_off, tok_end, n_tokens, above_req, pool->tok2slot, pool->freebits,
                                        pool->free_snap, pool->C / 32, above_pool, status);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}

extern "C" int echo_pool_select(int B, const int64_t* tok_off, const int32_t* sel, int k, int32_t* sel_pool,
                                echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || k <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !sel || !sel_pool) return ECHO_EINVAL;
    const int blocks = static_cast<int>((static_cast<int64_t>(B) * k + kPT * kPer - 1) / (kPT * kPer));
    pool_map_kernel<<<blocks, kPT, (B + 1) * sizeof(int32_t), static_cast<cudaStream_t>(stream)>>>(
        B, tok_off, sel, k, false, sel_pool, nullptr);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}

extern "C" int echo_pool_slots(int B, const int32_t* sel, int k, const int32_t* slot_pool, int32_t* sel_slot,
                               echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || k <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!sel || !slot_pool || !sel_slot) return ECHO_EINVAL;
    const int blocks = static_cast<int>((static_cast<int64_t>(B) * k + kPT * kPer - 1) / (kPT * kPer));
    pool_map_kernel<<<blocks, kPT, (B + 1) * sizeof(int32_t), static_cast<cudaStream_t>(stream)>>>(
        B, nullptr, sel, k, true, const_cast<int32_t*>(slot_pool), sel_slot);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}
