// echo_prefill.cu -- chunked prefill, one block of query rows at a time.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2,
// panel "Prefill: one-round histogram": while the indexer scores query block
// i+1, the tokens of block i are fetched; the real kernel bins scores into
// 256 bins over the top 8 bits of each score shifted by the predicted
// threshold.
//
// echo_prefill_block enqueues, on `stream`:
//   quantize_kernel      the block's R query rows (each row is its own "request")
//   prefill_score_kernel row r at position row0 + r scores keys [0, row0 + r]
//                        (causal, itself included) into scores[r*W + s], 8 rows per
//                        key tile, with the per-row histogram shifted by the block's
//                        threshold (echo_prefill_scores.cu)
//   select_kernel        one block per row: exact top-k of the row, its boundary
//                        bin taken from the row's histogram, the row's scores read
//                        once (the tokens above the bin into a bitmap, the bin's
//                        entries into shared memory; echo_select.cu)
//   union_mark_kernel    marks every token some row selected
//   union_compact_kernel ascending list of the marked tokens (the block's
//                        selection for the cache), its bit words, and the
//                        block threshold update: EMA (alpha) of the last row's
//                        k-th score
//   cache_step_kernel    free / allocate for the union (after the previous
//                        block's recall has read its lists),
// and the recall of the misses on `copy_stream`, so that the next block's
// scoring on `stream` overlaps it.
#include <mutex>

#include "echo_common.cuh"
#include "echo_internal.h"

namespace echo {
namespace {

constexpr int kPT = 1024;

__global__ void union_mark_kernel(const int32_t* __restrict__ sel, int64_t total, uint8_t* __restrict__ mark,
                                  int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t s = sel[i];
        if (s >= 0 && s < n) mark[s] = 1;
    }
}

__device__ __forceinline__ float block_ema(float theta, float kth, float alpha) {
    if (isinf(kth) && kth < 0) return theta;
    if (isinf(theta)) return kth;
    return __fadd_rn(__fmul_rn(alpha, kth), __fmul_rn(__fsub_rn(1.0f, alpha), theta));
}

__global__ void __launch_bounds__(kPT) union_compact_kernel(const uint8_t* __restrict__ mark, int64_t n, int64_t m,
                                                            int32_t* __restrict__ list, uint32_t* union_bits,
                                                            int32_t* count, int64_t* tok_off2, int64_t n_keys,
                                                            const float* kth, int R, float* theta, float alpha) {
    __shared__ uint32_t scan[40];
    uint32_t done = 0;
    const int64_t words = (n + 31) / 32;
    for (int64_t w0 = 0; w0 < words; w0 += kPT) {
        const int64_t w = w0 + threadIdx.x;
        uint32_t bits = 0;
        if (w < words) {
            for (int j = 0; j < 32; ++j) {
                const int64_t s = 32 * w + j;
                if (s < n && mark[s]) bits |= 1u << j;
            }
            if (union_bits) union_bits[w] = bits;
        }
        uint32_t tot;
        uint32_t pos = done + block_exclusive_scan<kPT>(__popc(bits), scan, &tot);
        while (bits) {
            const int j = __ffs(bits) - 1;
            bits &= bits - 1;
            if (pos < m) list[pos] = static_cast<int32_t>(32 * w + j);
            ++pos;
        }
        done += tot;
    }
    for (int64_t i = done + threadIdx.x; i < m; i += kPT) list[i] = -1;
    if (threadIdx.x == 0) {
        *count = static_cast<int32_t>(done);
        tok_off2[0] = 0;
        tok_off2[1] = n_keys;
        if (theta) *theta = block_ema(*theta, kth[R - 1], alpha);
    }
}

struct PrefillWs {
    uint8_t* q8;
    float* qscale;
    float* wfold;
    uint8_t* mark;
    int64_t* tok_off2;
};

size_t prefill_ws_bytes(int R, int64_t W) {
    const size_t r = static_cast<size_t>(R);
    return round_up(r * ECHO_HEADS * ECHO_DIM, 256) + 2 * round_up(r * ECHO_HEADS * 4, 256) +
           round_up(static_cast<size_t>(W), 256) + 256;
}

// tok_off2 | q8 | qscale | wfold | mark.  The request range the recall reads
// sits at the same place whatever R and W are, so the blocks before a call's
// wait on the copy stream never write where an earlier call's recall (of a
// prompt with another W, sharing the workspace) still reads.
PrefillWs carve(void* ws, int R, int64_t W) {
    (void)W;
    uint8_t* p = static_cast<uint8_t*>(ws);
    const size_t r = static_cast<size_t>(R);
    PrefillWs o;
    o.tok_off2 = reinterpret_cast<int64_t*>(p);
    p += 256;
    o.q8 = p;
    p += round_up(r * ECHO_HEADS * ECHO_DIM, 256);
    o.qscale = reinterpret_cast<float*>(p);
    p += round_up(r * ECHO_HEADS * 4, 256);
    o.wfold = reinterpret_cast<float*>(p);
    p += round_up(r * ECHO_HEADS * 4, 256);
    o.mark = p;
    return o;
}

}  // namespace
}  // namespace echo

extern "C" size_t echo_prefill_workspace_size(int R, int64_t W) {
    if (R <= 0 || W <= 0) return 0;
    return echo::prefill_ws_bytes(R, W);
}

extern "C" int echo_prefill_block(int R, int64_t row0, int64_t n_keys, const float* q, const float* w,
                                  const uint8_t* k8, const float* ks, int k, float* theta_hat, float alpha,
                                  float* scores, int64_t W, uint32_t* hist, int32_t* sel_idx, float* kth,
                                  int32_t* union_list, int32_t* union_count, uint32_t* union_bits,
                                  const echo_cache* cache, int32_t* sel_slot, void* ws, size_t ws_bytes,
                                  int32_t* status, uint32_t* stats, echo_stream_t stream, echo_stream_t copy_stream) {
    using namespace echo;
    if (R <= 0 || row0 < 0 || n_keys <= 0 || k <= 0 || W <= 0) return ECHO_EINVAL;
    if (R > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!q || !w || !k8 || !ks || !theta_hat || !scores || !hist || !sel_idx || !kth || !union_list ||
        !union_count || !ws || !status)
        return ECHO_EINVAL;
    if (row0 + R > n_keys || W < row0 + R) return ECHO_EINVAL;
    if (W > (1ll << 31) || n_keys >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    if (!is_aligned(q, 16) || !is_aligned(k8, 16) || !is_aligned(ws, 256)) return ECHO_EINVAL;
    if (ws_bytes < prefill_ws_bytes(R, W)) return ECHO_ECAPACITY;
    if (cache) {
        const int rc = check_cache_step_args(1, n_keys, union_list, static_cast<int>(W), cache, sel_slot);
        if (rc) return rc;
    }
    const PrefillWs p = carve(ws, R, W);
    if (launch_quantize(R, q, w, p.q8, p.qscale, p.wfold, hist, nullptr, status, stream) != cudaSuccess) return ECHO_ECUDA;
    int rc = echo_prefill_scores(R, row0, n_keys, p.q8, p.wfold, k8, ks, scores, W, theta_hat, hist, status, stream);
    if (rc) return rc;
    rc = launch_topk(R, nullptr, nullptr, 0, row0, W, scores, k, hist, theta_hat, alpha, sel_idx, kth, status, stats, stream);
    if (rc) return rc;
    const int64_t n = row0 + R;
    ECHO_CUDA_OK(cudaMemsetAsync(p.mark, 0, static_cast<size_t>(n), stream));
    const int64_t total = static_cast<int64_t>(R) * k;
    const int sms = sm_count();
    if (sms <= 0) return ECHO_ECUDA;
    int64_t grid = (total + 255) / 256;
    if (grid > 8 * sms) grid = 8 * sms;
    ECHO_CUDA_OK(prefer_max_shared(union_mark_kernel));
    ECHO_CUDA_OK(prefer_max_shared(union_compact_kernel));
    union_mark_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(sel_idx, total, p.mark, n);
    ECHO_CUDA_OK(cudaGetLastError());
    if (cache) {
        // the previous block's recall, still running on copy_stream, reads the request range
        // (workspace tok_off2, which union_compact_kernel writes next) and the miss lists (which
        // the cache step rewrites): both wait for it.  Only the tiny union kernels follow the
        // wait; the quantiser, the scores and top-k above overlap that recall.
        rc = stream_wait(stream, copy_stream);
        if (rc) return rc;
    }
    union_compact_kernel<<<1, kPT, 0, stream>>>(p.mark, n, W, union_list, union_bits, union_count, p.tok_off2,
                                                n_keys, kth, R, theta_hat, alpha);
    ECHO_CUDA_OK(cudaGetLastError());
    if (!cache) return ECHO_OK;
    // the union holds at most the n = row0 + R tokens the block's rows see, the rest of the list is
    // padding: the cache step walks the first n entries and the padding's slots are set to -1 here
    if (W > n) ECHO_CUDA_OK(cudaMemsetAsync(sel_slot + n, 0xFF, static_cast<size_t>(W - n) * sizeof(int32_t), stream));
    return enqueue_cache_step(1, p.tok_off2, nullptr, n_keys, union_list, static_cast<int>(n), nullptr, 0, cache, sel_slot,
                              status, stats, stream, copy_stream, false, false, false);
}

// ---------------------------------------------------------------------------
// Allocation-free prefill block.
//
// Some callers cannot hand this library a workspace: a serving runtime whose
// device memory is carved up once at start-up and forbids new allocations
// afterwards, an embedder that has no allocator of its own to call, or a
// latency-critical thread where cudaMalloc's implicit device synchronisation
// is not acceptable.  For them, echo_prefill_block_static runs the same
// prefill block as echo_prefill_block, with its workspace in the fixed device
// array below instead of caller memory.  The array is part of the library
// image: every GPU that loads the library holds ECHO_PREFILL_STATIC_SCRATCH_BYTES
// of device memory for it until the process exits.
// ---------------------------------------------------------------------------
namespace echo {
namespace {

static __device__ __align__(256) uint8_t g_prefill_scratch[ECHO_PREFILL_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};   // the context the address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The current context, through the runtime's driver entry point (no libcuda link).
CUcontext current_context() {
    static CtxGetCurrentFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    }
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of the scratch array on the current device, looked up with
// that device current and remembered per device; looked up again when the
// device's context is a new one (after cudaDeviceReset the library image, and
// the array with it, is loaded anew).  A lookup is not made while `stream` is
// being captured into a graph: ECHO_EINVAL then.
int static_scratch(cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ECHO_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return ECHO_EUNSUPPORTED;
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
            cudaGetLastError();
            return ECHO_ECUDA;
        }
        if (cs != cudaStreamCaptureStatusNone) return ECHO_EINVAL;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return ECHO_ECUDA;
        }
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return ECHO_OK;
}

}  // namespace
}  // namespace echo

extern "C" int echo_prefill_block_static(int R, int64_t row0, int64_t n_keys, const float* q, const float* w,
                                         const uint8_t* k8, const float* ks, int k, float* theta_hat, float alpha,
                                         float* scores, int64_t W, uint32_t* hist, int32_t* sel_idx, float* kth,
                                         int32_t* union_list, int32_t* union_count, uint32_t* union_bits,
                                         const echo_cache* cache, int32_t* sel_slot, int32_t* status,
                                         uint32_t* stats, echo_stream_t stream, echo_stream_t copy_stream) {
    using namespace echo;
    if (R <= 0 || W <= 0) return ECHO_EINVAL;
    if (prefill_ws_bytes(R, W) > static_cast<size_t>(ECHO_PREFILL_STATIC_SCRATCH_BYTES)) return ECHO_ETOOLARGE;
    void* scratch = nullptr;
    const int rc = static_scratch(static_cast<cudaStream_t>(stream), &scratch);
    if (rc) return rc;
    // Everything the block needs zeroed (the union marks) it clears itself on
    // the stream; the rest of the scratch is written before it is read.
    return echo_prefill_block(R, row0, n_keys, q, w, k8, ks, k, theta_hat, alpha, scores, W, hist, sel_idx, kth,
                              union_list, union_count, union_bits, cache, sel_slot, scratch,
                              static_cast<size_t>(ECHO_PREFILL_STATIC_SCRATCH_BYTES), status, stats, stream,
                              copy_stream);
}
