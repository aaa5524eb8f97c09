// echo_append.cu -- one new token per request: the offload write path.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2,
// panel "One layer, one step: free -> allocate -> recall": the host holds every
// token's KV row, so an evicted row needs no write-back.  A decode step's new
// token therefore goes to the host pool when it is made; its indexer key joins
// the FP8 key array the score kernel scans (the DeepSeek-V3.2 lightning
// indexer: E4M3 keys, one fp32 scale per token).  The row also takes the
// request's lowest free cache slot when there is one, so the next step finds
// it resident instead of recalling the row it just wrote.
//
// One block per request:
//   key     thread d < 128 holds component d; block max |k| -> scale =
//           amax / 448 (fp32), code = E4M3 RN satfinite of k / scale;
//   slot    the first free bit of the request's free-bit words (a block-wide
//           minimum over the words), claimed in freebits / tok2slot / slot2tok;
//   row     16-byte pieces of the KV row to the host pool (zero-copy stores
//           through the pool's device alias) and to the slot's device row.
#include <cuda_fp8.h>

#include <climits>

#include "echo_common.cuh"
#include "echo_internal.h"

namespace echo {
namespace {

constexpr int kAT = 256;  // threads per request

__global__ void __launch_bounds__(kAT)
    append_kernel(const int64_t* __restrict__ tok_off, int64_t* __restrict__ tok_end, int64_t n_tokens,
                  const float* __restrict__ k_new, const uint8_t* __restrict__ kv_new, int64_t row_bytes,
                  uint8_t* __restrict__ k8, float* __restrict__ ks, int32_t* __restrict__ tok2slot,
                  int32_t* __restrict__ slot2tok, uint32_t* __restrict__ freebits, uint8_t* host, uint8_t* dev, int C,
                  int32_t* status) {
    __shared__ float red[kAT / 32];
    __shared__ int s_slot;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t lo = tok_off[b], hi = tok_off[b + 1], pos = tok_end[b];
    if (lo < 0 || hi < lo || hi > n_tokens || pos < lo || pos > hi) {  // the same for every thread
        if (tid == 0) set_status(status, ECHO_ST_BADDATA);
        return;
    }
    if (pos == hi) {  // the region is full
        if (tid == 0) set_status(status, ECHO_ST_FULL);
        return;
    }
    // ---- the key
    const float v = (tid < ECHO_DIM) ? k_new[static_cast<int64_t>(b) * ECHO_DIM + tid] : 0.f;
    if (__syncthreads_or(!isfinite(v))) {
        if (tid == 0) set_status(status, ECHO_ST_NAN);
        return;
    }
    float a = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) red[warp] = a;
    if (tid == 0) s_slot = INT_MAX;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int w = 1; w < kAT / 32; ++w) amax = fmaxf(amax, red[w]);
    const float scale = amax / 448.0f;
    if (tid < ECHO_DIM) {
        uint8_t code = 0;
        if (amax > 0.f) code = static_cast<uint8_t>(__nv_cvt_float_to_fp8(v / scale, __NV_SATFINITE, __NV_E4M3));
        k8[pos * ECHO_DIM + tid] = code;
    }
    if (tid == 0) ks[pos] = scale;
    // ---- the lowest free slot of the request
    const int words = C / 32;
    uint32_t* fb = freebits + static_cast<int64_t>(b) * words;
    for (int w = tid; w < words; w += kAT) {
        const uint32_t bits = fb[w];
        if (bits) {
            atomicMin(&s_slot, w * 32 + __ffs(static_cast<int>(bits)) - 1);
            break;  // a thread's later words hold higher slots
        }
    }
    __syncthreads();
    const int slot = (s_slot < C) ? s_slot : -1;
    if (tid == 0 && slot >= 0) {
        fb[slot >> 5] &= ~(1u << (slot & 31));
        tok2slot[pos] = slot;
        slot2tok[static_cast<int64_t>(b) * C + slot] = static_cast<int32_t>(pos - lo);
        tok_end[b] = pos + 1;
    } else if (tid == 0) {
        tok_end[b] = pos + 1;
    }
    // ---- the row: host pool, and the slot's device row
    const int chunks = static_cast<int>(row_bytes / 16);
    const int4* src = reinterpret_cast<const int4*>(kv_new + static_cast<int64_t>(b) * row_bytes);
    int4* hdst = reinterpret_cast<int4*>(host + pos * row_bytes);
    int4* ddst = slot >= 0 ? reinterpret_cast<int4*>(dev + (static_cast<int64_t>(b) * C + slot) * row_bytes) : nullptr;
    for (int c = tid; c < chunks; c += kAT) {
        const int4 x = src[c];
        hdst[c] = x;
        if (ddst) ddst[c] = x;
    }
}

}  // namespace
}  // namespace echo

extern "C" int echo_append_tokens(int B, const int64_t* tok_off, int64_t* tok_end, int64_t n_tokens,
                                  const float* k_new, const void* kv_new, uint8_t* k8, float* ks,
                                  const echo_cache* cache, int32_t* status, echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || n_tokens <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !tok_end || !k_new || !kv_new || !k8 || !ks || !status) return ECHO_EINVAL;
    const int rc = check_cache(cache, B, 0);
    if (rc) return rc;
    if (!is_aligned(kv_new, 16)) return ECHO_EINVAL;
    append_kernel<<<B, kAT, 0, static_cast<cudaStream_t>(stream)>>>(
        tok_off, tok_end, n_tokens, k_new, static_cast<const uint8_t*>(kv_new), cache->row_bytes, k8, ks,
        cache->tok2slot, cache->slot2tok, cache->freebits,
        static_cast<uint8_t*>(const_cast<void*>(cache->host_kv)), static_cast<uint8_t*>(cache->dev_kv), cache->C,
        status);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}
