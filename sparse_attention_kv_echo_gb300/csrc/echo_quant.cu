// echo_quant.cu -- query quantisation for the FP8 score GEMM.
//
// One warp per (request, head): the 128 query values are read as one float4
// per lane, the absolute maximum is reduced across the warp, and the scale is
// the smallest power of two 2^e with amax <= 448 * 2^e (e >= -126), found
// from the exponent and mantissa bits of amax.  Multiplying by 2^-e is exact,
// so each value is rounded once, to E4M3 round-to-nearest-even (satfinite;
// nothing saturates since |q| * 2^-e <= 448).  The weight is folded with the
// scale so the score kernel applies one factor per head.  The same launch
// zeroes the per-request histogram the score kernel accumulates into.
#include <cuda_fp8.h>

#include "echo_common.cuh"
#include "echo_internal.h"

namespace echo {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ int scale_exponent(float amax) {
    const uint32_t u = __float_as_uint(amax);
    const int ebits = static_cast<int>((u >> 23) & 0xFFu);
    if (amax == 0.0f || ebits == 0xFF) return 0;     // zero row, or non-finite (flagged)
    if (ebits == 0) return -126;                      // subnormal amax: the floor
    const int E = ebits - 127;                        // amax = 1.m * 2^E
    const int e = ((u & 0x7FFFFFu) <= 0x600000u) ? E - 8 : E - 7;  // 1.m <= 1.75 ?
    return e < -126 ? -126 : e;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32) quantize_kernel(int B, const float* __restrict__ q,
                                                                       const float* __restrict__ w,
                                                                       uint8_t* __restrict__ q8,
                                                                       float* __restrict__ qscale,
                                                                       float* __restrict__ wfold,
                                                                       uint32_t* __restrict__ hist,
                                                                       int32_t* __restrict__ cand_cnt,
                                                                       int32_t* status) {
    pdl_launch_dependents();  // the score kernel may start its prologue and key loads
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);  // (request, head) row
    if (gw >= B * ECHO_HEADS) return;
    if (hist && (gw % ECHO_HEADS) == 0) {
        uint32_t* h = hist + static_cast<size_t>(gw / ECHO_HEADS) * 256;
#pragma unroll
        for (int i = 0; i < 8; ++i) h[lane + 32 * i] = 0u;
    }
    if (cand_cnt && (gw % ECHO_HEADS) == 0 && lane == 0) cand_cnt[gw / ECHO_HEADS] = 0;
    const float4 v = reinterpret_cast<const float4*>(q + static_cast<size_t>(gw) * ECHO_DIM)[lane];
    const float wv = w[gw];
    bool bad = !(isfinite(v.x) && isfinite(v.y) && isfinite(v.z) && isfinite(v.w));
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    bad = __any_sync(0xffffffffu, bad) || !isfinite(wv);
    if (bad && lane == 0) set_status(status, ECHO_ST_NAN);
    const int e = scale_exponent(amax);
    const float scale = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(v.x * inv, v.y * inv), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(v.z * inv, v.w * inv), __NV_SATFINITE, __NV_E4M3);
    const uint32_t packed = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    reinterpret_cast<uint32_t*>(q8 + static_cast<size_t>(gw) * ECHO_DIM)[lane] = packed;
    if (lane == 0) {
        qscale[gw] = scale;
        wfold[gw] = __fmul_rn(wv, scale);
    }
}

}  // namespace

cudaError_t launch_quantize(int B, const float* q, const float* w, uint8_t* q8, float* qscale, float* wfold,
                            uint32_t* hist_to_zero, int32_t* cand_cnt_to_zero, int32_t* status, cudaStream_t s) {
    const int rows = B * ECHO_HEADS;
    const int blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const cudaError_t e = prefer_max_shared(quantize_kernel);
    if (e != cudaSuccess) return e;
    quantize_kernel<<<blocks, kWarpsPerBlock * 32, 0, s>>>(B, q, w, q8, qscale, wfold, hist_to_zero,
                                                            cand_cnt_to_zero, status);
    return cudaGetLastError();
}

}  // namespace echo

extern "C" int echo_quantize_q(int B, const float* q, const float* w, uint8_t* q8, float* qscale, float* wfold,
                               uint32_t* hist, int32_t* cand_cnt, int32_t* status, echo_stream_t stream) {
    if (B < 0 || B > ECHO_MAX_REQUESTS) return B < 0 ? ECHO_EINVAL : ECHO_EUNSUPPORTED;
    if (B == 0) return ECHO_OK;
    if (!q || !w || !q8 || !qscale || !wfold) return ECHO_EINVAL;
    if (!echo::is_aligned(q, 16) || !echo::is_aligned(q8, 16) || !echo::is_aligned(w, 4) ||
        !echo::is_aligned(wfold, 16) || !echo::is_aligned(qscale, 4) || !echo::is_aligned(hist, 4) ||
        !echo::is_aligned(cand_cnt, 4))
        return ECHO_EINVAL;
    return echo::launch_quantize(B, q, w, q8, qscale, wfold, hist, cand_cnt, status, stream) == cudaSuccess ? ECHO_OK
                                                                                                 : ECHO_ECUDA;
}
