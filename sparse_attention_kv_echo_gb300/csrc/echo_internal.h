// echo_internal.h -- host-side helpers shared by the libecho translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "echo.h"


namespace echo {

inline bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// SM count of the current device.
int sm_count();

// 2-D tensor map over a row-major byte matrix [rows, inner_bytes] with a box
// of [box_rows, box_inner] bytes and the 128-byte swizzle.  0 on success.
int encode_tmap_bytes_2d(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                         uint32_t box_inner, uint32_t box_rows);

// 1-D tensor map over n 4-byte elements (float32 or int32), box of `box`
// elements (box * 4 a multiple of 16), no swizzle, zero fill out of range.
int encode_tmap_1d(CUtensorMap* map, const void* base, bool is_float, uint64_t n, uint32_t box);

// Make `to` wait for everything enqueued so far on `from` (no-op when equal).
int stream_wait(cudaStream_t to, cudaStream_t from);

// Host-side checks of an echo_cache for B requests and selections of up to m tokens.
int check_cache(const echo_cache* c, int B, int m);

// Launchers shared across translation units.
cudaError_t launch_quantize(int B, const float* q, const float* w, uint8_t* q8, float* qscale, float* wfold,
                            uint32_t* hist_to_zero, int32_t* cand_cnt_to_zero, int32_t* status, cudaStream_t s);
cudaError_t launch_recall(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, int C, const int32_t* tok_list,
                          const int32_t* slot_list, const int32_t* cnt, const void* host_kv, void* dev_kv,
                          int64_t row_bytes, int32_t* status, cudaStream_t s, bool programmatic);

// Ask for the largest shared-memory carveout.  An SM reconfigures its
// L1/shared split only when it drains, so a block of a kernel that needs little
// shared memory, resident under a small carveout, would keep a large-smem block
// of a concurrent kernel (top-k, scores) off that SM until it finishes.
template <class Kernel>
cudaError_t prefer_max_shared(Kernel kernel) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

constexpr int kMaxSlots = 1 << 19;   // slots per request: per-slot-word tables fit shared memory

// Enqueue helpers shared by the decode calls and the prefill block call.
int launch_topk(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, int64_t row0, int64_t W, const float* scores, int k,
                const uint32_t* hist, float* theta_hat, float alpha, int32_t* sel_idx, float* kth, int32_t* status,
                uint32_t* stats, cudaStream_t stream);
// Prefill rows' top-k (select_kernel, one block per row): row b of R at position row0 + b selects
// among scores[b * W + s], s <= row0 + b; theta_hat[0] shifts the rows' histograms and is not updated.
int launch_select_rows(int R, int64_t row0, int64_t W, const float* scores, int k, const uint32_t* hist,
                       float* theta_hat, int32_t* sel_idx, float* kth, int32_t* status, uint32_t* stats,
                       cudaStream_t stream);
int check_cache_step_args(int B, int64_t n_tokens, const int32_t* sel, int m, const echo_cache* cache,
                          const int32_t* sel_slot);
int enqueue_cache_step(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, const int32_t* sel,
                       int m,
                       const uint32_t* above, int early_cap, const echo_cache* cache, int32_t* sel_slot,
                       int32_t* status, uint32_t* stats, cudaStream_t stream, cudaStream_t copy_stream,
                       bool resolved, bool hold_early, bool lazy);

}  // namespace echo

#define ECHO_CUDA_OK(expr)                               \
    do {                                                 \
        if ((expr) != cudaSuccess) return ECHO_ECUDA;    \
    } while (0)
