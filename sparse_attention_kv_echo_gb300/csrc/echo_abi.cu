// echo_abi.cu -- host-side plumbing of the libecho C ABI: TMA descriptor
// encoding through the driver entry point, stream ordering, argument checks
// and small queries.
#include <string.h>

#include "echo_internal.h"

namespace echo {

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

int encode_tmap_bytes_2d(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                         uint32_t box_inner, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return ECHO_ECUDA;
    if (!is_aligned(base, 16) || inner_bytes % 16 != 0 || rows == 0 || rows > (1ull << 31)) return ECHO_EINVAL;
    const cuuint64_t dims[2] = {inner_bytes, rows};
    const cuuint64_t strides[1] = {inner_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    memset(map, 0, sizeof(*map));
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ECHO_OK : ECHO_ECUDA;
}

int encode_tmap_1d(CUtensorMap* map, const void* base, bool is_float, uint64_t n, uint32_t box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return ECHO_ECUDA;
    if (!is_aligned(base, 16) || n == 0 || n > (1ull << 31) || (box * 4u) % 16u != 0) return ECHO_EINVAL;
    const cuuint64_t dims[1] = {n};
    const cuuint64_t strides[1] = {n * 4};  // not read for rank 1, but the encoder wants the array
    const cuuint32_t boxd[1] = {box};
    const cuuint32_t estr[1] = {1};
    memset(map, 0, sizeof(*map));
    const CUresult r = fn(map, is_float ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_INT32, 1,
                          const_cast<void*>(base), dims, strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ECHO_OK : ECHO_ECUDA;
}

int stream_wait(cudaStream_t to, cudaStream_t from) {
    if (to == from) return ECHO_OK;
    cudaEvent_t ev;
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return ECHO_ECUDA;
    cudaError_t e = cudaEventRecord(ev, from);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(to, ev, 0);
    cudaEventDestroy(ev);
    return e == cudaSuccess ? ECHO_OK : ECHO_ECUDA;
}

int check_cache(const echo_cache* c, int B, int m) {
    if (!c) return ECHO_EINVAL;
    if (!c->tok2slot || !c->slot2tok || !c->freebits || !c->miss_tok || !c->miss_slot || !c->miss_cnt ||
        !c->early_tok || !c->early_slot || !c->early_cnt || !c->host_kv || !c->dev_kv)
        return ECHO_EINVAL;
    if (c->C <= 0 || c->C % 32 != 0) return ECHO_ECAPACITY;
    if (m > c->C) return ECHO_ECAPACITY;
    if (c->row_bytes <= 0 || c->row_bytes % 16 != 0) return ECHO_EUNSUPPORTED;
    if (!is_aligned(c->host_kv, 16) || !is_aligned(c->dev_kv, 16)) return ECHO_EINVAL;
    if (static_cast<int64_t>(B) * c->C > (1ll << 31)) return ECHO_EUNSUPPORTED;
    return ECHO_OK;
}

}  // namespace echo

extern "C" {

int echo_host_device_alias(const void* host_ptr, const void** device_ptr) {
    if (!host_ptr || !device_ptr) return ECHO_EINVAL;
    void* d = nullptr;
    if (cudaHostGetDevicePointer(&d, const_cast<void*>(host_ptr), 0) != cudaSuccess) {
        cudaGetLastError();
        return ECHO_ECUDA;
    }
    *device_ptr = d;
    return ECHO_OK;
}

int echo_device_sm_count(void) { return echo::sm_count(); }

}  // extern "C"
