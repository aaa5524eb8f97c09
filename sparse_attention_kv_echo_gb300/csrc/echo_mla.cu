// echo_mla.cu -- sparse MLA decode attention over the slots the cache step gave
// the selected tokens (the consumer of the GPU cache).
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2:
// a decode step attends over the k selected tokens only, whose KV rows the GPU
// cache holds.  The attention is DeepSeek-V3.2's sparse MLA in its absorbed
// form: one latent KV row of 576 bf16 per token (512 latent + 64 rotary dims)
// shared by the 128 query heads,
//   s_t = scale * q[h] . kv[slot_t]   (576 dims),   out[h] = softmax(s) . kv[slot_t][0:512].
//
// CTA (request b, output half, split of the selection) takes the 128 heads and
// the split's tokens, 16 at a time:
//   S = Q K^T   tcgen05.mma kind::f16 (bf16 in, fp32 in TMEM), M = 128 heads,
//               N = 16 tokens, K = 576 in 36 steps; Q stays in shared memory
//               (128-byte swizzle, K-major), the 16 gathered KV rows are B;
//   softmax     one thread per head reads its S row from TMEM, keeps the
//               running max and sum in fp32, writes its P row (bf16) to shared
//               memory and rescales its O row in TMEM when the max grows;
//   O += P V    M = 128 heads, N = 256 dims (the CTA's half), K = 16 tokens:
//               P is A; the tile's value dims, transposed in shared memory into
//               the same K-major swizzled layout (a row per dim), are B.
// Every operand uses the one K-major 128-byte-swizzle layout.
// Each split leaves its unnormalised O and its (max, sum) per head; a second
// kernel combines the splits.
#include <cuda_bf16.h>

#include "echo_common.cuh"
#include "echo_internal.h"

namespace echo {
namespace {

constexpr int kHeads = ECHO_MLA_HEADS;      // 128
constexpr int kDqk = ECHO_MLA_DQK;          // 576
constexpr int kDv = ECHO_MLA_DV;            // 512
constexpr int kRowBytes = kDqk * 2;         // 1152
constexpr int kTok = 16;                    // tokens per tile
constexpr int kSplit = ECHO_MLA_SPLIT;      // tokens per CTA
constexpr int kThreads = 128;               // one thread per head
constexpr int kAtoms = kDqk / 64;           // 9 swizzle atoms of 64 bf16 along the 576 dims
constexpr int kChunks = kRowBytes / 16;     // 72 16-byte pieces per row
constexpr uint32_t kQBytes = kAtoms * kHeads * 128;   // Q: 9 x (128 rows x 128 B)
constexpr uint32_t kKBytes = kAtoms * kTok * 128;     // tile: 9 x (16 rows x 128 B)
constexpr uint32_t kPBytes = kHeads * 128;            // P: 128 rows x 128 B (first 32 B used)
constexpr uint32_t kVBytes = 256 * 128;               // V^T of the half: 256 rows x 128 B (first 32 B used)
constexpr uint32_t kTmemCols = 512;                   // S [0, 32) | O [32, 288)
constexpr uint32_t kOCol = 32;
constexpr uint64_t kMlaWaitNs = 100000000ull;         // 0.1 s: a tile's MMA takes microseconds

struct MlaCtl {
    uint64_t s_bar;      // S MMA of the tile done
    uint64_t pv_bar;     // PV MMA of the tile done
    uint32_t tmem;       // TMEM base address
    int abort;
};
constexpr uint32_t kSmem = kQBytes + kKBytes + kPBytes + kVBytes + 1024 /* control */ + 1024 /* alignment */;
static_assert(kSmem <= 227u * 1024u, "MLA shared memory");

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major), fp32
// accumulator, shape M x N: D format [4,6) = 1 (f32), A / B format [7,10) /
// [10,13) = 1 (bf16), N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
constexpr uint32_t kIdescS = idesc_bf16_f32(128, kTok);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256);

// Bounded wait on an mbarrier phase (this kernel's own limit).
__device__ __forceinline__ bool mla_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > kMlaWaitNs) return false;
    }
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, float (&r)[32]) {
    uint32_t u[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
          "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]),
          "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]),
          "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __uint_as_float(u[i]);
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const float (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
        " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
        " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(r[0])), "r"(__float_as_uint(r[1])), "r"(__float_as_uint(r[2])),
        "r"(__float_as_uint(r[3])), "r"(__float_as_uint(r[4])), "r"(__float_as_uint(r[5])),
        "r"(__float_as_uint(r[6])), "r"(__float_as_uint(r[7])), "r"(__float_as_uint(r[8])),
        "r"(__float_as_uint(r[9])), "r"(__float_as_uint(r[10])), "r"(__float_as_uint(r[11])),
        "r"(__float_as_uint(r[12])), "r"(__float_as_uint(r[13])), "r"(__float_as_uint(r[14])),
        "r"(__float_as_uint(r[15])), "r"(__float_as_uint(r[16])), "r"(__float_as_uint(r[17])),
        "r"(__float_as_uint(r[18])), "r"(__float_as_uint(r[19])), "r"(__float_as_uint(r[20])),
        "r"(__float_as_uint(r[21])), "r"(__float_as_uint(r[22])), "r"(__float_as_uint(r[23])),
        "r"(__float_as_uint(r[24])), "r"(__float_as_uint(r[25])), "r"(__float_as_uint(r[26])),
        "r"(__float_as_uint(r[27])), "r"(__float_as_uint(r[28])), "r"(__float_as_uint(r[29])),
        "r"(__float_as_uint(r[30])), "r"(__float_as_uint(r[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte piece c of row r of a swizzled K-major tile whose 64-element atoms
// (rows x 128 B) are atom_bytes apart.
__device__ __forceinline__ uint32_t sw_offset(int r, int c, uint32_t atom_bytes) {
    return static_cast<uint32_t>(c >> 3) * atom_bytes + static_cast<uint32_t>(r) * 128u +
           (static_cast<uint32_t>((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_split_kernel(int k, const uint16_t* __restrict__ q, const int32_t* __restrict__ sel_slot,
                     const uint8_t* __restrict__ dev_kv, int64_t C, float scale_log2, float* __restrict__ opart,
                     float* __restrict__ mpart, float* __restrict__ lpart, int splits, int32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    // Q [9 atoms x 128 rows] | tile [9 atoms x 16 rows] | P [128 rows] | V^T [256 rows] | control
    const uint32_t sQ = base, sK = sQ + kQBytes, sP = sK + kKBytes, sV = sP + kPBytes;
    uint8_t* const gK = gbase + kQBytes;
    uint8_t* const gP = gK + kKBytes;
    uint8_t* const gV = gP + kPBytes;
    MlaCtl* ctl = reinterpret_cast<MlaCtl*>(gV + kVBytes);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int split = blockIdx.x % splits;
    const int half = (blockIdx.x / splits) & 1;
    const int b = blockIdx.x / (2 * splits);
    const int t_lo = split * kSplit, t_hi = min(k, t_lo + kSplit);
    const int32_t* sl = sel_slot + static_cast<int64_t>(b) * k;
    const uint8_t* kv = dev_kv + static_cast<int64_t>(b) * C * kRowBytes;

    if (tid == 0) {
        mbar_init(smem_addr(&ctl->s_bar), 1);
        mbar_init(smem_addr(&ctl->pv_bar), 1);
        ctl->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(&ctl->tmem), kTmemCols);
        tmem_relinquish();
    }
    // Q of the request: row h = head h, 72 pieces
    {
        const uint8_t* qrow = reinterpret_cast<const uint8_t*>(q) + (static_cast<int64_t>(b) * kHeads + tid) * kRowBytes;
        for (int c = 0; c < kChunks; ++c) cp_async_16(sQ + sw_offset(tid, c, kHeads * 128u), qrow + 16 * c);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;  // this warp's TMEM lanes
    volatile int* abort = &ctl->abort;
    bool failed = false;
    uint32_t pending = 0, phase = 0;  // the barrier and phase a timed-out wait was on

    float m = -INFINITY, l = 0.f;  // this thread's head: running max (of log2-scaled scores) and sum
    const int tiles = (t_hi - t_lo + kTok - 1) / kTok;
    for (int it = 0; it < tiles; ++it) {
        const int t0 = t_lo + it * kTok;
        // ---- gather the tile's KV rows (8 threads per row, 9 pieces each); rows
        // without a slot are zero (their scores are masked in the softmax)
        {
            const int r = tid >> 3;
            const int i = t0 + r;
            const int32_t slot = (i < t_hi) ? sl[i] : -1;
            if (slot >= 0 && slot < C) {
                const uint8_t* row = kv + static_cast<int64_t>(slot) * kRowBytes;
                for (int c = tid & 7; c < kChunks; c += 8) cp_async_16(sK + sw_offset(r, c, kTok * 128u), row + 16 * c);
            } else {
                for (int c = tid & 7; c < kChunks; c += 8)
                    *reinterpret_cast<uint4*>(gK + sw_offset(r, c, kTok * 128u)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        cp_async_wait_all();
        __syncthreads();
        // ---- V^T of this half: row n = value dim 256 * half + n, its 16 tokens in
        // the first 32 bytes (two 16-byte pieces, swizzled like every operand)
        {
#pragma unroll
            for (int jn = 0; jn < 2; ++jn) {
                const int n = 2 * tid + jn;
                const int d = 256 * half + n;
                uint32_t w[8];
#pragma unroll
                for (int t = 0; t < kTok; t += 2) {
                    const uint16_t* r0 = reinterpret_cast<const uint16_t*>(gK + sw_offset(t, d >> 3, kTok * 128u));
                    const uint16_t* r1 = reinterpret_cast<const uint16_t*>(gK + sw_offset(t + 1, d >> 3, kTok * 128u));
                    w[t >> 1] = static_cast<uint32_t>(r0[d & 7]) | (static_cast<uint32_t>(r1[d & 7]) << 16);
                }
                uint8_t* vrow = gV + n * 128;
                *reinterpret_cast<uint4*>(vrow + (((0 ^ (n & 7)) & 7) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(vrow + (((1 ^ (n & 7)) & 7) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // ---- S = Q K^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll 4
            for (int kk = 0; kk < kAtoms * 4; ++kk) {
                const uint32_t a = static_cast<uint32_t>(kk >> 2), off = static_cast<uint32_t>(kk & 3) * 32u;
                mma_bf16(tmem, sw128_kmajor_desc(sQ + a * kHeads * 128u + off),
                         sw128_kmajor_desc(sK + a * kTok * 128u + off), kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit(smem_addr(&ctl->s_bar));
        }
        if (__syncthreads_or(!mla_wait(smem_addr(&ctl->s_bar), it & 1, abort))) {  // block-uniform
            failed = true;
            pending = smem_addr(&ctl->s_bar);
            phase = it & 1;
            break;
        }
        tc_fence_after();
        // ---- online softmax of this head's row; P row to shared memory
        {
            float s[16];
            {
                uint32_t u[16];
                tmem_ld_x16(tmem + lane_base, u);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; ++t) s[t] = __uint_as_float(u[t]);
            }
            float mx = m;
#pragma unroll
            for (int t = 0; t < kTok; ++t) {
                const bool v = t0 + t < t_hi && sl[t0 + t] >= 0 && sl[t0 + t] < C;
                s[t] = v ? s[t] * scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[t]);
            }
            const float corr = (mx == -INFINITY) ? 1.f : exp2f(m - mx);
            float sum = 0.f;
            uint32_t packed[8];
#pragma unroll
            for (int t = 0; t < kTok; t += 2) {
                const float p0 = (mx == -INFINITY) ? 0.f : exp2f(s[t] - mx);
                const float p1 = (mx == -INFINITY) ? 0.f : exp2f(s[t + 1] - mx);
                const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                sum += __low2float(pb) + __high2float(pb);  // the sum of the values the MMA uses
                packed[t >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
            }
            l = l * corr + sum;
            m = mx;
            uint8_t* prow = gP + tid * 128;
            *reinterpret_cast<uint4*>(prow + (((0 ^ (tid & 7)) & 7) << 4)) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
            *reinterpret_cast<uint4*>(prow + (((1 ^ (tid & 7)) & 7) << 4)) =
                make_uint4(packed[4], packed[5], packed[6], packed[7]);
            // O holds earlier tiles: bring it to the new max.  tcgen05.ld / st are
            // warp-collective, so the whole warp rescales when any of its heads must.
            if (it > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < 256; c += 32) {
                    float o[32];
                    tmem_ld_x32(tmem + lane_base + kOCol + c, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= corr;
                    tmem_st_x32(tmem + lane_base + kOCol + c, o);
                }
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        // ---- O += P V (this CTA's 256 dims), one K step of 16 tokens
        if (tid == 0) {
            tc_fence_after();
            mma_bf16(tmem + kOCol, sw128_kmajor_desc(sP), sw128_kmajor_desc(sV), kIdescPV, it > 0 ? 1u : 0u);
            mma_commit(smem_addr(&ctl->pv_bar));
        }
        // the tile, P and V^T are free again once the PV MMA is done
        if (__syncthreads_or(!mla_wait(smem_addr(&ctl->pv_bar), it & 1, abort))) {
            failed = true;
            pending = smem_addr(&ctl->pv_bar);
            phase = it & 1;
            break;
        }
        tc_fence_after();
    }
    cp_async_wait_all();
    if (failed) {  // every thread took this branch; give the late MMA one more bounded wait
        if (tid == 0) {
            set_status(status, ECHO_ST_TIMEOUT);
            mla_wait(pending, phase, abort);
            *abort = 1;
        }
    }
    __syncthreads();
    // ---- the split's unnormalised O, max and sum of each head
    if (!*abort) {
        float* orow = opart + ((static_cast<int64_t>(b) * splits + split) * kHeads + tid) * kDv + half * 256;
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
            float o[32];
            tmem_ld_x32(tmem + lane_base + kOCol + c, o);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(orow + c + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
        }
        if (half == 0) {
            mpart[(static_cast<int64_t>(b) * splits + split) * kHeads + tid] = m;
            lpart[(static_cast<int64_t>(b) * splits + split) * kHeads + tid] = l;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// The splits of one (request, head): out = sum_j 2^(m_j - M) O_j / L with
// L = sum_j 2^(m_j - M) l_j (scores in log2 units), lse = ln(2) (M + log2 L).
__global__ void __launch_bounds__(128)
    mla_combine_kernel(int splits, const float* __restrict__ opart, const float* __restrict__ mpart,
                       const float* __restrict__ lpart, float* __restrict__ out, float* __restrict__ lse) {
    const int bh = blockIdx.x, b = bh / kHeads, h = bh % kHeads;
    float M = -INFINITY;
    for (int j = 0; j < splits; ++j) M = fmaxf(M, mpart[(static_cast<int64_t>(b) * splits + j) * kHeads + h]);
    float L = 0.f;
    for (int j = 0; j < splits; ++j) {
        const int64_t e = (static_cast<int64_t>(b) * splits + j) * kHeads + h;
        if (mpart[e] > -INFINITY) L += lpart[e] * exp2f(mpart[e] - M);
    }
    for (int d = threadIdx.x; d < kDv; d += blockDim.x) {
        float acc = 0.f;
        for (int j = 0; j < splits; ++j) {
            const int64_t e = (static_cast<int64_t>(b) * splits + j) * kHeads + h;
            if (mpart[e] > -INFINITY) acc += exp2f(mpart[e] - M) * opart[e * kDv + d];
        }
        out[static_cast<int64_t>(bh) * kDv + d] = (L > 0.f) ? acc / L : 0.f;
    }
    if (threadIdx.x == 0) lse[bh] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace

int mla_splits(int k) { return (k + kSplit - 1) / kSplit; }

size_t mla_workspace_bytes(int B, int k) {
    const size_t parts = static_cast<size_t>(B) * mla_splits(k) * kHeads;
    return parts * (kDv + 2) * sizeof(float) + 256;
}

int launch_mla(int B, int k, const uint16_t* q, const int32_t* sel_slot, const void* dev_kv, int64_t C, float scale,
               float* out, float* lse, void* ws, int32_t* status, cudaStream_t stream) {
    const int splits = mla_splits(k);
    const size_t parts = static_cast<size_t>(B) * splits * kHeads;
    float* opart = static_cast<float*>(ws);
    float* mpart = opart + parts * kDv;
    float* lpart = mpart + parts;
    ECHO_CUDA_OK(prefer_max_shared(mla_split_kernel));
    ECHO_CUDA_OK(cudaFuncSetAttribute(mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kSmem)));
    const float scale_log2 = scale * 1.4426950408889634f;
    mla_split_kernel<<<B * 2 * splits, kThreads, kSmem, stream>>>(k, q, sel_slot, static_cast<const uint8_t*>(dev_kv),
                                                                  C, scale_log2, opart, mpart, lpart, splits, status);
    ECHO_CUDA_OK(cudaGetLastError());
    mla_combine_kernel<<<B * kHeads, 128, 0, stream>>>(splits, opart, mpart, lpart, out, lse);
    ECHO_CUDA_OK(cudaGetLastError());
    return ECHO_OK;
}

}  // namespace echo

extern "C" size_t echo_mla_workspace_size(int B, int k) {
    if (B <= 0 || k <= 0) return 0;
    return echo::mla_workspace_bytes(B, k);
}

extern "C" int echo_mla_decode(int B, int k, const uint16_t* q, const int32_t* sel_slot, const void* dev_kv, int64_t C,
                               float scale, float* out, float* lse, void* ws, size_t ws_bytes, int32_t* status,
                               echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || k <= 0 || C <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!q || !sel_slot || !dev_kv || !out || !lse || !ws || !status) return ECHO_EINVAL;
    if (!is_aligned(q, 16) || !is_aligned(dev_kv, 16) || !is_aligned(out, 16) || !is_aligned(ws, 16))
        return ECHO_EINVAL;
    if (ws_bytes < mla_workspace_bytes(B, k)) return ECHO_ECAPACITY;
    return launch_mla(B, k, q, sel_slot, dev_kv, C, scale, out, lse, ws, status, static_cast<cudaStream_t>(stream));
}
