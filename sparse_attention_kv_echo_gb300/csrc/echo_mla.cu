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
// the split's tokens, 32 at a time, through a four-stage ring of gathered tiles
// (three tiles in flight while one is computed).  Warps 0-3 (thread = head =
// TMEM lane) gather the tiles and run the softmax; warp 4 issues every MMA, so
// the next tile's S runs on the tensor pipe while this tile's softmax runs;
// mbarriers carry the hand-offs (tile landed, S done, P written, P.V done):
//   S = Q K^T   tcgen05.mma kind::f16 (bf16 in, fp32 in TMEM, two S buffers),
//               M = 128 heads, N = 32 tokens, K = 576 in 36 steps; Q is the A
//               operand from TMEM for its first 384 dims (two bf16 per column,
//               lane = head) and from shared memory for the last 192 (128-byte
//               swizzle, K-major), which keeps shared memory for the ring; the
//               gathered KV rows of the tile (same layout, a row per token) are B;
//   softmax     one thread per head reads its S row from TMEM and keeps a
//               running reference max and sum in fp32.  The reference moves
//               only when a score exceeds it by more than 2^8 (P <= 256 in
//               bf16, exact after the final division); O in TMEM is rescaled
//               then.  The P row (bf16) goes to the tile's atoms of the other
//               output half, which S no longer needs;
//   O += P V    M = 128 heads, N = 256 dims (the CTA's half), K = 32 tokens in
//               2 steps: P is A (K-major); V is the tile's value dims read in
//               place as an MN-major B operand (dims contiguous in a 128-byte
//               swizzled row, tokens across rows).
// The splits of one (request, half) -- at most 8, sized on the host so the
// grid runs in the fewest waves of resident clusters -- form one thread-block cluster and combine in distributed shared memory:
// each CTA publishes its (reference max, sum) per head, scales its O rows by
// 2^(m_j - M) / L and stages them in shared memory; CTA r of the cluster then
// sums its share of the heads over the cluster and writes out and lse.  No
// partial result goes to global memory.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "echo_common.cuh"
#include "echo_internal.h"

namespace echo {
namespace {

constexpr int kHeads = ECHO_MLA_HEADS;      // 128
constexpr int kDqk = ECHO_MLA_DQK;          // 576
constexpr int kDv = ECHO_MLA_DV;            // 512
constexpr int kRowBytes = kDqk * 2;         // 1152
constexpr int kTok = 32;                    // tokens per tile
constexpr int kMaxSplits = ECHO_MLA_MAX_SPLITS;      // 8: CTAs of one cluster
constexpr int kSplitMax = ECHO_MLA_MAX_K / ECHO_MLA_MAX_SPLITS;  // 1024: most tokens per split
constexpr int kThreads = 160;               // warps 0-3: one thread per head; warp 4: the MMAs
constexpr int kHeadThreads = 128;
constexpr int kAtoms = kDqk / 64;           // 9 swizzle atoms of 64 bf16 along the 576 dims
constexpr int kChunks = kRowBytes / 16;     // 72 16-byte pieces per row
constexpr int kQTmemAtoms = 6;              // Q atoms 0..5 in TMEM (192 columns), 6..8 in shared memory
constexpr uint32_t kQBytes = (kAtoms - kQTmemAtoms) * kHeads * 128;   // Q in shared memory: 3 x (128 rows x 128 B)
constexpr uint32_t kAtomBytes = kTok * 128;           // one atom of a tile: 32 rows x 128 B
constexpr uint32_t kKBytes = kAtoms * kAtomBytes;     // a tile: 9 atoms
constexpr int kStages = 4;
constexpr uint32_t kTmemCols = 512;                   // Q [0, 192) | S0 [192, 224) | S1 [224, 256) | O [256, 512)
constexpr uint32_t kSCol = kQTmemAtoms * 32;
constexpr uint32_t kOCol = kSCol + 2 * kTok;
static_assert(kOCol + 256 <= kTmemCols, "TMEM columns");
constexpr float kLazy = 8.f;                          // log2 headroom before the reference max moves
constexpr uint64_t kMlaWaitNs = 100000000ull;         // 0.1 s: a tile's MMA takes microseconds

struct MlaCtl {
    uint64_t tile_full[4];  // a stage's tile landed (one arrival per head thread's copies)
    uint64_t s_full[2];     // S of a tile done (per S buffer)
    uint64_t p_full[2];     // P of a tile written, O rescaled (one arrival per head thread)
    uint64_t pv_done[2];    // P.V of a tile done
    uint32_t tmem;       // TMEM base address
    int abort;
    uint32_t valid[kStages];  // tokens of the staged tile with a slot (bit t)
    float m[kHeads];          // this split's reference max (log2 units) per head
    float l[kHeads];          // this split's sum per head
    int32_t slot[kSplitMax];  // the split's slots
};
constexpr uint32_t kCtlBytes = (sizeof(MlaCtl) + 1023u) & ~1023u;
constexpr uint32_t kSmem = kQBytes + kStages * kKBytes + kCtlBytes + 1024 /* alignment */;
static_assert(kSmem <= 227u * 1024u, "MLA shared memory");
static_assert(kHeads * 128 == 4 * kAtomBytes, "P fills the 4 atoms of the other output half");
static_assert(kHeads * 256 * 4 <= kQBytes + (kStages - 1) * kKBytes, "the scaled O rows fit where Q and the ring were");

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major), fp32
// accumulator, shape M x N: D format [4,6) = 1 (f32), A / B format [7,10) /
// [10,13) = 1 (bf16), N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
constexpr uint32_t kIdescS = idesc_bf16_f32(128, kTok);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256) | (1u << 16);  // B (V) MN-major

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzle: 64
// MN elements contiguous in a 128-byte row, K across rows (8-row groups 1024
// bytes apart: stride byte offset), successive 64-element MN groups lbo bytes
// apart (leading byte offset).  Same version and swizzle fields as the K-major one.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t lbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

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

// D[tmem] (+)= A[tmem] x B[smem desc]^T: A (M x K) in TMEM, row m in lane m,
// two 16-bit elements per 32-bit column (the lower K index in the low half).
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st_x32u(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
        " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
        " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Arrive on bar once this thread's earlier cp.async copies have landed (the
// arrival is one of the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
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

// 2^x by the hardware's approximate base-2 exponential (ex2.approx.ftz): the
// softmax weights are rounded to bf16 right after, far coarser than its error.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

// 16-byte asynchronous copy global -> shared; src_bytes 0 writes zeros without reading.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes = 16u) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// The gather of tile `it` of the split into stage buffer sT: 4 threads per row,
// 18 pieces each; rows without a slot are zero-filled (their scores are masked
// and their V rows must be finite).  Warp 0 also records the tile's valid mask.
// sl: the split's slots in shared memory, from token t0 - t_lo on; n: tokens left.
__device__ __forceinline__ void gather_tile(uint32_t sT, const int32_t* sl, int n, const uint8_t* kv, int64_t C,
                                            int tid, uint32_t* valid) {
    const int r = tid >> 2;
    const int32_t slot = (r < n) ? sl[r] : -1;
    const bool ok = slot >= 0 && slot < C;
    const uint8_t* row = kv + (ok ? static_cast<int64_t>(slot) * kRowBytes : 0);
#pragma unroll 6
    for (int c = tid & 3; c < kChunks; c += 4) cp_async_16(sT + sw_offset(r, c, kAtomBytes), row + 16 * c, ok ? 16u : 0u);
    if (tid < 32) {
        const int32_t sj = (tid < n) ? sl[tid] : -1;
        const uint32_t m = __ballot_sync(0xffffffffu, sj >= 0 && sj < C);
        if (tid == 0) *valid = m;
    }
}

// Byte offset of float4 c (0..63) of staged O row h: the 16-byte pieces of a row
// are permuted by h so a warp writing one piece of 32 rows spreads over the banks.
__device__ __forceinline__ uint32_t ostage_offset(int h, int c) {
    return static_cast<uint32_t>(h) * 1024u + (static_cast<uint32_t>(c ^ (h & 7)) << 4);
}

// Grid: B x 2 halves x splits CTAs, split index fastest; cluster = the splits
// of one (request, half).
__global__ void __launch_bounds__(kThreads, 1)
    mla_split_kernel(int k, int split_tokens, const uint16_t* __restrict__ q, const int32_t* __restrict__ sel_slot,
                     const uint8_t* __restrict__ dev_kv, int64_t C, float scale_log2, float* __restrict__ out,
                     float* __restrict__ lse, int32_t* status) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    // Q atoms 6..8 [3 x 128 rows] | tile stages 0..3 (later, from the start: the scaled O rows) | control
    const uint32_t sQ = base, sT0 = sQ + kQBytes;
    uint8_t* const gT0 = gbase + kQBytes;
    MlaCtl* ctl = reinterpret_cast<MlaCtl*>(gT0 + kStages * kKBytes);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int splits = static_cast<int>(cluster.num_blocks());
    const int split = static_cast<int>(cluster.block_rank());
    const int half = (blockIdx.x / splits) & 1;
    const int b = blockIdx.x / (2 * splits);
    const int t_lo = split * split_tokens, t_hi = min(k, t_lo + split_tokens);
    const int n_tok = max(0, t_hi - t_lo);
    const uint8_t* kv = dev_kv + static_cast<int64_t>(b) * C * kRowBytes;
    // P of a tile lives in the 4 atoms of the other output half (128 rows x 128 B)
    const uint32_t p_off = static_cast<uint32_t>(4 * (1 - half)) * kAtomBytes;
    const uint32_t v_off = static_cast<uint32_t>(4 * half) * kAtomBytes;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(smem_addr(&ctl->tile_full[i]), kHeadThreads);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&ctl->s_full[i]), 1);
            mbar_init(smem_addr(&ctl->p_full[i]), kHeadThreads);
            mbar_init(smem_addr(&ctl->pv_done[i]), 1);
        }
        ctl->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(&ctl->tmem), kTmemCols);
        tmem_relinquish();
    }
    // Q atoms 6..8 of the request (row h = head h) into shared memory, piece-major
    {
        const uint8_t* qb = reinterpret_cast<const uint8_t*>(q) + static_cast<int64_t>(b) * kHeads * kRowBytes;
        constexpr int kQc = kChunks - 8 * kQTmemAtoms;  // 24 pieces per row
#pragma unroll 8
        for (int g = tid; g < kHeads * kQc; g += kThreads) {
            const int h = g / kQc, c = g - h * kQc;
            cp_async_16(sQ + sw_offset(h, c, kHeads * 128u),
                        qb + static_cast<int64_t>(h) * kRowBytes + 16 * (8 * kQTmemAtoms + c));
        }
        cp_async_commit();
    }
    // the split's slots (one read of the selection)
    {
        const int32_t* sl = sel_slot + static_cast<int64_t>(b) * k + t_lo;
        for (int i = tid; i < n_tok; i += kThreads) ctl->slot[i] = sl[i];
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // Q's pieces landed
    fence_proxy_async_smem();
    __syncthreads();
    const int tiles = (n_tok + kTok - 1) / kTok;
    const bool head = tid < kHeadThreads;
    if (head)
        for (int t = 0; t < min(tiles, kStages - 1); ++t) {  // the first three tiles of the ring
            gather_tile(sT0 + static_cast<uint32_t>(t) * kKBytes, ctl->slot + t * kTok, n_tok - t * kTok, kv, C, tid,
                        &ctl->valid[t]);
            cp_async_arrive_noinc(smem_addr(&ctl->tile_full[t]));
        }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;  // a head warp's TMEM lanes
    // Q atoms 0..5 into TMEM: each head thread its row, 32 columns (64 bf16) per store
    if (head) {
        const uint4* qrow = reinterpret_cast<const uint4*>(q + (static_cast<int64_t>(b) * kHeads + tid) * kDqk);
#pragma unroll 1
        for (int a = 0; a < kQTmemAtoms; ++a) {
            uint32_t u[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 v = __ldg(qrow + 8 * a + j);
                u[4 * j] = v.x;
                u[4 * j + 1] = v.y;
                u[4 * j + 2] = v.z;
                u[4 * j + 3] = v.w;
            }
            tmem_st_x32u(tmem + lane_base + 32u * a, u);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    volatile int* abort = &ctl->abort;
    float m = -INFINITY, l = 0.f;  // a head thread's head: reference max (log2-scaled scores) and sum

    if (tid == kHeadThreads) {
        // ---- warp 4, lane 0: S(it) as soon as tile it lands, then P.V(it - 1) once P(it - 1) is written
        for (int it = 0; it <= tiles && !*abort; ++it) {
            if (it < tiles) {
                const int st = it % kStages;
                const uint32_t sT = sT0 + static_cast<uint32_t>(st) * kKBytes;
                const uint32_t sCol = kSCol + static_cast<uint32_t>(it & 1) * kTok;
                if (!mla_wait(smem_addr(&ctl->tile_full[st]), static_cast<uint32_t>(it / kStages) & 1u, abort)) {
                    *abort = 1;
                    break;
                }
                fence_proxy_async_smem();  // the head threads' copies, seen by the MMAs
                tc_fence_after();
#pragma unroll 4
                for (int kk = 0; kk < kQTmemAtoms * 4; ++kk) {
                    const uint32_t a = static_cast<uint32_t>(kk >> 2), off = static_cast<uint32_t>(kk & 3) * 32u;
                    mma_bf16_ta(tmem + sCol, tmem + 8u * kk, sw128_kmajor_desc(sT + a * kAtomBytes + off), kIdescS,
                                kk > 0 ? 1u : 0u);
                }
#pragma unroll 4
                for (int kk = kQTmemAtoms * 4; kk < kAtoms * 4; ++kk) {
                    const uint32_t a = static_cast<uint32_t>(kk >> 2), off = static_cast<uint32_t>(kk & 3) * 32u;
                    mma_bf16(tmem + sCol, sw128_kmajor_desc(sQ + (a - kQTmemAtoms) * kHeads * 128u + off),
                             sw128_kmajor_desc(sT + a * kAtomBytes + off), kIdescS, 1u);
                }
                mma_commit(smem_addr(&ctl->s_full[it & 1]));
            }
            if (it > 0) {
                const int pt = it - 1;
                if (!mla_wait(smem_addr(&ctl->p_full[pt & 1]), static_cast<uint32_t>(pt >> 1) & 1u, abort)) {
                    *abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t pT = sT0 + static_cast<uint32_t>(pt % kStages) * kKBytes;
#pragma unroll
                for (int kk = 0; kk < kTok / 16; ++kk)
                    mma_bf16(tmem + kOCol, sw128_kmajor_desc(pT + p_off + kk * 32u),
                             sw128_mnmajor_desc(pT + v_off + kk * 2048u, kAtomBytes), kIdescPV,
                             (pt > 0 || kk > 0) ? 1u : 0u);
                mma_commit(smem_addr(&ctl->pv_done[pt & 1]));
            }
        }
    } else if (head) {
        // ---- warps 0-3: softmax of tile it, P into the tile's dead atoms, then the gather of tile it + 3
        for (int it = 0; it < tiles; ++it) {
            const int st = it % kStages;
            uint8_t* const gT = gT0 + st * kKBytes;
            const uint32_t sCol = kSCol + static_cast<uint32_t>(it & 1) * kTok;
            if (!mla_wait(smem_addr(&ctl->s_full[it & 1]), static_cast<uint32_t>(it >> 1) & 1u, abort)) {
                *abort = 1;
                break;
            }
            // P.V(it - 1) done: O may be rescaled and tile it - 1's stage takes tile it + 3
            if (it > 0 && !mla_wait(smem_addr(&ctl->pv_done[(it - 1) & 1]), static_cast<uint32_t>((it - 1) >> 1) & 1u,
                                    abort)) {
                *abort = 1;
                break;
            }
            tc_fence_after();
            {
                float s[kTok];
                tmem_ld_x32(tmem + lane_base + sCol, s);
                const uint32_t vm = ctl->valid[st];
#pragma unroll
                for (int t = 0; t < kTok; ++t) s[t] = ((vm >> t) & 1u) ? s[t] : -INFINITY;
                float mx[kTok / 2];
#pragma unroll
                for (int t = 0; t < kTok / 2; ++t) mx[t] = fmaxf(s[2 * t], s[2 * t + 1]);
#pragma unroll
                for (int w = kTok / 4; w >= 1; w >>= 1)
#pragma unroll
                    for (int t = 0; t < w; ++t) mx[t] = fmaxf(mx[t], mx[t + w]);
                const float tmx = mx[0] * scale_log2;
                const bool need = tmx > m + kLazy;  // also m = -inf with a valid token
                // tcgen05.ld / st are warp-collective: the whole warp rescales when any head moves
                const bool warp_moves = __any_sync(0xffffffffu, need);
                float corr = 1.f;
                if (warp_moves && tmx > m) {
                    corr = ex2_approx(m - tmx);  // 0 when m = -inf
                    m = tmx;
                }
                const float neg_m = (m == -INFINITY) ? 0.f : -m;
                float part[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t packed[kTok / 2];
#pragma unroll
                for (int t = 0; t < kTok; t += 2) {
                    const float p0 = ex2_approx(fmaf(s[t], scale_log2, neg_m));
                    const float p1 = ex2_approx(fmaf(s[t + 1], scale_log2, neg_m));
                    const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                    part[(t >> 1) & 3] += __low2float(pb) + __high2float(pb);  // the values the MMA uses
                    packed[t >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
                }
                l = l * corr + ((part[0] + part[1]) + (part[2] + part[3]));
                uint8_t* prow = gT + p_off + tid * 128;
#pragma unroll
                for (int c = 0; c < kTok / 8; ++c)
                    *reinterpret_cast<uint4*>(prow + ((c ^ (tid & 7)) << 4)) =
                        make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
                if (it > 0 && warp_moves) {  // O holds earlier tiles: bring it to the new reference
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
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_addr(&ctl->p_full[it & 1]));
            if (it + kStages - 1 < tiles) {  // tile it + 3 into the stage tile it - 1 had
                const int t = it + kStages - 1, ts = t % kStages;
                gather_tile(sT0 + static_cast<uint32_t>(ts) * kKBytes, ctl->slot + t * kTok, n_tok - t * kTok, kv, C,
                            tid, &ctl->valid[ts]);
                cp_async_arrive_noinc(smem_addr(&ctl->tile_full[ts]));
            }
        }
        // the last P.V done
        if (!*abort && tiles > 0 &&
            !mla_wait(smem_addr(&ctl->pv_done[(tiles - 1) & 1]), static_cast<uint32_t>((tiles - 1) >> 1) & 1u, abort))
            *abort = 1;
    }
    __syncthreads();
    tc_fence_after();
    const bool failed = *abort != 0;
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (failed) {  // every thread sees it
        if (tid == 0) set_status(status, ECHO_ST_TIMEOUT);
        m = -INFINITY;  // this split then adds nothing
        l = 0.f;
    }
    // ---- combine over the cluster.  Every CTA passes the same three cluster
    // barriers whatever happened above.
    const int hh = head ? tid : 0;  // warp 4 takes no head
    if (head) {
        ctl->m[tid] = m;
        ctl->l[tid] = l;
    }
    cluster.sync();  // (1) every split's (m, l) is published
    float mj[kMaxSplits], lj[kMaxSplits];
#pragma unroll
    for (int j = 0; j < kMaxSplits; ++j) {  // all loads in flight at once
        mj[j] = (j < splits) ? cluster.map_shared_rank(ctl->m, j)[hh] : -INFINITY;
        lj[j] = (j < splits) ? cluster.map_shared_rank(ctl->l, j)[hh] : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxSplits; ++j) M = fmaxf(M, mj[j]);
    float L = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxSplits; ++j)
        if (M > -INFINITY && mj[j] > -INFINITY) L += lj[j] * exp2f(mj[j] - M);
    const float f = (M > -INFINITY && L > 0.f && m > -INFINITY) ? exp2f(m - M) / L : 0.f;
    // this head's O row, scaled, staged at the start of shared memory (the MMAs are done with it)
    if (head) {
        const bool have_o = !failed && tiles > 0;
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
            float o[32];
            if (have_o) {
                tmem_ld_x32(tmem + lane_base + kOCol + c, o);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(gbase + ostage_offset(tid, (c + j) >> 2)) =
                    make_float4(o[j] * f, o[j + 1] * f, o[j + 2] * f, o[j + 3] * f);
        }
    }
    cluster.sync();  // (2) every split's scaled O is staged
    // CTA `split` sums heads [h0, h1) over the cluster: one float4 of a head row per thread and pass
    {
        const int per = (kHeads + splits - 1) / splits;
        const int h0 = split * per, h1 = min(kHeads, h0 + per);
        for (int g = tid; g < (h1 - h0) * 64; g += kThreads) {
            const int h = h0 + (g >> 6), c = g & 63;
            float4 v[kMaxSplits];
#pragma unroll
            for (int j = 0; j < kMaxSplits; ++j)  // all loads in flight at once
                v[j] = (j < splits) ? *reinterpret_cast<const float4*>(cluster.map_shared_rank(
                                          reinterpret_cast<float*>(gbase + ostage_offset(h, c)), j))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 acc = v[0];
#pragma unroll
            for (int j = 1; j < kMaxSplits; ++j) {
                acc.x += v[j].x;
                acc.y += v[j].y;
                acc.z += v[j].z;
                acc.w += v[j].w;
            }
            *reinterpret_cast<float4*>(out + (static_cast<int64_t>(b) * kHeads + h) * kDv + half * 256 + 4 * c) = acc;
        }
        if (half == 0 && tid >= h0 && tid < h1)  // this thread's head is in the share: its lse
            lse[static_cast<int64_t>(b) * kHeads + tid] =
                (M > -INFINITY && L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
    cluster.sync();  // (3) no CTA leaves while another reads its shared memory
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// How many clusters of `size` CTAs of this kernel the device holds at once
// (queried once per device and size).
int max_active_clusters(int size) {
    static int cache[64][kMaxSplits + 1];
    static bool init = false;
    if (!init) {
        for (auto& row : cache)
            for (int& v : row) v = -1;
        init = true;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    int& v = cache[dev][size];
    if (v < 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(size));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(size);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mla_split_kernel, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        v = n;
    }
    return v;
}

// Splits of the selection for B requests: the cluster size (at most 8) whose
// grid of B x 2 clusters finishes soonest -- waves of resident clusters times
// the tiles of a split plus about two tiles of fixed work (Q, combine).
void mla_plan(int B, int k, int* split_tokens, int* splits) {
    long best = -1;
    for (int size = kMaxSplits; size >= 1; --size) {
        int per = (k + size - 1) / size;
        per = (per + kTok - 1) / kTok * kTok;
        if (per > kSplitMax) break;
        const int n = (k + per - 1) / per;
        const int active = max_active_clusters(n);
        if (active <= 0) continue;
        const long waves = (2L * B + active - 1) / active;
        const long cost = waves * (per / kTok + 2);
        if (best < 0 || cost < best) {
            best = cost;
            *split_tokens = per;
            *splits = n;
        }
    }
    if (best < 0) {  // no residency figure: 8 splits
        *split_tokens = ((k + kMaxSplits - 1) / kMaxSplits + kTok - 1) / kTok * kTok;
        *splits = (k + *split_tokens - 1) / *split_tokens;
    }
}

int launch_mla(int B, int k, const uint16_t* q, const int32_t* sel_slot, const void* dev_kv, int64_t C, float scale,
               float* out, float* lse, int32_t* status, cudaStream_t stream) {
    ECHO_CUDA_OK(prefer_max_shared(mla_split_kernel));
    ECHO_CUDA_OK(cudaFuncSetAttribute(mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kSmem)));
    int split_tokens = 0, splits = 0;
    mla_plan(B, k, &split_tokens, &splits);
    const float scale_log2 = scale * 1.4426950408889634f;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B * 2 * splits));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ECHO_CUDA_OK(cudaLaunchKernelEx(&cfg, mla_split_kernel, k, split_tokens, q, sel_slot,
                                    static_cast<const uint8_t*>(dev_kv), C, scale_log2, out, lse, status));
    return ECHO_OK;
}

}  // namespace echo

extern "C" int echo_mla_decode(int B, int k, const uint16_t* q, const int32_t* sel_slot, const void* dev_kv, int64_t C,
                               float scale, float* out, float* lse, int32_t* status, echo_stream_t stream) {
    using namespace echo;
    if (B <= 0 || k <= 0 || C <= 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS || k > ECHO_MLA_MAX_K) return ECHO_EUNSUPPORTED;
    if (!q || !sel_slot || !dev_kv || !out || !lse || !status) return ECHO_EINVAL;
    if (!is_aligned(q, 16) || !is_aligned(dev_kv, 16) || !is_aligned(out, 16)) return ECHO_EINVAL;
    return launch_mla(B, k, q, sel_slot, dev_kv, C, scale, out, lse, status, static_cast<cudaStream_t>(stream));
}
