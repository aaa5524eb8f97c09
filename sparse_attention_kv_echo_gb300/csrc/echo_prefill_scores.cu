// echo_prefill_scores.cu -- the indexer scores of a block of prefill query rows, four rows per MMA.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2,
// panel "Prefill: one-round histogram": every query row of the block scores the
// keys before it (causal), and each row's scores are binned by the top 8 bits
// of score - theta_hat (one block threshold) for its top-k.
//
//   scores[r * W + t] = ks[t] * sum_h wfold[r, h] * max(0, sum_d q8[r, h, d] * k8[t, d]),
//   t <= row0 + r (row r sits at position row0 + r, itself included).
//
// A decode request has one query against many keys; a prefill block has many
// query rows against the same keys, so the score is a real GEMM.  Four
// consecutive rows form a group whose 4 x 64 head vectors are the B operand of
// one tcgen05.mma kind::f8f6f4 (M = 128 keys, N = 256, K = 32, four K-steps), so
// a key tile is read once per four rows and one MMA does the work of four.
//
// A unit is 8 consecutive rows: all of TMEM (512 columns) holds their 8 x 64
// head sums for one 128-key tile, as two accumulators of 256 columns, so a key
// tile leaves L2 once per 8 rows.  (N = 128 -- four MMAs of two rows -- measured
// slower: an MMA of N <= 128 costs nearly as much as one of N = 256.)
//
// Design (one persistent CTA per SM, 576 threads, warp-specialised):
//   warp 0      TMA producer: 128-key x 128-byte tiles into a 6-stage ring
//               (128-byte swizzle); the unit's 512 q8 rows (64 KB, two boxes)
//               into the q buffer when the unit changes.
//   warp 1      TMEM owner (512 columns) and single-thread MMA issuer: per
//               tile, two MMAs (rows 0-3 and 4-7 of the unit) of four K-steps.
//   warps 2-17  sixteen epilogue warps, four per TMEM lane quarter; each owns
//               two rows of the unit and, per thread, one key of the tile:
//               tcgen05.ld of the rows' head sums 32 columns at a time, ReLU,
//               the weighted sum in packed f32x2 FMAs over four chains, times
//               the key scale, the causal mask, store, and a warp-private
//               histogram per row (match.any groups, red.shared counts)
//               flushed with global atomics when the unit changes.  An
//               accumulator goes back to the MMA as soon as the eight warps
//               that drain it have loaded their columns.
// The epilogue is the bound, not the tensor pipe: per (key, row) it issues a
// ReLU and half an FMA pair per head against the MMA's 256 FLOPs, so it gets
// as many warps as 96 registers a thread allow (four per scheduler) to hide
// the TMEM-load and FMA latencies.
// The tiles of all units (ceil(keys of the unit's last row / 128) each) form
// one list; CTA c takes a contiguous share.  The keys of the prompt's prefix
// stay in L2 (at most 102400 x 132 B), so the kernel is bound by the tensor pipe
// and its epilogue rather than by HBM.
#include "echo_common.cuh"
#include "echo_internal.h"

namespace echo {
namespace {

constexpr int kN = 256;                                // the MMA's N: 4 rows x 64 heads
constexpr int kRows = 8;                               // rows per unit
constexpr int kG = kN / ECHO_HEADS;                    // rows per MMA (4)
constexpr int kAcc = kRows / kG;                       // accumulators (MMAs per tile): 2
constexpr int kTmemCols = kAcc * kN;                   // 512
constexpr int kStages = 6;                             // key ring
constexpr int kTileM = 128;                            // keys per tile (MMA M)
constexpr int kKeyBytes = kTileM * ECHO_DIM;           // 16 KB
constexpr int kQBytes = kRows * ECHO_HEADS * ECHO_DIM; // 64 KB: a unit's q8
constexpr int kQBox = 256;                             // q8 rows per TMA box
constexpr int kEpiWarps = 16;                          // four per TMEM lane quarter
constexpr int kSlots = kEpiWarps / 4;                  // epilogue warps per lane quarter
constexpr int kRPW = kRows / kSlots;                   // rows of a unit per epilogue warp (2)
constexpr int kAccWarps = 4 * (kG / kRPW);             // epilogue warps that drain one accumulator (8)
constexpr int kPieces = 2 * kRPW;                      // 32-column TMEM loads per warp and tile
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr uint32_t kIdesc = idesc_e4m3_f32(kTileM, kN);
static_assert(kG % kRPW == 0, "a warp's rows sit in one accumulator");

struct PfArgs {
    int R;                   // rows of the block
    int units;               // ceil(R / 8)
    int64_t row0;            // position of row 0
    int64_t n_keys;
    int64_t W;               // row stride of scores
    const float* ks;         // [n_keys] key scales
    const float* wfold;      // [R, 64]
    float* scores;           // [R, W]
    const float* theta_hat;  // one block threshold (may be null)
    uint32_t* hist;          // [R, 256] (may be null)
    int32_t* status;
};

struct __align__(128) PfCtl {
    float wv[kEpiWarps][kRPW][ECHO_HEADS];       // each epilogue warp's copy of its rows' weights
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t qfull;
    uint64_t qempty;
    uint64_t accfull[kAcc];
    uint64_t accempty[kAcc];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    uint32_t scan[kThreads / 32 + 1];
    uint32_t hist[kEpiWarps][kRPW][256];         // per epilogue warp, per row
};

// keys | q8 | PfCtl | tstart[units + 1] (int32)
__host__ __device__ constexpr size_t pf_smem_bytes(int units) {
    return 1024 + static_cast<size_t>(kStages) * kKeyBytes + kQBytes + sizeof(PfCtl) +
           4 * static_cast<size_t>(units + 1);
}

// Keys seen by the last row of unit u (the unit's longest row).
__device__ __forceinline__ int64_t unit_keys(const PfArgs& a, int u) {
    const int last = min(a.R, kRows * u + kRows) - 1;
    return a.row0 + last + 1;
}

// Largest unit u in [0, U) whose first tile is <= t.
__device__ __forceinline__ int find_unit(const int32_t* tstart, int U, uint32_t t) {
    int lo = 0, hi = U - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<uint32_t>(tstart[mid]) <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}


// d = a * b + c on two fp32 lanes at once.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}

__device__ __forceinline__ float sum2(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return __fadd_rn(lo, hi);
}

// 32 lanes x 32 consecutive 32-bit columns; thread i of the warp gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Adds w[h] * max(0, x[h]) for 32 heads into kChains pair accumulators (FMA pair m of the piece
// goes to p[m % kChains]), so that the dependent chains stay short.
constexpr int kChains = 4;
__device__ __forceinline__ void weighted_relu32(const uint32_t* r, const float* w, uint64_t* p) {
    const float4* wp = reinterpret_cast<const float4*>(w);
#pragma unroll
    for (int i = 0; i < 8; ++i) {          // heads 4i .. 4i+3
        const float4 w4 = wp[i];
        const float x0 = fmaxf(__uint_as_float(r[4 * i + 0]), 0.f), x1 = fmaxf(__uint_as_float(r[4 * i + 1]), 0.f);
        const float x2 = fmaxf(__uint_as_float(r[4 * i + 2]), 0.f), x3 = fmaxf(__uint_as_float(r[4 * i + 3]), 0.f);
        p[(2 * i) % kChains] = ffma2(pack2(x0, x1), pack2(w4.x, w4.y), p[(2 * i) % kChains]);
        p[(2 * i + 1) % kChains] = ffma2(pack2(x2, x3), pack2(w4.z, w4.w), p[(2 * i + 1) % kChains]);
    }
}

// The row's sum of the kChains pair accumulators (a fixed tree).
__device__ __forceinline__ float chains_sum(const uint64_t* p) {
    float s[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) s[c] = sum2(p[c]);
#pragma unroll
    for (int w = kChains / 2; w >= 1; w /= 2)
#pragma unroll
        for (int c = 0; c < w; ++c) s[c] = __fadd_rn(s[c], s[c + w]);
    return s[0];
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_score_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                         const PfArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* keys = smem;
    uint8_t* qbuf = smem + kStages * kKeyBytes;
    PfCtl* ctl = reinterpret_cast<PfCtl*>(qbuf + kQBytes);
    int32_t* tstart = reinterpret_cast<int32_t*>(ctl + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int U = a.units;
    pdl_launch_dependents();

    // ---- first tile of every unit (ceil(keys of its last row / 128) tiles each)
    {
        const int per = (U + kThreads - 1) / kThreads;
        const int u0 = min(U, tid * per), u1 = min(U, u0 + per);
        uint32_t local = 0;
        for (int u = u0; u < u1; ++u) local += static_cast<uint32_t>((unit_keys(a, u) + kTileM - 1) / kTileM);
        uint32_t total;
        uint32_t run = block_exclusive_scan<kThreads>(local, ctl->scan, &total);
        for (int u = u0; u < u1; ++u) {
            tstart[u] = static_cast<int32_t>(run);
            run += static_cast<uint32_t>((unit_keys(a, u) + kTileM - 1) / kTileM);
        }
        if (tid == 0) tstart[U] = static_cast<int32_t>(total);
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1);
            mbar_init(smem_addr(&ctl->empty[s]), 1);
        }
        mbar_init(smem_addr(&ctl->qfull), 1);
        mbar_init(smem_addr(&ctl->qempty), 1);
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(smem_addr(&ctl->accfull[i]), 1);
            mbar_init(smem_addr(&ctl->accempty[i]), kAccWarps);   // the warps that drain it
        }
        mbar_init(smem_addr(&ctl->done), 1);
        ctl->abort = 0;
        fence_barrier_init();
    }
    for (int i = tid; i < kEpiWarps * kRPW * 256; i += kThreads) (&ctl->hist[0][0][0])[i] = 0u;
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&kmap);
        prefetch_tmap(&qmap);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = ctl->tmem_base;
    const uint32_t T = static_cast<uint32_t>(tstart[U]);
    const uint32_t G = gridDim.x, c = blockIdx.x;
    const uint32_t t_begin = static_cast<uint32_t>((static_cast<uint64_t>(T) * c) / G);
    const uint32_t t_end = static_cast<uint32_t>((static_cast<uint64_t>(T) * (c + 1)) / G);
    const uint32_t ntiles = t_end - t_begin;
    volatile int* abort = &ctl->abort;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (ntiles > 0 && lane == 0) {
            const uint32_t prefill = ntiles < static_cast<uint32_t>(kStages) ? ntiles : kStages;
            int ku = find_unit(tstart, U, t_begin);
            uint32_t issued = 0, qn = 0;
            bool ok = true;
            auto issue_keys = [&](uint32_t it) -> bool {
                const uint32_t t = t_begin + it;
                while (t >= static_cast<uint32_t>(tstart[ku + 1])) ++ku;
                const uint32_t s = it % kStages;
                if (!mbar_wait(smem_addr(&ctl->empty[s]), ((it / kStages) & 1) ^ 1, abort)) return false;
                const int32_t tok0 = static_cast<int32_t>(t - tstart[ku]) * kTileM;
                const uint32_t full = smem_addr(&ctl->full[s]);
                mbar_arrive_expect_tx(full, kKeyBytes);
                tma_load_2d(smem_addr(keys + s * kKeyBytes), &kmap, full, 0, tok0);
                return true;
            };
            auto issue_q = [&](int u) -> bool {
                if (qn > 0 && !mbar_wait(smem_addr(&ctl->qempty), (qn - 1) & 1, abort)) return false;
                // a box that starts past the last q8 row is not loaded: the rows it would hold
                // are rows >= R, whose scores the epilogue drops
                const int y0 = u * kRows * ECHO_HEADS;
                const int nbox = min(kQBytes / (kQBox * ECHO_DIM), (a.R * ECHO_HEADS - y0 + kQBox - 1) / kQBox);
                const uint32_t qf = smem_addr(&ctl->qfull);
                mbar_arrive_expect_tx(qf, static_cast<uint32_t>(nbox) * kQBox * ECHO_DIM);
                for (int bx = 0; bx < nbox; ++bx)
                    tma_load_2d(smem_addr(qbuf + bx * kQBox * ECHO_DIM), &qmap, qf, 0, y0 + bx * kQBox);
                ++qn;
                return true;
            };
            // the first key tiles do not depend on the quantiser; q8 does
            for (; issued < prefill; ++issued)
                if (!issue_keys(issued)) {
                    ok = false;
                    break;
                }
            pdl_wait();
            int cur_u = -1, u = find_unit(tstart, U, t_begin);
            for (uint32_t it = 0; it < ntiles && ok; ++it) {
                const uint32_t t = t_begin + it;
                while (t >= static_cast<uint32_t>(tstart[u + 1])) ++u;
                if (it >= issued) {   // this tile's keys first: they do not wait for the MMA to leave the unit
                    if (!issue_keys(it)) {
                        ok = false;
                        break;
                    }
                    ++issued;
                }
                if (u != cur_u) {
                    if (!issue_q(u)) {
                        ok = false;
                        break;
                    }
                    cur_u = u;
                }
            }
            if (!ok) {
                set_status(a.status, ECHO_ST_TIMEOUT);
                *abort = 1;
            }
            // every copy this thread started lands before the CTA exits
            for (uint32_t j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
                mbar_wait(smem_addr(&ctl->full[j % kStages]), (j / kStages) & 1, nullptr);
            if (qn > 0) mbar_wait(smem_addr(&ctl->qfull), (qn - 1) & 1, nullptr);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && ntiles > 0) {
            const uint32_t keys_s = smem_addr(keys), q_s = smem_addr(qbuf);
            int u = find_unit(tstart, U, t_begin), cur_u = -1;
            uint32_t qn = 0;
            bool ok = true;
            for (uint32_t it = 0; it < ntiles && ok; ++it) {
                const uint32_t t = t_begin + it;
                while (t >= static_cast<uint32_t>(tstart[u + 1])) ++u;
                if (u != cur_u) {
                    if (cur_u >= 0) mma_commit(smem_addr(&ctl->qempty));   // the previous unit's MMAs read q
                    if (!mbar_wait(smem_addr(&ctl->qfull), qn & 1, abort)) {
                        ok = false;
                        break;
                    }
                    cur_u = u;
                    ++qn;
                }
                const uint32_t s = it % kStages;
                if (!mbar_wait(smem_addr(&ctl->full[s]), (it / kStages) & 1, abort)) {
                    ok = false;
                    break;
                }
                const uint64_t ad = sw128_kmajor_desc(keys_s + s * kKeyBytes);
#pragma unroll
                for (int acc = 0; acc < kAcc; ++acc) {
                    if (!mbar_wait(smem_addr(&ctl->accempty[acc]), (it & 1) ^ 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = sw128_kmajor_desc(q_s + acc * kN * ECHO_DIM);
                    const uint32_t d = tmem_base + acc * kN;
#pragma unroll
                    for (int kk = 0; kk < ECHO_DIM / 32; ++kk)
                        mma_f8f6f4(d, ad + 2 * kk, bd + 2 * kk, kIdesc, kk > 0 ? 1u : 0u);
                    mma_commit(smem_addr(&ctl->accfull[acc]));
                }
                if (ok) mma_commit(smem_addr(&ctl->empty[s]));
            }
            if (!ok) {
                set_status(a.status, ECHO_ST_TIMEOUT);
                *abort = 1;
            }
            // all MMAs of this thread complete before TMEM is released
            mma_commit(smem_addr(&ctl->done));
            mbar_wait(smem_addr(&ctl->done), 0, nullptr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        pdl_wait();                            // wfold and the cleared histogram come from the quantiser
        const int ew = warp - 2;               // 0 .. kEpiWarps-1
        const int quarter = warp & 3;          // TMEM lanes this warp may access
        const int slot = ew >> 2;              // which of the quarter's warps
        const int ur0 = slot * kRPW;           // the warp's first row of the unit
        const int acc = ur0 / kG;              // the accumulator holding its rows
        const int row = quarter * 32 + lane;   // key within the tile
        const uint32_t base_addr =
            tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kN + (ur0 % kG) * ECHO_HEADS;
        float (*wv)[ECHO_HEADS] = ctl->wv[ew];
        uint32_t (*whist)[256] = ctl->hist[ew];
        float shift = 0.f;
        if (a.theta_hat) {
            const float th = *a.theta_hat;
            shift = isfinite(th) ? th : 0.f;
        }
        auto flush_hist = [&](int uu) {
            __syncwarp();
#pragma unroll
            for (int l = 0; l < kRPW; ++l) {
                const int r = kRows * uu + ur0 + l;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t v = whist[l][lane + 32 * j];
                    if (v) {
                        if (r < a.R) atomicAdd(a.hist + static_cast<size_t>(r) * 256 + lane + 32 * j, v);
                        whist[l][lane + 32 * j] = 0u;
                    }
                }
            }
            __syncwarp();
        };
        int u = (ntiles > 0) ? find_unit(tstart, U, t_begin) : 0;
        int cur_u = -1;
        bool ok = true;
        uint32_t rb[32];
        for (uint32_t it = 0; ok && it < ntiles; ++it) {
            const uint32_t t = t_begin + it;
            while (t >= static_cast<uint32_t>(tstart[u + 1])) ++u;
            if (u != cur_u) {
                if (cur_u >= 0 && a.hist) flush_hist(cur_u);
                cur_u = u;
                __syncwarp();
#pragma unroll
                for (int l = 0; l < kRPW; ++l) {
                    const int r = kRows * u + ur0 + l;
                    const bool in = r < a.R;
                    wv[l][lane] = in ? a.wfold[static_cast<size_t>(r) * ECHO_HEADS + lane] : 0.f;
                    wv[l][lane + 32] = in ? a.wfold[static_cast<size_t>(r) * ECHO_HEADS + lane + 32] : 0.f;
                }
                __syncwarp();
            }
            const int64_t tok = static_cast<int64_t>(t - tstart[u]) * kTileM + row;
            const float ksv = tok < a.n_keys ? __ldg(a.ks + tok) : 0.f;
            if (!mbar_wait(smem_addr(&ctl->accfull[acc]), it & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // pieces of 32 head sums in order (row l = piece / 2, its heads 32 (piece % 2) ..)
            uint64_t p[kChains];
#pragma unroll
            for (int c = 0; c < kChains; ++c) p[c] = 0ull;
#pragma unroll
            for (int pc = 0; pc < kPieces; ++pc) {
                tmem_ld_x32(base_addr + pc * 32, rb);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(rb[i]));
                if (pc + 1 == kPieces) {
                    // every column this warp reads has arrived: hand the accumulator back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&ctl->accempty[acc]));
                }
                const int l = pc >> 1, hh = pc & 1;
                weighted_relu32(rb, &wv[l][hh * 32], p);
                if (hh == 1) {
                    const float sc = __fmul_rn(chains_sum(p), ksv);
#pragma unroll
                    for (int c = 0; c < kChains; ++c) p[c] = 0ull;
                    const int r = kRows * u + ur0 + l;
                    const bool valid = r < a.R && tok <= a.row0 + r;
                    const unsigned vm = __ballot_sync(0xffffffffu, valid);
                    if (valid) {
                        a.scores[static_cast<int64_t>(r) * a.W + tok] = sc;
                        if (a.hist) {
                            const uint32_t bin = shifted_bin(sc, shift);
                            const unsigned grp = __match_any_sync(vm, bin);
                            if (lane == __ffs(grp) - 1) atomicAdd(&whist[l][bin], static_cast<uint32_t>(__popc(grp)));
                        }
                    }
                }
            }
        }
        if (!ok) {
            set_status(a.status, ECHO_ST_TIMEOUT);
            *abort = 1;
        }
        if (cur_u >= 0 && a.hist) flush_hist(cur_u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace
}  // namespace echo

extern "C" int echo_prefill_scores(int R, int64_t row0, int64_t n_keys, const uint8_t* q8, const float* wfold,
                                   const uint8_t* k8, const float* ks, float* scores, int64_t W,
                                   const float* theta_hat, uint32_t* hist, int32_t* status, echo_stream_t stream) {
    using namespace echo;
    if (R <= 0 || row0 < 0 || n_keys <= 0) return ECHO_EINVAL;
    if (R > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!q8 || !wfold || !k8 || !ks || !scores || !status) return ECHO_EINVAL;
    if (row0 + R > n_keys || W < row0 + R) return ECHO_EINVAL;
    if (n_keys >= (1ll << 31) || static_cast<int64_t>(R) * W >= (1ll << 40)) return ECHO_EUNSUPPORTED;
    if (!is_aligned(q8, 16) || !is_aligned(wfold, 16) || !is_aligned(k8, 16) || !is_aligned(ks, 16))
        return ECHO_EINVAL;
    CUtensorMap kmap, qmap;
    int rc = encode_tmap_bytes_2d(&kmap, k8, ECHO_DIM, static_cast<uint64_t>(n_keys), ECHO_DIM, kTileM);
    if (rc) return rc;
    rc = encode_tmap_bytes_2d(&qmap, q8, ECHO_DIM, static_cast<uint64_t>(R) * ECHO_HEADS, ECHO_DIM, kQBox);
    if (rc) return rc;
    const int sms = sm_count();
    if (sms <= 0) return ECHO_ECUDA;
    const int units = (R + kRows - 1) / kRows;
    PfArgs args{R, units, row0, n_keys, W, ks, wfold, scores, theta_hat, hist, status};
    // an upper bound of the tiles: every unit sees at most row0 + R keys
    const int64_t tiles_ub = static_cast<int64_t>(units) * ((row0 + R + kTileM - 1) / kTileM);
    const int grid = static_cast<int>(tiles_ub < sms ? tiles_ub : sms);
    const size_t smem = pf_smem_bytes(units);
    ECHO_CUDA_OK(prefer_max_shared(prefill_score_kernel));
    ECHO_CUDA_OK(cudaFuncSetAttribute(prefill_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
    // Programmatic dependent launch: the prologue and first key loads overlap
    // the quantiser; the kernel waits for it before touching q8, wfold, hist.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ECHO_CUDA_OK(cudaLaunchKernelEx(&cfg, prefill_score_kernel, kmap, qmap, args));
    return ECHO_OK;
}
