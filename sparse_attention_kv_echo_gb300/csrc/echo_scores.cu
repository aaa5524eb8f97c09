// echo_scores.cu -- indexer score of every context token on the tcgen05 tensor cores.
//
// I[t] = ks[t] * sum_h wfold[b,h] * max(0, sum_d q8[b,h,d] * k8[t,d])
// (the DeepSeek-V3.2 lightning-indexer score over E4M3 keys, with the query
// scales folded into the head weights), plus the per-request 256-bin
// histogram of the threshold-shifted scores that top-k selection starts from
// ("ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2,
// panel "Prefill: one-round histogram").
//
// Design (one persistent CTA per SM, 320 threads, warp-specialised):
//   warp 0      TMA producer: 128-token x 128-byte key tiles (16 KB, 128-byte
//               swizzle) into an 8-stage shared-memory ring; the request's
//               q8 [64 x 128] into one of two q buffers when the request changes.
//   warp 1      TMEM owner + single-thread MMA issuer: per tile, four
//               tcgen05.mma kind::f8f6f4 (M=128 tokens, N=64 heads, K=32)
//               into one of four fp32 accumulators of 64 TMEM columns.
//   warps 2-9   two epilogue groups of four warps; group g drains the tiles
//               with local index = g (mod 2).  Each thread owns one token:
//               tcgen05.ld of its 64 head sums, ReLU, weighted sum, times the
//               token scale, store, and a warp-private histogram in shared
//               memory flushed with global atomics when the request changes.
//               With candidate lists, the tokens whose score key reaches the
//               request's cut go to a warp-private buffer in shared memory
//               that is appended to the request's list 32 entries at a time
//               (one atomic per 32 candidates).
// Tiles of all requests form one list; CTA c takes a contiguous share of it.
// The scan of the keys is the HBM-bound part: 132 bytes per token (128 key
// bytes + 4 scale bytes) against 16384 FP8 MAC-flops.
#include "echo_common.cuh"
#include "echo_internal.h"

namespace echo {
namespace {

constexpr int kStages = 8;                             // key ring (released when the MMA is done)
constexpr int kSideStages = 12;                        // side ring (released when the epilogue read it)
constexpr int kTileM = 128;                            // tokens per tile (MMA M)
constexpr int kKeyBytes = kTileM * ECHO_DIM;           // 16 KB per key tile
constexpr int kQBytes = ECHO_HEADS * ECHO_DIM;         // 8 KB q8 per request
constexpr int kAccBufs = 4;                            // TMEM accumulators
constexpr int kTmemCols = kAccBufs * ECHO_HEADS;       // 256 columns
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + kEpiWarps * 32;          // 320
// Per-token side loads (key scale; cache slot for the residency filter) are
// 1-D TMA boxes of 132 elements starting at the tile's first token rounded
// down to a multiple of 4 (16 bytes), so that the box start is aligned; the
// tile's 128 values sit at offset (first token & 3) inside the box.
constexpr int kSideBox = 132;
constexpr int kSidePitch = 160;                        // 640-byte smem rows (128-byte multiple)
constexpr uint32_t kSideBytes = kSideBox * 4;
constexpr uint32_t kIdesc = idesc_e4m3_f32(kTileM, ECHO_HEADS);

// Segments: decode requests (keys and scores at rows [tok_off[b], end) with
// end = tok_end[b] when given, else tok_off[b+1]).
struct ScoreArgs {
    int B;
    const int64_t* tok_off;
    const int64_t* tok_end;    // optional current ends (growing contexts)
    int64_t n_tokens;
    const float* wfold;
    float* scores;
    const float* theta_hat;
    uint32_t* hist;
    uint32_t* above;
    int has_res;               // with above: mark only tokens that are not resident (slots from rmap)
    int32_t* status;
    const uint32_t* freebits;  // copied to free_snap (fb_words words) for the early fetch
    uint32_t* free_snap;
    int64_t fb_words;
    // candidate lists (cand_key null: none): tokens with order key >= cand_cut[b]
    uint32_t* cand_key;
    int32_t* cand_idx;
    int32_t* cand_cnt;
    const uint32_t* cand_cut;
    int cand_cap;
};

constexpr uint32_t kNoCut = 0xFFFFFFFFu;   // a request without a candidate list

// Failure-path test (echo_debug_stall_epilogue): >= 0, the epilogue first waits
// on a barrier that nothing arrives on, giving up after this many ns, which
// takes the kernel down its timeout path; < 0 (the default), no such wait.  The
// other waits, and every wait that drains copies or MMAs before TMEM is freed,
// keep kWaitNs.
__device__ int64_t g_epilogue_stall_ns = -1;
constexpr int kCandBuf = 64;               // per epilogue warp: < 32 waiting + one tile's 32

struct __align__(128) ScoreCtl {
    float ks[kSideStages][kSidePitch];    // per-token key scales of each side stage's tile
    int32_t res[kSideStages][kSidePitch]; // per-token cache slot (>= 0: resident) when above is filtered
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t sfull[kSideStages];
    uint64_t sempty[kSideStages];
    uint64_t qfull[2];
    uint64_t qempty[2];
    uint64_t accfull[kAccBufs];
    uint64_t accempty[kAccBufs];
    uint64_t done;
    uint64_t never;                       // arrived on by nothing (failure-path test)
    uint32_t tmem_base;
    int abort;
    uint32_t scan[16];
    uint32_t hist[kEpiWarps][256];
    uint32_t cbuf_key[kEpiWarps][kCandBuf];   // candidates waiting to be appended
    uint32_t cbuf_idx[kEpiWarps][kCandBuf];
};

// keys | q8 x 2 | ScoreCtl | tstart[B+1] | seg_lo[B] | seg_len[B]  (int32)
__host__ __device__ constexpr size_t smem_bytes(int B) {
    return 1024 + static_cast<size_t>(kStages) * kKeyBytes + 2 * kQBytes + sizeof(ScoreCtl) +
           4 * static_cast<size_t>(3 * B + 1);
}

// Largest request b in [0, B) whose first tile is <= t.
__device__ __forceinline__ int find_request(const int32_t* tstart, int B, uint32_t t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<uint32_t>(tstart[mid]) <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

struct Seg {
    int64_t key_lo;   // first key row
    int64_t len;      // keys (= scores) of the segment
    int64_t out;      // index of its first score
};

// Segment of request b from the arguments; bad segments are empty.
__device__ __forceinline__ Seg segment(const ScoreArgs& a, int b, bool* bad) {
    int64_t lo, hi;
    if (!seg_bounds(a.tok_off, a.tok_end, a.n_tokens, b, &lo, &hi)) {
        *bad = true;
        return Seg{0, 0, 0};
    }
    return Seg{lo, hi - lo, lo};
}

// The same, from the copy the prologue keeps in shared memory.
__device__ __forceinline__ Seg cached_segment(const ScoreArgs& a, const int32_t* seg_lo, const int32_t* seg_len,
                                              int b) {
    const int64_t lo = seg_lo[b], len = seg_len[b];
    return Seg{lo, len, lo};
}

__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                 const __grid_constant__ CUtensorMap smap, const __grid_constant__ CUtensorMap rmap,
                 const ScoreArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* keys = smem;
    uint8_t* qbuf = smem + kStages * kKeyBytes;
    ScoreCtl* ctl = reinterpret_cast<ScoreCtl*>(qbuf + 2 * kQBytes);
    int32_t* tstart = reinterpret_cast<int32_t*>(ctl + 1);
    int32_t* seg_lo = tstart + (a.B + 1);
    int32_t* seg_len = seg_lo + a.B;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B;
    // The next kernel of the stream (the early fetch) may be scheduled as this
    // grid's CTAs retire; it waits for the whole grid before reading anything.
    pdl_launch_dependents();

    // ---- first tile of every request (ceil(N_b / 128) tiles each)
    {
        const int per = (B + kThreads - 1) / kThreads;
        const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
        bool bad = false;
        uint32_t local = 0;
        for (int b = b0; b < b1; ++b) {
            const Seg sg = segment(a, b, &bad);
            seg_lo[b] = static_cast<int32_t>(sg.key_lo);
            seg_len[b] = static_cast<int32_t>(sg.len);
            local += static_cast<uint32_t>((sg.len + kTileM - 1) / kTileM);
        }
        uint32_t total;
        uint32_t run = block_exclusive_scan<kThreads>(local, ctl->scan, &total);
        for (int b = b0; b < b1; ++b) {
            tstart[b] = static_cast<int32_t>(run);
            run += static_cast<uint32_t>((seg_len[b] + kTileM - 1) / kTileM);
        }
        if (tid == 0) tstart[B] = static_cast<int32_t>(total);
        if (bad) set_status(a.status, ECHO_ST_BADDATA);
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1);
            mbar_init(smem_addr(&ctl->empty[s]), 1);      // the MMA is done with the keys
        }
        for (int s = 0; s < kSideStages; ++s) {
            mbar_init(smem_addr(&ctl->sfull[s]), 1);
            mbar_init(smem_addr(&ctl->sempty[s]), 4);     // the tile's 4 epilogue warps read the side boxes
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&ctl->qfull[i]), 1);
            mbar_init(smem_addr(&ctl->qempty[i]), 1);
        }
        for (int i = 0; i < kAccBufs; ++i) {
            mbar_init(smem_addr(&ctl->accfull[i]), 1);
            mbar_init(smem_addr(&ctl->accempty[i]), 4);
        }
        mbar_init(smem_addr(&ctl->done), 1);
        mbar_init(smem_addr(&ctl->never), 1);
        ctl->abort = 0;
        fence_barrier_init();
    }
    for (int i = tid; i < kEpiWarps * 256; i += kThreads) (&ctl->hist[0][0])[i] = 0u;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + tid; i < a.fb_words;
         i += static_cast<int64_t>(gridDim.x) * kThreads)
        a.free_snap[i] = a.freebits[i];
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&kmap);
        prefetch_tmap(&smap);
        if (a.has_res) prefetch_tmap(&rmap);
    }
    if (warp == 1 && lane == 0) prefetch_tmap(&qmap);
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = ctl->tmem_base;
    const uint32_t T = static_cast<uint32_t>(tstart[B]);
    const uint32_t G = gridDim.x, c = blockIdx.x;
    const uint32_t t_begin = static_cast<uint32_t>((static_cast<uint64_t>(T) * c) / G);
    const uint32_t t_end = static_cast<uint32_t>((static_cast<uint64_t>(T) * (c + 1)) / G);
    const uint32_t ntiles = t_end - t_begin;
    volatile int* abort = &ctl->abort;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Lane 0 issues, per tile, the TMA copies of the 128 keys and of the
        // side boxes (scales; slots), all on the stage barrier.  The first
        // stages' loads go out before waiting for the quantiser (their inputs
        // do not depend on it); the q8 of every request after the first (which
        // the MMA warp loads) come after that wait.
        if (ntiles > 0 && lane == 0) {
            // keys and scales stream through L2 once; the slot table stays in L2 for the
            // cache step, which looks up the selected tokens' slots in it (a miss to HBM
            // waits behind the host-link traffic of the early fetch)
            const uint64_t pol = policy_evict_first(), pol_keep = policy_evict_last();
            const uint32_t prefill = ntiles < static_cast<uint32_t>(kStages) ? ntiles : kStages;
            const uint32_t side_tx = kSideBytes * (a.has_res ? 2u : 1u);
            int kb = find_request(tstart, B, t_begin);   // request of the next key load
            int64_t key_lo = 0;
            int kcur = -1;
            uint32_t issued = 0, qn = 0;
            bool ok = true;
            auto issue_keys = [&](uint32_t it) -> bool {
                const uint32_t t = t_begin + it;
                while (t >= static_cast<uint32_t>(tstart[kb + 1])) ++kb;
                if (kb != kcur) {
                    key_lo = seg_lo[kb];
                    kcur = kb;
                }
                const uint32_t s = it % kStages, ss = it % kSideStages;
                if (!mbar_wait(smem_addr(&ctl->empty[s]), ((it / kStages) & 1) ^ 1, abort)) return false;
                if (!mbar_wait(smem_addr(&ctl->sempty[ss]), ((it / kSideStages) & 1) ^ 1, abort)) return false;
                const int64_t tok0 = key_lo + static_cast<int64_t>(t - tstart[kb]) * kTileM;
                const int32_t x0 = static_cast<int32_t>(tok0 & ~int64_t(3));   // 16-byte aligned box start
                const uint32_t full = smem_addr(&ctl->full[s]), sfull = smem_addr(&ctl->sfull[ss]);
                mbar_arrive_expect_tx(full, kKeyBytes);
                tma_load_2d_hint(smem_addr(keys + s * kKeyBytes), &kmap, full, 0, static_cast<int32_t>(tok0), pol);
                mbar_arrive_expect_tx(sfull, side_tx);
                tma_load_1d_hint(smem_addr(&ctl->ks[ss][0]), &smap, sfull, x0, pol);
                if (a.has_res) tma_load_1d_hint(smem_addr(&ctl->res[ss][0]), &rmap, sfull, x0, pol_keep);
                return true;
            };
            for (; issued < prefill; ++issued)
                if (!issue_keys(issued)) {
                    ok = false;
                    break;
                }
            pdl_wait();  // q8 comes from the quantiser
            int cur_b = -1, b = find_request(tstart, B, t_begin);
            for (uint32_t it = 0; it < ntiles && ok; ++it) {
                const uint32_t t = t_begin + it;
                while (t >= static_cast<uint32_t>(tstart[b + 1])) ++b;
                if (b != cur_b) {
                    if (qn > 0) {  // the first request's q8 is loaded by the MMA warp
                        const uint32_t qi = qn & 1;
                        if (!mbar_wait(smem_addr(&ctl->qempty[qi]), ((qn >> 1) & 1) ^ 1, abort)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(smem_addr(&ctl->qfull[qi]), kQBytes);
                        tma_load_2d(smem_addr(qbuf + qi * kQBytes), &qmap, smem_addr(&ctl->qfull[qi]), 0,
                                    b * ECHO_HEADS);
                    }
                    cur_b = b;
                    ++qn;
                }
                if (it >= issued) {
                    if (!issue_keys(it)) {
                        ok = false;
                        break;
                    }
                    ++issued;
                }
            }
            if (!ok) {
                set_status(a.status, ECHO_ST_TIMEOUT);
                *abort = 1;
            }
            // Let every copy this thread started land before the CTA exits.
            for (uint32_t j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
                mbar_wait(smem_addr(&ctl->full[j % kStages]), (j / kStages) & 1, nullptr);
            for (uint32_t j = (issued > kSideStages ? issued - kSideStages : 0); j < issued; ++j)
                mbar_wait(smem_addr(&ctl->sfull[j % kSideStages]), (j / kSideStages) & 1, nullptr);
            for (uint32_t j = (qn > 2 ? qn - 2 : 1); j < qn; ++j)
                mbar_wait(smem_addr(&ctl->qfull[j & 1]), (j >> 1) & 1, nullptr);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && ntiles > 0) {
            const uint32_t keys_s = smem_addr(keys), q_s = smem_addr(qbuf);
            int b = find_request(tstart, B, t_begin), cur_b = -1;
            // q8 of the first request, as soon as the quantiser is done (the
            // producer is busy with the first key loads meanwhile)
            pdl_wait();
            mbar_arrive_expect_tx(smem_addr(&ctl->qfull[0]), kQBytes);
            tma_load_2d(q_s, &qmap, smem_addr(&ctl->qfull[0]), 0, b * ECHO_HEADS);
            bool q0_landed = false;
            uint32_t qn = 0;
            bool ok = true;
            for (uint32_t it = 0; it < ntiles; ++it) {
                const uint32_t t = t_begin + it;
                while (t >= static_cast<uint32_t>(tstart[b + 1])) ++b;
                if (b != cur_b) {
                    if (cur_b >= 0) mma_commit(smem_addr(&ctl->qempty[(qn - 1) & 1]));
                    const uint32_t qi = qn & 1;
                    if (!mbar_wait(smem_addr(&ctl->qfull[qi]), (qn >> 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    if (qn == 0) q0_landed = true;
                    cur_b = b;
                    ++qn;
                }
                const uint32_t acc = it % kAccBufs;
                if (!mbar_wait(smem_addr(&ctl->accempty[acc]), ((it / kAccBufs) & 1) ^ 1, abort)) {
                    ok = false;
                    break;
                }
                const uint32_t s = it % kStages;
                if (!mbar_wait(smem_addr(&ctl->full[s]), (it / kStages) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sw128_kmajor_desc(keys_s + s * kKeyBytes);
                const uint64_t bd = sw128_kmajor_desc(q_s + ((qn - 1) & 1) * kQBytes);
                const uint32_t d = tmem_base + acc * ECHO_HEADS;
#pragma unroll
                for (int kk = 0; kk < ECHO_DIM / 32; ++kk)
                    mma_f8f6f4(d, ad + 2 * kk, bd + 2 * kk, kIdesc, kk > 0 ? 1u : 0u);
                mma_commit(smem_addr(&ctl->empty[s]));
                mma_commit(smem_addr(&ctl->accfull[acc]));
            }
            if (!ok) {
                set_status(a.status, ECHO_ST_TIMEOUT);
                *abort = 1;
            }
            if (!q0_landed) mbar_wait(smem_addr(&ctl->qfull[0]), 0, nullptr);  // its copy lands before exit
            // All MMAs of this thread complete before TMEM is released.
            mma_commit(smem_addr(&ctl->done));
            mbar_wait(smem_addr(&ctl->done), 0, nullptr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        pdl_wait();                            // wfold and the cleared histogram come from the quantiser
        const int64_t stall_ns = g_epilogue_stall_ns;
        const int ew = warp - 2;               // 0..7
        const int group = ew >> 2;             // tiles with local index = group (mod 2)
        const int quarter = warp & 3;          // TMEM lanes this warp may access
        const int row = quarter * 32 + lane;   // token row within the tile
        uint32_t* whist = ctl->hist[ew];
        uint32_t* cbk = ctl->cbuf_key[ew];
        uint32_t* cbi = ctl->cbuf_idx[ew];
        uint32_t nbuf = 0, cut = kNoCut;
        // append the first cnt waiting candidates to request bb's list (one atomic for the
        // warp), keep the rest at the front of the buffer
        auto cand_flush = [&](int bb, uint32_t cnt) {
            __syncwarp();
            uint32_t base = 0;
            if (lane == 0) base = static_cast<uint32_t>(atomicAdd(a.cand_cnt + bb, static_cast<int>(cnt)));
            base = __shfl_sync(0xffffffffu, base, 0);
            const uint32_t cap = static_cast<uint32_t>(a.cand_cap);
            const uint32_t ul = static_cast<uint32_t>(lane);
            if (ul < cnt && base + ul < cap) {
                const int64_t o = static_cast<int64_t>(bb) * cap + base + ul;
                a.cand_key[o] = cbk[ul];
                a.cand_idx[o] = static_cast<int32_t>(cbi[ul]);
            }
            const uint32_t rest = nbuf - cnt;
            uint32_t k2 = 0, i2 = 0;
            if (ul < rest) {
                k2 = cbk[cnt + ul];
                i2 = cbi[cnt + ul];
            }
            __syncwarp();
            if (ul < rest) {
                cbk[ul] = k2;
                cbi[ul] = i2;
            }
            __syncwarp();
            nbuf = rest;
        };
        int b = (ntiles > 0) ? find_request(tstart, B, t_begin) : 0;
        int cur_b = -1;
        float wv[ECHO_HEADS];
        float shift = 0.f, theta = 0.f;
        bool theta_ok = false;
        int64_t nb = 0, obase = 0, abase = 0;
        int side = 0;   // offset of the tile's first token in its side boxes
        // (failure-path test) a wait that can only run out
        bool ok = stall_ns < 0 || mbar_wait_limit(smem_addr(&ctl->never), 0, abort, static_cast<uint64_t>(stall_ns));
        for (uint32_t it = group; ok && it < ntiles; it += 2) {
            const uint32_t t = t_begin + it;
            while (t >= static_cast<uint32_t>(tstart[b + 1])) ++b;
            if (b != cur_b) {
                if (cur_b >= 0 && a.hist) {
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t v = whist[lane + 32 * j];
                        if (v) {
                            atomicAdd(a.hist + static_cast<size_t>(cur_b) * 256 + lane + 32 * j, v);
                            whist[lane + 32 * j] = 0u;
                        }
                    }
                    __syncwarp();
                }
                if (cur_b >= 0 && nbuf) cand_flush(cur_b, nbuf);
                cur_b = b;
                cut = a.cand_key ? a.cand_cut[b] : kNoCut;
                const float4* wp = reinterpret_cast<const float4*>(a.wfold + static_cast<size_t>(b) * ECHO_HEADS);
#pragma unroll
                for (int i = 0; i < ECHO_HEADS / 4; ++i) {
                    const float4 x = wp[i];
                    wv[4 * i + 0] = x.x;
                    wv[4 * i + 1] = x.y;
                    wv[4 * i + 2] = x.z;
                    wv[4 * i + 3] = x.w;
                }
                const float th =
                    a.theta_hat ? a.theta_hat[b] : __int_as_float(0x7f800000);

                theta_ok = isfinite(th);
                theta = th;
                shift = theta_ok ? th : 0.f;
                const Seg sg = cached_segment(a, seg_lo, seg_len, b);
                side = static_cast<int>(sg.key_lo & 3);
                nb = sg.len;
                obase = sg.out;
                // the request's above-threshold words start at 4 * (floor(first row / 128) + b)
                abase = 4 * (sg.key_lo / kTileM + b - static_cast<int64_t>(tstart[b]));
            }
            const int64_t tok = static_cast<int64_t>(t - tstart[b]) * kTileM + row;
            const bool valid = tok < nb;
            const uint32_t acc = it % kAccBufs;
            if (!mbar_wait(smem_addr(&ctl->accfull[acc]), (it / kAccBufs) & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // the tile's side boxes: read the scales (and slots), then release them
            const uint32_t ss = it % kSideStages;
            if (!mbar_wait(smem_addr(&ctl->sfull[ss]), (it / kSideStages) & 1, abort)) {
                ok = false;
                break;
            }
            const float ksv = ctl->ks[ss][row + side];
            const bool resident = a.has_res && ctl->res[ss][row + side] >= 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&ctl->sempty[ss]));
            uint32_t r0[16], r1[16], r2[16], r3[16];
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * ECHO_HEADS;
            tmem_ld_x16(taddr + 0, r0);
            tmem_ld_x16(taddr + 16, r1);
            tmem_ld_x16(taddr + 32, r2);
            tmem_ld_x16(taddr + 48, r3);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r0[i]), "+r"(r1[i]), "+r"(r2[i]), "+r"(r3[i]));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&ctl->accempty[acc]));
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                s0 = fmaf(wv[i], fmaxf(__uint_as_float(r0[i]), 0.f), s0);
                s1 = fmaf(wv[16 + i], fmaxf(__uint_as_float(r1[i]), 0.f), s1);
                s2 = fmaf(wv[32 + i], fmaxf(__uint_as_float(r2[i]), 0.f), s2);
                s3 = fmaf(wv[48 + i], fmaxf(__uint_as_float(r3[i]), 0.f), s3);
            }
            const float score = __fmul_rn(__fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3)), ksv);
            const unsigned vm = __ballot_sync(0xffffffffu, valid);
            if (cut != kNoCut) {
                // candidates of the request's top-k: score key at or above the cut
                const uint32_t key = order_key(score);
                const bool cnd = valid && key >= cut;
                const unsigned cm = __ballot_sync(0xffffffffu, cnd);
                if (cm) {
                    if (cnd) {
                        const uint32_t p = nbuf + __popc(cm & ((1u << lane) - 1u));
                        cbk[p] = key;
                        cbi[p] = static_cast<uint32_t>(tok);
                    }
                    nbuf += __popc(cm);
                    if (nbuf >= 32) cand_flush(b, 32);
                }
            }
            if (a.cand_key && __any_sync(0xffffffffu, valid && isnan(score)) && lane == 0)
                set_status(a.status, ECHO_ST_NAN);
            if (a.above) {
                // tokens above the predicted threshold: one word per 32 rows of the tile
                const unsigned am = __ballot_sync(0xffffffffu, valid && theta_ok && score > theta && !resident);
                if (lane == 0) a.above[abase + 4 * static_cast<int64_t>(t) + quarter] = am;
            }
            if (valid) {
                a.scores[obase + tok] = score;
                if (a.hist) {
                    const uint32_t bin = shifted_bin(score, shift);
                    const unsigned grp = __match_any_sync(vm, bin);
                    if (lane == __ffs(grp) - 1) whist[bin] += __popc(grp);
                }
            }
        }
        if (!ok) {
            set_status(a.status, ECHO_ST_TIMEOUT);
            *abort = 1;
        }
        if (cur_b >= 0 && nbuf) cand_flush(cur_b, nbuf);
        if (cur_b >= 0 && a.hist) {
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t v = whist[lane + 32 * j];
                if (v) atomicAdd(a.hist + static_cast<size_t>(cur_b) * 256 + lane + 32 * j, v);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

static int launch_scores(const ScoreArgs& args, const uint8_t* q8, const uint8_t* k8, const float* ks,
                  const int32_t* tok2slot, int64_t key_rows, int64_t tiles_ub, int ctas, cudaStream_t stream) {
    CUtensorMap kmap, qmap, smap, rmap;
    int rc = encode_tmap_bytes_2d(&kmap, k8, ECHO_DIM, static_cast<uint64_t>(key_rows), ECHO_DIM, kTileM);
    if (rc) return rc;
    rc = encode_tmap_bytes_2d(&qmap, q8, ECHO_DIM, static_cast<uint64_t>(args.B) * ECHO_HEADS, ECHO_DIM,
                              ECHO_HEADS);
    if (rc) return rc;
    rc = encode_tmap_1d(&smap, ks, true, static_cast<uint64_t>(key_rows), kSideBox);
    if (rc) return rc;
    rc = encode_tmap_1d(&rmap, tok2slot ? static_cast<const void*>(tok2slot) : static_cast<const void*>(ks),
                        tok2slot == nullptr, static_cast<uint64_t>(key_rows), kSideBox);
    if (rc) return rc;
    const int sms = sm_count();
    if (sms <= 0) return ECHO_ECUDA;
    const int most = (ctas > 0 && ctas < sms) ? ctas : sms;
    const int grid = static_cast<int>(tiles_ub < most ? tiles_ub : most);
    const size_t smem = smem_bytes(args.B);
    ECHO_CUDA_OK(prefer_max_shared(score_kernel));
    ECHO_CUDA_OK(cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    ECHO_CUDA_OK(cudaLaunchKernelEx(&cfg, score_kernel, kmap, qmap, smap, rmap, args));
    return ECHO_OK;
}

}  // namespace echo

namespace echo {

static int index_scores(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens, const uint8_t* q8,
                        const float* wfold, const uint8_t* k8, const float* ks, float* scores,
                        const float* theta_hat, uint32_t* hist, uint32_t* above, const echo_cache* cache,
                        const echo_cands* cands, int ctas, int32_t* status, cudaStream_t stream) {
    if (B <= 0 || n_tokens < 0) return ECHO_EINVAL;
    if (B > ECHO_MAX_REQUESTS) return ECHO_EUNSUPPORTED;
    if (!tok_off || !q8 || !wfold || !status) return ECHO_EINVAL;
    if (n_tokens > 0 && (!k8 || !ks || !scores)) return ECHO_EINVAL;
    if (n_tokens >= (1ll << 31)) return ECHO_EUNSUPPORTED;
    if (!is_aligned(q8, 16) || !is_aligned(wfold, 16) || !is_aligned(k8, 16) || !is_aligned(ks, 16))
        return ECHO_EINVAL;
    if (cache) {
        if (!above) return ECHO_EINVAL;
        const int rc = check_cache(cache, B, 0);
        if (rc) return rc;
        if (!cache->free_snap || !is_aligned(cache->tok2slot, 16)) return ECHO_EINVAL;
    }
    if (cands && (!cands->key || !cands->idx || !cands->cnt || !cands->cut || cands->cap <= 0 ||
                  !is_aligned(cands->key, 4) || !is_aligned(cands->idx, 4) || !is_aligned(cands->cnt, 4) ||
                  !is_aligned(cands->cut, 4)))
        return ECHO_EINVAL;
    if (n_tokens == 0) return ECHO_OK;
    ScoreArgs args{B, tok_off, tok_end, n_tokens, wfold, scores, theta_hat, hist, above,
                   cache ? 1 : 0, status, cache ? cache->freebits : nullptr,
                   cache ? cache->free_snap : nullptr,
                   cache ? static_cast<int64_t>(B) * (cache->C / 32) : 0,
                   cands ? cands->key : nullptr, cands ? cands->idx : nullptr, cands ? cands->cnt : nullptr,
                   cands ? cands->cut : nullptr, cands ? cands->cap : 0};
    return launch_scores(args, q8, k8, ks, cache ? cache->tok2slot : nullptr, n_tokens, n_tokens / kTileM + B, ctas,
                         stream);
}

}  // namespace echo

extern "C" int echo_index_scores(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                                 const uint8_t* q8,
                                 const float* wfold, const uint8_t* k8, const float* ks, float* scores,
                                 const float* theta_hat, uint32_t* hist, uint32_t* above, const echo_cache* cache,
                                 int ctas, int32_t* status, echo_stream_t stream) {
    return echo::index_scores(B, tok_off, tok_end, n_tokens, q8, wfold, k8, ks, scores, theta_hat, hist, above, cache,
                              nullptr, ctas, status, stream);
}

extern "C" int echo_index_scores_cands(int B, const int64_t* tok_off, const int64_t* tok_end, int64_t n_tokens,
                                       const uint8_t* q8, const float* wfold, const uint8_t* k8, const float* ks,
                                       float* scores, const float* theta_hat, uint32_t* hist, uint32_t* above,
                                       const echo_cache* cache, const echo_cands* cands, int ctas, int32_t* status,
                                       echo_stream_t stream) {
    if (!cands) return ECHO_EINVAL;
    return echo::index_scores(B, tok_off, tok_end, n_tokens, q8, wfold, k8, ks, scores, theta_hat, hist, above, cache,
                              cands, ctas, status, stream);
}

extern "C" size_t echo_above_words(int B, int64_t n_tokens) {
    if (B <= 0 || n_tokens < 0) return 0;
    return 4 * static_cast<size_t>(n_tokens / 128 + B);
}

extern "C" int echo_debug_stall_epilogue(int64_t limit_ns) {
    const int64_t v = limit_ns < 0 ? -1 : limit_ns;
    if (cudaMemcpyToSymbol(echo::g_epilogue_stall_ns, &v, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return ECHO_ECUDA;
    }
    return ECHO_OK;
}
