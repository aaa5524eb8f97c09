// echo_slots.cuh -- block-wide free-slot bookkeeping shared by the cache-step
// and early-fetch kernels.
//
// "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", section 2:
// panel "One layer, one step: free -> allocate -> recall" (misses take free
// slots) and panel "Decode: fetch above a predicted threshold" (tokens above
// the predicted threshold are fetched before top-k completes, up to a cap).
// The early set is computed twice from the same inputs, by the early-fetch
// kernel (to copy its rows) and by the cache-step kernel (to enter it in the
// tables); early_assign is the one definition both use.
#pragma once

#include "echo_common.cuh"

namespace echo {

// The GPU-cache tables of one layer, as the kernels see them.
struct CacheArgs {
    int32_t* tok2slot;
    int32_t* slot2tok;
    uint32_t* freebits;
    int32_t* miss_tok;
    int32_t* miss_slot;
    int32_t* miss_cnt;
    int32_t* early_tok;
    int32_t* early_slot;
    int32_t* early_cnt;
    int32_t C;
};

inline CacheArgs cache_args(const echo_cache& c) {
    return CacheArgs{c.tok2slot, c.slot2tok, c.freebits, c.miss_tok, c.miss_slot, c.miss_cnt,
                     c.early_tok, c.early_slot, c.early_cnt, c.C};
}

// Free-slot prefix of one request: fbs[w] = its free-bit word w, wpre[w] =
// free slots in the words before w, wpre[words] = all free slots (returned).
// Block-wide (NT threads); wpre: words + 1, fbs: words entries of shared memory.
template <int NT>
__device__ uint32_t free_prefix(const uint32_t* fb, int words, uint32_t* scan, uint32_t* wpre, uint32_t* fbs) {
    uint32_t run = 0;
    for (int w0 = 0; w0 < words; w0 += NT) {
        const int w = w0 + threadIdx.x;
        const uint32_t f = (w < words) ? fb[w] : 0u;
        if (w < words) fbs[w] = f;
        uint32_t tot;
        const uint32_t ex = block_exclusive_scan<NT>(__popc(f), scan, &tot);
        if (w < words) wpre[w] = run + ex;
        run += tot;
    }
    if (threadIdx.x == 0) wpre[words] = run;
    __syncthreads();
    return run;
}

// Walks the free slots of a request in ascending order from free rank r
// (r < wpre[words]): next() returns the slot of rank r, r + 1, ...
// Position of the k-th (0-based) set bit of f; k < popc(f).  Five halving
// steps on popcounts instead of clearing k bits one by one.
__device__ __forceinline__ int nth_set_bit(uint32_t f, uint32_t k) {
    int base = 0;
#pragma unroll
    for (int width = 16; width > 0; width >>= 1) {
        const uint32_t low = f & ((1u << width) - 1u);
        const uint32_t c = static_cast<uint32_t>(__popc(low));
        if (k >= c) {
            k -= c;
            f >>= width;
            base += width;
        } else {
            f = low;
        }
    }
    return base;
}

struct FreeWalk {
    const uint32_t* fbs;
    int words, w;
    uint32_t f;
    __device__ FreeWalk() {}
    __device__ FreeWalk(const uint32_t* wpre, const uint32_t* fbs_, int words_, uint32_t r) {
        init(wpre, fbs_, words_, r);
    }
    __device__ void init(const uint32_t* wpre, const uint32_t* fbs_, int words_, uint32_t r) {
        fbs = fbs_;
        words = words_;
        int lo = 0, hi = words - 1;  // largest w with wpre[w] <= r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (wpre[mid] <= r)
                lo = mid;
            else
                hi = mid - 1;
        }
        w = lo;
        f = fbs[lo];
        const uint32_t k = r - wpre[lo];
        if (k < static_cast<uint32_t>(__popc(f))) {
            const int bit = nth_set_bit(f, k);  // the walk starts at the k-th free slot of the word
            f &= ~((1u << bit) - 1u);
        } else {
            f = 0u;
        }
    }
    // -1 once the free slots run out (a caller that keeps r < wpre[words] never sees it)
    __device__ int next() {
        while (f == 0) {
            if (++w >= words) return -1;
            f = fbs[w];
        }
        const int slot = w * 32 + (__ffs(f) - 1);
        f &= f - 1;
        return slot;
    }
};

// The lowest `take` free slots are now used: clear them in the free-bit words
// fbs (shared memory, in place; wpre: their prefix before the update).  No
// thread may still be walking fbs: the caller synchronises first.
template <int NT>
__device__ void take_lowest_free(uint32_t* fbs, int words, uint32_t take, const uint32_t* wpre) {
    for (int w = threadIdx.x; w < words; w += NT) {
        if (wpre[w] >= take) continue;
        if (wpre[w + 1] <= take) {  // every free slot of the word is taken
            fbs[w] = 0u;
            continue;
        }
        // the boundary word: its lowest take - wpre[w] free slots are taken, the
        // rest (from its (take - wpre[w])-th free bit on) stay free
        const uint32_t f = fbs[w];
        const int bit = nth_set_bit(f, take - wpre[w]);
        fbs[w] = f & ~((1u << bit) - 1u);
    }
}

// Above-threshold words of one request: v = words w0 .. w0+P-1 of ab[0, nw),
// zero past nw, the last word masked at the request end.
template <int P>
__device__ __forceinline__ void early_words(const uint32_t* ab, int nw, uint32_t tail_mask, int w0, uint32_t (&v)[P]) {
#pragma unroll
    for (int j = 0; j < P; ++j) {
        const int w = w0 + j;
        v[j] = (w < nw) ? __ldcg(ab + w) : 0u;
        if (w == nw - 1) v[j] &= tail_mask;
    }
}

// The early set of one request (block-wide, NT threads, P words per thread):
// the tokens marked in ab[0, nw) (bit j of word w = token 32*w + j), in
// ascending order, those of rank < limit, take the free slots of ranks 0, 1,
// ... in ascending order (wpre/fbs: the request's free-slot prefix).  Calls
// emit(rank, token, slot) for the ranks in [r_lo, r_hi), each from the thread
// that owns the token; a thread owns P consecutive words, so its tokens have
// consecutive ranks and take consecutive free slots: one binary search, then
// a walk over the free bits.  v holds this thread's words w = P*threadIdx.x
// .. (early_words) on entry.  Returns the number of marked tokens counted,
// which is >= r_hi when more than r_hi tokens are marked, else all of them.
template <int NT, int P, class Emit>
__device__ uint32_t early_assign(const uint32_t* ab, int nw, uint32_t tail_mask, uint32_t limit, uint32_t r_lo,
                                 uint32_t r_hi, const uint32_t* wpre, const uint32_t* fbs, int words, uint32_t* scan,
                                 uint32_t (&v)[P], Emit emit) {
    uint32_t found = 0;
    for (int c0 = 0; c0 < nw && found < r_hi; c0 += NT * P) {
        const int w0 = c0 + static_cast<int>(threadIdx.x) * P;
        if (c0 > 0) early_words<P>(ab, nw, tail_mask, w0, v);
        uint32_t cnt = 0;
#pragma unroll
        for (int j = 0; j < P; ++j) cnt += __popc(v[j]);
        uint32_t tot;
        const uint32_t rank0 = found + block_exclusive_scan<NT>(cnt, scan, &tot);
        const uint32_t hi = min(min(limit, r_hi), rank0 + cnt);
        if (rank0 < hi && rank0 + cnt > r_lo) {
            FreeWalk walk(wpre, fbs, words, rank0);
            uint32_t rank = rank0;
#pragma unroll
            for (int j = 0; j < P; ++j) {
                uint32_t m = v[j];
                while (m && rank < hi) {
                    const int tok = 32 * (w0 + j) + (__ffs(m) - 1);
                    m &= m - 1;
                    const int slot = walk.next();
                    if (rank >= r_lo) emit(rank, tok, slot);
                    ++rank;
                }
            }
        }
        found += tot;
    }
    return found;
}

}  // namespace echo
