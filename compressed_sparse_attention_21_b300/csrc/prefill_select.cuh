// Selection pieces shared by the prefill-sized indexers (index_block.cu,
// index_tc.cu): the per-query record of a query block, a warp-level radix
// select, the top-k of one query by one warp from its candidates, and the
// block-wide exact selection used when a warp cannot finish a query.
#pragma once

#include "common.cuh"

namespace csa {
namespace {

constexpr int kBT = 512;             // threads of a prefill indexer CTA (16 warps)
constexpr int kBRows = 256;          // entries per chunk
constexpr int kBSample = 256;        // sampled entries for the threshold
constexpr int kBCap = 4096;          // candidates kept per query
constexpr int kBMaxN = 32768;        // longest row: bitmaps of 1024 words
constexpr int kBMaxK = 1024;
constexpr int kBWords = kBMaxN / 32;
constexpr int kBFallKeys = kBMaxN / kBT;   // keys per thread of the exact fallback


struct BlockQ {           // per-query record of the current block
    int b;                // sequence
    int n;                // visible entries
    int64_t e0;           // first entry row of the sequence
    int ok;               // layout consistent
};

// The k-th largest of a warp's keys (k >= 1; at least k keys exist): 8-bit
// radix levels over the keys that `get(i, key)` hands out for i < count
// (lane-strided, U loads in flight per lane), with a warp-private 256-bin
// histogram `hist` and two words `dig` of shared memory.  Every key lies in
// [lo, hi], so the bits above the highest bit where lo and hi differ are
// common to all of them and the levels start at the byte holding that bit.
// Stops at the first level whose bin is taken whole.  Returns the prefix
// found (its lower bits zero when it stopped early) in *kstar and the number
// of keys equal to it still to take in *need_eq (0xffffffff when every key at
// or above *kstar is taken).  Every lane of the warp calls it.
template <int U = 8, typename Get>
__device__ __forceinline__ void warp_radix_select(Get get, int count, uint32_t k, uint32_t *hist, uint32_t *dig,
                                                  uint32_t *kstar, uint32_t *need_eq, uint32_t lo = 0u,
                                                  uint32_t hi = 0xffffffffu)
{
    const int lane = threadIdx.x & 31;
    const uint32_t diff = lo ^ hi;
    const int top = diff ? 31 - __clz(diff) : 0;          // highest bit that can differ
    const int sh0 = 8 * (top / 8);
    const uint32_t low = sh0 >= 24 ? 0xffffffffu : (1u << (sh0 + 8)) - 1u;   // the bits the levels resolve
    uint32_t prefix = lo & ~low, pmask = ~low, remaining = k;
    bool whole = false;
#pragma unroll 1
    for (int sh = sh0; sh >= 0 && !whole; sh -= 8) {
#pragma unroll
        for (int i = 0; i < 8; i++) hist[lane * 8 + i] = 0;
        __syncwarp();
#pragma unroll 1
        for (int base = 0; base < count; base += 32 * U) {
            uint32_t kk[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int i = base + 32 * u + lane;
                kk[u] = 0;
                if (i < count) get(i, kk[u]);
            }
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int i = base + 32 * u + lane;
                hist_add(hist, (kk[u] >> sh) & 255u, i < count && (kk[u] & pmask) == prefix);
            }
        }
        __syncwarp();
        find_digit_256(hist, remaining, &dig[0], &dig[1]);
        __syncwarp();
        const uint32_t d = dig[0];
        remaining -= dig[1];
        prefix |= d << sh;
        pmask |= 255u << sh;
        whole = hist[d] == remaining;
        __syncwarp();   // hist and dig are rewritten by the next level
    }
    *kstar = prefix;
    *need_eq = whole ? 0xffffffffu : remaining;
}

// One query's top-k by one warp, from its `cnt` candidates (key << 32 | entry,
// every key in [lo, hi]; `cand(i)` loads candidate i from global memory): the exact k-th key, then a bitmap
// of the taken entries, and the selection written in index order.  Without
// scores the entries are emitted from the bitmap itself; with scores a second
// pass over the candidates places each (entry, score) by the bitmap's word
// prefixes.  Returns false, writing nothing, when keys equal to the k-th key
// would have to be split (the block-wide selection resolves that case).
// U candidates are in flight per lane.
template <int U = 16, typename Cand>
__device__ __forceinline__ bool warp_select_write(Cand cand, int cnt, int n, int top_k,
                                                  uint8_t *scratch, uint32_t *dig, int32_t *idx_row, float *sc_row,
                                                  uint32_t lo = 0u, uint32_t hi = 0xffffffffu)
{
    const int lane = threadIdx.x & 31;
    uint32_t *hist = reinterpret_cast<uint32_t *>(scratch);
    uint32_t *taken = hist + 256;
    uint16_t *pre = reinterpret_cast<uint16_t *>(taken + kBWords);
    const uint32_t k_eff = (uint32_t)(n < top_k ? n : top_k);
    uint32_t kstar, need_eq;
    warp_radix_select<U>([&](int i, uint32_t &key) { key = (uint32_t)(cand(i) >> 32); }, cnt, k_eff, hist,
                         dig, &kstar, &need_eq, lo, hi);
    if (need_eq != 0xffffffffu) return false;   // ties at the k-th key: the block-wide path
    const int words = (n + 31) >> 5;
    for (int w = lane; w < words; w += 32) taken[w] = 0;
    __syncwarp();
#pragma unroll 1
    for (int base = 0; base < cnt; base += 32 * U) {
        uint64_t v[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int i = base + 32 * u + lane;
            v[u] = i < cnt ? cand(i) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int i = base + 32 * u + lane;
            const uint32_t e = (uint32_t)v[u];
            if (i < cnt && (uint32_t)(v[u] >> 32) >= kstar) atomicOr(&taken[e >> 5], 1u << (e & 31));
        }
    }
    __syncwarp();
    if (!sc_row) {
        // 32 words at a time: a scan of their counts gives each lane the place
        // of its word's first entry, and the lane writes the word's entries
        uint32_t at = 0;
        for (int w0 = 0; w0 < words; w0 += 32) {
            const int w = w0 + lane;
            uint32_t bits = w < words ? taken[w] : 0u;
            const uint32_t c = (uint32_t)__popc(bits);
            uint32_t incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            uint32_t pos = at + incl - c;
            while (bits) {
                const int j = __ffs(bits) - 1;
                bits &= bits - 1u;
                if (pos < (uint32_t)top_k) idx_row[pos] = (int32_t)((w << 5) + j);
                pos++;
            }
            at += __shfl_sync(0xffffffffu, incl, 31);
        }
    } else {
        // word prefixes: lane takes a contiguous run of words
        const int wpl = (words + 31) / 32;
        const int w0 = lane * wpl, w1 = w0 + wpl < words ? w0 + wpl : words;
        uint32_t mine = 0;
        for (int w = w0; w < w1; w++) mine += (uint32_t)__popc(taken[w]);
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        uint32_t run = incl - mine;
        for (int w = w0; w < w1; w++) {
            pre[w] = (uint16_t)run;
            run += (uint32_t)__popc(taken[w]);
        }
        __syncwarp();
#pragma unroll 1
        for (int base = 0; base < cnt; base += 32 * U) {
            uint64_t v[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int i = base + 32 * u + lane;
                v[u] = i < cnt ? cand(i) : 0ull;
            }
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int i = base + 32 * u + lane;
                const uint32_t key = (uint32_t)(v[u] >> 32), e = (uint32_t)v[u];
                if (i < cnt && key >= kstar) {
                    const uint32_t pos = pre[e >> 5] + (uint32_t)__popc(taken[e >> 5] & ((1u << (e & 31)) - 1u));
                    if (pos < (uint32_t)top_k) {
                        idx_row[pos] = (int32_t)e;
                        sc_row[pos] = key_score(key);
                    }
                }
            }
        }
    }
    for (int i = (int)k_eff + lane; i < top_k; i += 32) {
        idx_row[i] = -1;
        if (sc_row) sc_row[i] = -INFINITY;
    }
    return true;
}

// Exact selection of one query's top-k among the (key, entry) pairs that
// `src` hands out: src(i, key, ent) for i < NPT gives this thread's i-th pair
// (false when there is none).  Writes the row of idx/score in index order.
template <int NPT, typename Src>
__device__ void select_write(Src src, int n, int top_k, uint8_t *sm_gt, uint8_t *sm_eq, uint8_t *sm_pre,
                             uint32_t *s_hist, uint32_t *s_w, uint32_t *s_dig, int32_t *idx_row, float *sc_row)
{
    const int tid = threadIdx.x;
    uint32_t *gt = reinterpret_cast<uint32_t *>(sm_gt);
    uint32_t *eq = reinterpret_cast<uint32_t *>(sm_eq);
    uint32_t *pre = reinterpret_cast<uint32_t *>(sm_pre);
    const uint32_t k_eff = (uint32_t)(n < top_k ? n : top_k);
    // k-th largest key: four 8-bit radix levels
    uint32_t prefix = 0, pmask = 0, remaining = k_eff;
    for (int sh = 24; sh >= 0 && k_eff > 0; sh -= 8) {
        for (int i = tid; i < 256; i += kBT) s_hist[i] = 0;
        __syncthreads();
#pragma unroll 1
        for (int i = 0; i < NPT; i++) {
            uint32_t key;
            int32_t ent;
            if (src(i, key, ent) && (key & pmask) == prefix) atomicAdd(&s_hist[(key >> sh) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) find_digit_256(s_hist, remaining, &s_dig[0], &s_dig[1]);
        __syncthreads();
        remaining -= s_dig[1];
        prefix |= s_dig[0] << sh;
        pmask |= 255u << sh;
        __syncthreads();
    }
    const uint32_t kstar = prefix, need_eq = remaining;
    // bitmaps of the entries above and equal to the k-th key
    const int words = (n + 31) >> 5;
    for (int i = tid; i < words; i += kBT) {
        gt[i] = 0;
        eq[i] = 0;
    }
    __syncthreads();
    if (k_eff > 0) {
#pragma unroll 1
        for (int i = 0; i < NPT; i++) {
            uint32_t key;
            int32_t ent;
            if (!src(i, key, ent)) continue;
            if (key > kstar) atomicOr(&gt[ent >> 5], 1u << (ent & 31));
            else if (key == kstar) atomicOr(&eq[ent >> 5], 1u << (ent & 31));
        }
    }
    __syncthreads();
    // exclusive prefix of (popc gt << 16 | popc eq) over the words, two words per thread
    {
        const int w0 = 2 * tid, w1 = 2 * tid + 1;
        const uint32_t v0 = w0 < words ? ((uint32_t)__popc(gt[w0]) << 16) | (uint32_t)__popc(eq[w0]) : 0u;
        const uint32_t v1 = w1 < words ? ((uint32_t)__popc(gt[w1]) << 16) | (uint32_t)__popc(eq[w1]) : 0u;
        uint32_t tot;
        const uint32_t ex = block_scan<kBT>(v0 + v1, s_w, tot);
        if (w0 < words) pre[w0] = ex;
        if (w1 < words) pre[w1] = ex + v0;
    }
    __syncthreads();
    if (k_eff > 0) {
#pragma unroll 1
        for (int i = 0; i < NPT; i++) {
            uint32_t key;
            int32_t e;
            if (!src(i, key, e)) continue;
            const int w = e >> 5;
            const uint32_t below = (1u << (e & 31)) - 1u;
            const uint32_t gt_before = (pre[w] >> 16) + (uint32_t)__popc(gt[w] & below);
            const uint32_t eq_before = (pre[w] & 0xffffu) + (uint32_t)__popc(eq[w] & below);
            bool take = false;
            uint32_t pos = 0;
            if (key > kstar) {
                take = true;
                pos = gt_before + (eq_before < need_eq ? eq_before : need_eq);
            } else if (key == kstar && eq_before < need_eq) {
                take = true;
                pos = gt_before + eq_before;
            }
            if (take && pos < (uint32_t)top_k) {
                idx_row[pos] = e;
                if (sc_row) sc_row[pos] = key_score(key);
            }
        }
    }
    for (int i = (int)k_eff + tid; i < top_k; i += kBT) {
        idx_row[i] = -1;
        if (sc_row) sc_row[i] = -INFINITY;
    }
    __syncthreads();
}

}  // namespace
}  // namespace csa
