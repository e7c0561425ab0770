// Lightning indexer + top-k ("DeepSeek-V4 core architecture", §2.2 CSA step 2:
// a light scorer rates each query against every compressed entry and only the
// top-k entries take part in attention).
//
// Score of visible entry j (j < n(t) = floor((t+1)/m)) for the query at t:
//     s = fp32 sum over indexer heads h of q_{t,h} . k_j
// computed as (sum_h q_{t,h}) . k_j: the head sum is formed once per query in
// fp32 and the dot product runs in fp32 FMAs.  Ties go to the lower index and
// the kept indices are written in ascending order, padded with -1.
//
// Scores are mapped onto order-preserving 32-bit keys.  Two paths:
//  * per-query CTA (prefill-sized batches, n(t) <= kCtaMaxN): the query's
//    whole key row lives in shared memory; an 8-bit radix select finds the
//    k-th key exactly and one ordered pass emits the selection in index
//    order (ties resolved by rank among equal keys);
//  * multi-CTA (decode-sized batches or long rows): many CTAs per query scan
//    the indexer keys (the HBM-bound part), write the key row to the
//    workspace and build a 4096-bin histogram of the keys' top 12 bits.
//    For rows of up to kSelMaxN entries a cluster of CTAs per query then
//    selects from the key row (path 3 below).  Longer rows: the last scan
//    CTA of a query (atomic ticket, no waiting) locates the bin that holds
//    the k-th key; a second kernel keeps everything above that bin,
//    collects the bin's members as candidates, and its last CTA per query
//    resolves them with a radix select on (key, index), then sorts the k
//    winners by index.
// The full score matrix is never stored; only one key row per query in the
// multi-CTA path.
#include <cuda_fp8.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace csa {

namespace {

constexpr int kCtaThreads = 512;
constexpr int kCtaMaxN = 40960;       // key row in shared memory: 160 KiB
constexpr int kMaxTopK = 2048;
constexpr int kScanThreads = 256;
constexpr int kScanChunk = 1024;      // entries per scan/filter CTA
constexpr int kHistBits = 12;
constexpr int kHistBins = 1 << kHistBits;
constexpr int kFilterSmemCand = 3072;  // boundary candidates resolved in shared memory
constexpr int kSelCluster = 8;        // CTAs per query in the select cluster (rows up to 131072 entries)
constexpr int kSelClusterMax = 16;    // ... and for longer rows (a non-portable cluster size)
constexpr int kSelCandCta = 512;      // boundary-bin members one select CTA ranks directly
constexpr int kSelCandTotal = 2048;   // ... and the whole cluster
constexpr int kMetaWords = 8;         // per-query: ticket1, ticket2, n_sel, n_cand, bin, above
constexpr int64_t kGroupBudget = int64_t(1) << 30;   // max workspace of the multi-CTA path

__host__ __device__ inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Workspace carving of the multi-CTA path for `gq` queries.
struct WsD {
    uint32_t *keys;   // [gq][key_stride]
    uint32_t *hist;   // [gq][kHistBins]          zero between calls
    uint32_t *meta;   // [gq][kMetaWords]         zero between calls
    uint64_t *sel;    // [gq][top_k]
    uint64_t *cand;   // [gq][cand_stride]
    int64_t key_stride, cand_stride;
};

__host__ __device__ inline int64_t wsd_bytes_per_query(int64_t max_n, int top_k)
{
    return align_up(max_n, 64) * 4 + kHistBins * 4 + kMetaWords * 4 + align_up(top_k, 32) * 8 +
           align_up(max_n, 32) * 8;
}

inline WsD carve_wsd(void *ws, int64_t gq, int64_t max_n, int top_k)
{
    WsD w;
    char *p = static_cast<char *>(ws);
    w.key_stride = align_up(max_n, 64);
    w.cand_stride = align_up(max_n, 32);
    w.hist = reinterpret_cast<uint32_t *>(p);
    p += align_up(gq * kHistBins * 4, 256);
    w.meta = reinterpret_cast<uint32_t *>(p);
    p += align_up(gq * kMetaWords * 4, 256);
    w.keys = reinterpret_cast<uint32_t *>(p);
    p += align_up(gq * w.key_stride * 4, 256);
    w.sel = reinterpret_cast<uint64_t *>(p);
    p += align_up(gq * align_up(top_k, 32) * 8, 256);
    w.cand = reinterpret_cast<uint64_t *>(p);
    return w;
}

inline int64_t wsd_total_bytes(int64_t gq, int64_t max_n, int top_k)
{
    return align_up(gq * kHistBins * 4, 256) + align_up(gq * kMetaWords * 4, 256) +
           align_up(gq * align_up(max_n, 64) * 4, 256) + align_up(gq * align_up(top_k, 32) * 8, 256) +
           align_up(gq * align_up(max_n, 32) * 8, 256);
}

// ---------------------------------------------------------------------------
// shared pieces
// ---------------------------------------------------------------------------
template <int DI>
__device__ __forceinline__ void load_qsum(const uint16_t *__restrict__ qI, int64_t qi, int HI, float *s_q)
{
    for (int i = threadIdx.x; i < DI; i += blockDim.x) {
        float s = 0.f;
        for (int h = 0; h < HI; h++) {
            const uint32_t bits = __ldg(qI + (qi * HI + h) * DI + i);
            s += __uint_as_float(bits << 16);
        }
        s_q[i] = s;
    }
}

template <int DI>
__device__ __forceinline__ float score_row(const uint16_t *__restrict__ krow, const float *s_q)
{
    const uint4 *p = reinterpret_cast<const uint4 *>(krow);
    uint4 v[DI / 8];
#pragma unroll
    for (int c = 0; c < DI / 8; c++) v[c] = __ldg(p + c);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < DI / 8; c++) {
        const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            acc = fmaf(s_q[8 * c + 2 * k], bf16_lo(w[k]), acc);
            acc = fmaf(s_q[8 * c + 2 * k + 1], bf16_hi(w[k]), acc);
        }
    }
    return acc;
}

__device__ __forceinline__ void write_row_padding(int32_t *idx_row, float *score_row_out, int from, int top_k)
{
    for (int i = from + threadIdx.x; i < top_k; i += blockDim.x) {
        idx_row[i] = -1;
        if (score_row_out) score_row_out[i] = -INFINITY;
    }
}

__device__ __forceinline__ bool entry_count_ok(const int64_t *, const QueryPos &p, int ratio)
{
    return p.ne == p.L / ratio && p.t >= 0 && p.t < p.L;
}

// ---------------------------------------------------------------------------
// path 1: one CTA per query, key row in shared memory
// ---------------------------------------------------------------------------
template <int DI>
__global__ void __launch_bounds__(kCtaThreads)
index_topk_cta_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                      const int64_t *__restrict__ cu_csa, int64_t q_begin, const uint16_t *__restrict__ qI,
                      const uint16_t *__restrict__ kI, int HI, int ratio, int top_k, int n_cap,
                      int32_t *__restrict__ idx_out, float *__restrict__ score_out, int *err)
{
    extern __shared__ uint32_t s_keys[];
    __shared__ float s_q[DI];
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_w[2 * (kCtaThreads / 32) + 1];
    __shared__ uint32_t s_digit, s_above;

    const int tid = threadIdx.x;
    const int64_t qi = q_begin + blockIdx.x;
    const QueryPos p = query_pos(cu_kv, cu_q, cu_csa, batch, qi);
    int32_t *idx_row = idx_out + qi * top_k;
    float *sc_row = score_out ? score_out + qi * top_k : nullptr;
    const int64_t n64 = (p.t + 1) / ratio;
    if (!entry_count_ok(cu_csa, p, ratio) || n64 > n_cap) {
        if (tid == 0) set_error(err, CSA_ERR_DEVICE);
        write_row_padding(idx_row, sc_row, 0, top_k);
        return;
    }
    const int n = (int)n64;
    const uint16_t *kbase = kI + p.e0 * DI;

    load_qsum<DI>(qI, qi, HI, s_q);
    __syncthreads();
    for (int j = tid; j < n; j += kCtaThreads) s_keys[j] = score_key(score_row<DI>(kbase + (int64_t)j * DI, s_q));
    __syncthreads();

    if (n <= top_k) {
        for (int i = tid; i < n; i += kCtaThreads) {
            idx_row[i] = i;
            if (sc_row) sc_row[i] = key_score(s_keys[i]);
        }
        write_row_padding(idx_row, sc_row, n, top_k);
        return;
    }

    // exact k-th largest key: four 8-bit radix passes
    uint32_t prefix = 0, pmask = 0, remaining = (uint32_t)top_k;
    for (int sh = 24; sh >= 0; sh -= 8) {
        for (int i = tid; i < 256; i += kCtaThreads) s_hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < n; base += kCtaThreads) {
            const int j = base + tid;
            const uint32_t key = j < n ? s_keys[j] : 0u;
            hist_add(s_hist, (key >> sh) & 255u, j < n && (key & pmask) == prefix);
        }
        __syncthreads();
        if (tid < 32) find_digit_256(s_hist, remaining, &s_digit, &s_above);
        __syncthreads();
        remaining -= s_above;
        prefix |= s_digit << sh;
        pmask |= 255u << sh;
        __syncthreads();
    }
    const uint32_t kstar = prefix;
    const uint32_t need_eq = remaining;   // members equal to kstar still to take, lowest index first

    // one ordered pass: emit the selection in ascending index order
    uint32_t sel_base = 0, eq_base = 0;
    for (int base = 0; base < n; base += kCtaThreads) {
        const int j = base + tid;
        const uint32_t key = j < n ? s_keys[j] : 0u;
        const bool gt = j < n && key > kstar;
        const bool eq = j < n && key == kstar;
        uint32_t eq_tot, sel_tot;
        const uint32_t eq_rank = eq_base + block_scan<kCtaThreads>(eq ? 1u : 0u, s_w, eq_tot);
        const bool sel = gt || (eq && eq_rank < need_eq);
        const uint32_t pos = sel_base + block_scan<kCtaThreads>(sel ? 1u : 0u, s_w, sel_tot);
        if (sel && pos < (uint32_t)top_k) {
            idx_row[pos] = j;
            if (sc_row) sc_row[pos] = key_score(key);
        }
        eq_base += eq_tot;
        sel_base += sel_tot;
    }
    if (tid == 0 && sel_base != (uint32_t)top_k) set_error(err, CSA_ERR_DEVICE);
}

// ---------------------------------------------------------------------------
// path 2: many CTAs per query
// ---------------------------------------------------------------------------
__device__ __forceinline__ int64_t chunks_of(int64_t n) { return n <= 0 ? 1 : (n + kScanChunk - 1) / kScanChunk; }

template <int DI>
__global__ void __launch_bounds__(kScanThreads)
index_scan_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                  const int64_t *__restrict__ cu_csa, int64_t q_begin, const uint16_t *__restrict__ qI,
                  const uint16_t *__restrict__ kI, int HI, int ratio, int top_k, WsD w, int32_t *__restrict__ idx_out,
                  float *__restrict__ score_out, int *err)
{
    __shared__ float s_q[DI];
    __shared__ uint32_t s_hist[kHistBins];
    __shared__ uint32_t s_sum[2 * (kScanThreads / 32) + 1];
    __shared__ int s_last;

    griddep_launch();   // the filter may launch now; it waits for this grid to finish
    const int tid = threadIdx.x;
    const int64_t qg = blockIdx.y;
    const int64_t qi = q_begin + qg;
    const QueryPos p = query_pos(cu_kv, cu_q, cu_csa, batch, qi);
    const int64_t n = (p.t + 1) / ratio;
    const int64_t nchunks = chunks_of(n);
    if ((int64_t)blockIdx.x >= nchunks) return;
    if (!entry_count_ok(cu_csa, p, ratio) || n > w.key_stride) {
        if (blockIdx.x == 0) {
            if (tid == 0) set_error(err, CSA_ERR_DEVICE);
            write_row_padding(idx_out + qi * top_k, score_out ? score_out + qi * top_k : nullptr, 0, top_k);
        }
        return;
    }
    for (int i = tid; i < kHistBins; i += kScanThreads) s_hist[i] = 0;
    load_qsum<DI>(qI, qi, HI, s_q);
    __syncthreads();

    // Coalesced scan: LPR lanes read one key row (16 bytes each), so one warp
    // load covers 32/LPR consecutive rows; the lanes' partial dot products are
    // summed with shuffles.  Each warp owns a contiguous run of the chunk.
    constexpr int LPR = DI / 8;                         // lanes per key row
    constexpr int RPW = 32 / LPR;                       // rows per warp load
    constexpr int ROWS_W = kScanChunk / (kScanThreads / 32);
    constexpr int ITER = ROWS_W / RPW;
    constexpr int UNR = ITER < 8 ? ITER : 8;
    static_assert(ITER % UNR == 0, "scan unroll");
    const int lane = tid & 31, warp = tid >> 5;
    const int cg = lane % LPR, sub = lane / LPR;
    float qv[8];
#pragma unroll
    for (int x = 0; x < 8; x++) qv[x] = s_q[cg * 8 + x];
    const uint16_t *kbase = kI + p.e0 * DI;
    uint32_t *keys = w.keys + qg * w.key_stride;
    const int64_t r0 = (int64_t)blockIdx.x * kScanChunk + warp * ROWS_W + sub;
    for (int it0 = 0; it0 < ITER; it0 += UNR) {
        uint4 v[UNR];
#pragma unroll
        for (int u = 0; u < UNR; u++) {
            const int64_t j = r0 + (int64_t)(it0 + u) * RPW;
            v[u] = j < n ? __ldg(reinterpret_cast<const uint4 *>(kbase + j * DI) + cg) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < UNR; u++) {
            const int64_t j = r0 + (int64_t)(it0 + u) * RPW;
            const uint32_t wd[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < 4; k++) {
                acc = fmaf(qv[2 * k], bf16_lo(wd[k]), acc);
                acc = fmaf(qv[2 * k + 1], bf16_hi(wd[k]), acc);
            }
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            const bool valid = cg == 0 && j < n;
            const uint32_t key = score_key(acc);
            if (valid) keys[j] = key;
            if (valid) atomicAdd(&s_hist[key >> (32 - kHistBits)], 1u);   // few lanes per step: no aggregation
        }
    }
    __syncthreads();
    uint32_t *ghist = w.hist + qg * kHistBins;
    for (int i = tid; i < kHistBins; i += kScanThreads) {
        const uint32_t c = s_hist[i];
        if (c) atomicAdd(ghist + i, c);
    }
    __threadfence();
    __syncthreads();
    uint32_t *meta = w.meta + qg * kMetaWords;
    if (tid == 0) s_last = atomicAdd(meta + 0, 1u) == (uint32_t)(nchunks - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // last CTA of this query: locate the bin of the k-th largest key
    const int64_t k_eff = n < top_k ? n : top_k;
    if (n <= top_k) {
        if (tid == 0) {
            meta[4] = 0xffffffffu;        // every bin is above: take all
            meta[5] = (uint32_t)n;
        }
    } else {
        // thread t owns bins [4095-16t-15, 4095-16t], walked from the top
        uint32_t c[16], sum = 0;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            c[i] = __ldcg(ghist + (kHistBins - 1 - 16 * tid - i));
            sum += c[i];
        }
        uint32_t tot;
        const uint32_t excl = block_scan<kScanThreads>(sum, s_sum, tot);
        if (excl < (uint32_t)k_eff && (uint32_t)k_eff <= excl + sum) {
            uint32_t acc = excl;
            for (int i = 0; i < 16; i++) {
                if (acc + c[i] >= (uint32_t)k_eff) {
                    meta[4] = (uint32_t)(kHistBins - 1 - 16 * tid - i);
                    meta[5] = acc;
                    break;
                }
                acc += c[i];
            }
        }
    }
    // leave the histogram and the ticket zeroed for the next call
    for (int i = tid; i < kHistBins; i += kScanThreads) ghist[i] = 0;
    if (tid == 0) meta[0] = 0;
}

template <int NT>
__device__ __forceinline__ void warp_append(bool flag, uint64_t value, uint32_t *counter, uint64_t *list)
{
    const unsigned m = __ballot_sync(0xffffffffu, flag);
    if (!m) return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(m) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(counter, (uint32_t)__popc(m));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (flag) list[base + __popc(m & ((1u << lane) - 1u))] = value;
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int64_t j)
{
    return ((uint64_t)key << 32) | (uint64_t)(0xffffffffu - (uint32_t)j);
}

__global__ void __launch_bounds__(kScanThreads)
index_filter_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                    const int64_t *__restrict__ cu_csa, int64_t q_begin, int ratio, int top_k, WsD w,
                    int32_t *__restrict__ idx_out, float *__restrict__ score_out, int *err)
{
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_digit, s_above, s_cnt;
    __shared__ int s_last;
    __shared__ int32_t s_idx[kMaxTopK];
    __shared__ uint32_t s_key[kMaxTopK];
    __shared__ uint64_t s_cand[kFilterSmemCand];

    griddep_launch();   // the attention after this kernel may launch now
    griddep_wait();     // the scan's key rows, histograms and boundary bins are complete
    const int tid = threadIdx.x;
    const int64_t qg = blockIdx.y;
    const int64_t qi = q_begin + qg;
    const QueryPos p = query_pos(cu_kv, cu_q, cu_csa, batch, qi);
    const int64_t n = (p.t + 1) / ratio;
    const int64_t nchunks = chunks_of(n);
    if ((int64_t)blockIdx.x >= nchunks) return;
    if (!entry_count_ok(cu_csa, p, ratio) || n > w.key_stride) return;   // reported by the scan

    uint32_t *meta = w.meta + qg * kMetaWords;
    const uint32_t bstar = meta[4];
    const uint32_t *keys = w.keys + qg * w.key_stride;
    uint64_t *sel = w.sel + qg * align_up(top_k, 32);
    uint64_t *cand = w.cand + qg * w.cand_stride;
    const int64_t c0 = (int64_t)blockIdx.x * kScanChunk;
#pragma unroll
    for (int i = 0; i < kScanChunk / kScanThreads; i++) {
        const int64_t j = c0 + i * kScanThreads + tid;
        const uint32_t key = j < n ? __ldcg(keys + j) : 0u;
        const uint32_t bin = key >> (32 - kHistBits);
        const bool above = j < n && (bstar == 0xffffffffu || bin > bstar);
        const bool at = j < n && bstar != 0xffffffffu && bin == bstar;
        warp_append<kScanThreads>(above, composite(key, j), meta + 2, sel);
        warp_append<kScanThreads>(at, composite(key, j), meta + 3, cand);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(meta + 1, 1u) == (uint32_t)(nchunks - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // last CTA of this query: resolve the boundary bin exactly
    const uint32_t n_sel = __ldcg(meta + 2);
    const uint32_t n_cand = __ldcg(meta + 3);
    const int64_t k_eff = n < top_k ? n : top_k;
    const uint32_t need = (uint32_t)k_eff - __ldcg(meta + 5);   // from the candidates
    // the candidates are read once into shared memory when they fit; the radix
    // passes and the gather below then read them from there
    const bool cand_smem = n_cand <= (uint32_t)kFilterSmemCand;
    if (cand_smem)
        for (uint32_t c = tid; c < n_cand; c += kScanThreads) s_cand[c] = __ldcg(cand + c);
    __syncthreads();
    auto cand_at = [&](uint32_t c) -> uint64_t { return cand_smem ? s_cand[c] : __ldcg(cand + c); };
    // composite keys of candidates share their top 12 bits; select on bits 51..0
    uint64_t prefix = 0, hmask = 0;
    bool take_none = need == 0;
    if (need > 0 && need < n_cand) {
        uint32_t remaining = need;
        for (int sh = 44; sh >= -4; sh -= 8) {
            const int s = sh < 0 ? 0 : sh;
            const uint64_t dmask = sh < 0 ? 0xfull : 0xffull;
            for (int i = tid; i < 256; i += kScanThreads) s_hist[i] = 0;
            __syncthreads();
            for (uint32_t base = 0; base < n_cand; base += kScanThreads) {
                const uint32_t c = base + tid;
                const uint64_t ck = c < n_cand ? cand_at(c) : 0ull;
                hist_add(s_hist, (uint32_t)((ck >> s) & dmask), c < n_cand && (ck & hmask) == prefix);
            }
            __syncthreads();
            if (tid < 32) find_digit_256(s_hist, remaining, &s_digit, &s_above);
            __syncthreads();
            const uint32_t dgt = s_digit;
            remaining -= s_above;
            prefix |= (uint64_t)dgt << s;
            hmask |= dmask << s;
            const bool done = s_hist[dgt] == remaining;
            __syncthreads();
            if (done) break;
        }
    }
    // gather the winners
    if (tid == 0) s_cnt = 0;
    __syncthreads();
    for (uint32_t c = tid; c < n_sel; c += kScanThreads) {
        const uint64_t ck = __ldcg(sel + c);
        const uint32_t pos = atomicAdd(&s_cnt, 1u);
        if (pos < kMaxTopK) {
            s_idx[pos] = (int32_t)(0xffffffffu - (uint32_t)ck);
            s_key[pos] = (uint32_t)(ck >> 32);
        }
    }
    if (!take_none) {
        for (uint32_t c = tid; c < n_cand; c += kScanThreads) {
            const uint64_t ck = cand_at(c);
            if ((ck & hmask) >= prefix) {
                const uint32_t pos = atomicAdd(&s_cnt, 1u);
                if (pos < kMaxTopK) {
                    s_idx[pos] = (int32_t)(0xffffffffu - (uint32_t)ck);
                    s_key[pos] = (uint32_t)(ck >> 32);
                }
            }
        }
    }
    __syncthreads();
    const uint32_t got = s_cnt;
    if (tid == 0 && got != (uint32_t)k_eff) set_error(err, CSA_ERR_DEVICE);
    int npow = 1;
    while (npow < (int)k_eff) npow <<= 1;
    for (int i = (int)(got < (uint32_t)kMaxTopK ? got : (uint32_t)kMaxTopK) + tid; i < npow; i += kScanThreads) {
        s_idx[i] = 0x7fffffff;
        s_key[i] = 0;
    }
    __syncthreads();
    // bitonic sort by index, ascending
    for (int size = 2; size <= npow; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < npow; i += kScanThreads) {
                const int jj = i ^ stride;
                if (jj > i) {
                    const bool up = (i & size) == 0;
                    const int32_t a = s_idx[i], bb = s_idx[jj];
                    if ((a > bb) == up) {
                        s_idx[i] = bb;
                        s_idx[jj] = a;
                        const uint32_t t = s_key[i];
                        s_key[i] = s_key[jj];
                        s_key[jj] = t;
                    }
                }
            }
            __syncthreads();
        }
    }
    int32_t *idx_row = idx_out + qi * top_k;
    float *sc_row = score_out ? score_out + qi * top_k : nullptr;
    for (int i = tid; i < top_k; i += kScanThreads) {
        const bool v = i < k_eff && s_idx[i] != 0x7fffffff;
        idx_row[i] = v ? s_idx[i] : -1;
        if (sc_row) sc_row[i] = v ? key_score(s_key[i]) : -INFINITY;
    }
    // leave the counters and the boundary record zeroed for the next call (every
    // other CTA of this query read meta[4] before taking its ticket)
    if (tid == 0) {
        meta[1] = 0;
        meta[2] = 0;
        meta[3] = 0;
        meta[4] = 0;
        meta[5] = 0;
    }
}

// ---------------------------------------------------------------------------
// path 3 (decode-sized batches, rows of up to kSelMaxN entries): a scan that
// only streams, then one selecting cluster per query.
//
// index_chunk_scan_kernel: each CTA takes a run of 32 KiB chunks of one
// query's indexer keys, streamed through a ring of three shared-memory stages
// by bulk copies (two CTAs per SM keep six chunks in flight), scores their
// rows, stores their keys and adds its histogram of the keys' top 12 bits
// into the query's global histogram (reductions, nothing waits on them).
//
// index_select_kernel: a cluster of kSelCluster CTAs per query holds the
// query's whole key row in registers (consecutive segments per CTA, a
// contiguous segment per thread) after one round trip.  Every CTA finds the
// 12-bit bin of the k-th key from the histogram and publishes its keys in
// that bin as (key, index) candidates; each CTA then gathers the cluster's
// candidates through distributed shared memory and ranks its own among them
// (key descending, index ascending), which decides the boundary exactly.
// With more candidates than the lists hold (heavy ties) the bin is refined
// 8 + 8 + 4 bits at a time instead, the CTAs' histograms summed over the
// cluster.  The selection is written in index order after a block-wide scan
// and a cluster-wide prefix of the CTAs' counts.  The cluster returns the
// histogram to zero.
// ---------------------------------------------------------------------------
// Sums V partial values per lane over groups of lanes (lane bits below 2M)
// so that the sums end spread over the group: at a mask bit m with v > 1
// values left, the lanes with bit m set keep the upper half of the values and
// send the lower half, the others the reverse, and each adds what it
// receives; with one value left the remaining bits are plain xor reductions.
// Lane L ends with its first max(1, V / 2M) entries holding the full sums of
// the original entries j + off(L), off(L) = sum over the halving steps of
// (bit m of L) * v / 2.
template <int V, int M>
__device__ __forceinline__ void row_butterfly(float *a, int lane)
{
    if constexpr (M >= 1) {
        if constexpr (V > 1) {
            const bool hi = (lane & M) != 0;
#pragma unroll
            for (int j = 0; j < V / 2; j++) {
                const float send = hi ? a[j] : a[j + V / 2];
                const float keep = hi ? a[j + V / 2] : a[j];
                a[j] = keep + __shfl_xor_sync(0xffffffffu, send, M);
            }
            row_butterfly<V / 2, M / 2>(a, lane);
        } else {
            a[0] += __shfl_xor_sync(0xffffffffu, a[0], M);
            row_butterfly<1, M / 2>(a, lane);
        }
    }
}

constexpr int kChunkBytes = 32 * 1024;
constexpr int kScanStages = 3;   // chunks in flight per CTA (two CTAs per SM)

template <int DI, bool FP8>
__global__ void __launch_bounds__(kScanThreads, 2)
index_chunk_scan_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                        const int64_t *__restrict__ cu_csa, int64_t q_begin, const uint16_t *__restrict__ qI,
                        const void *__restrict__ kI_, const float *__restrict__ k_scale, int HI, int ratio, int cpc,
                        WsD w, int *err)
{
    // bf16 keys: 2 DI bytes per row; FP8 keys: DI bytes per row and a scale
    constexpr int RB = FP8 ? DI : 2 * DI;
    constexpr int ROWS = kChunkBytes / RB;
    const uint8_t *kI = static_cast<const uint8_t *>(kI_);
    constexpr int LPR = DI / 8;                         // lanes per key row
    constexpr int RPW = 32 / LPR;                       // rows per warp step
    constexpr int NWARP = kScanThreads / 32;
    extern __shared__ __align__(128) uint8_t s_rows[];  // kScanStages chunks
    __shared__ float s_q[DI];
    // the CTA's histogram of the keys' top 12 bits, two 16-bit counts per word
    // (bins 2i, 2i + 1): at most cpc x ROWS <= 65535 keys per CTA (the launcher
    // bounds cpc), and half the shared memory lets a CTA of the step's
    // compression stay on the SM beside two scan CTAs
    __shared__ uint32_t s_hist[kHistBins / 2];
    __shared__ __align__(8) uint64_t s_bar[kScanStages];

    const int tid = threadIdx.x;
    const int64_t qg = blockIdx.y;
    const int64_t qi = q_begin + qg;
    const QueryPos p = query_pos(cu_kv, cu_q, cu_csa, batch, qi);
    const int64_t n = (p.t + 1) / ratio;
    const int64_t r_begin = (int64_t)blockIdx.x * cpc * ROWS;
    if (r_begin >= n || !entry_count_ok(cu_csa, p, ratio) || n > w.key_stride) {   // (errors: reported by the select)
        griddep_wait();
        return;
    }
    const int64_t r_end = n - r_begin < (int64_t)cpc * ROWS ? n : r_begin + (int64_t)cpc * ROWS;
    const int nchunks = (int)((r_end - r_begin + ROWS - 1) / ROWS);
    const uint8_t *kbase = kI + (p.e0 + r_begin) * RB;
    const float *sbase = FP8 ? k_scale + p.e0 + r_begin : nullptr;
    auto rows_of = [&](int c) { return (int)(r_end - r_begin - (int64_t)c * ROWS < ROWS ? r_end - r_begin - (int64_t)c * ROWS : ROWS); };
    auto issue = [&](int c) {
        const int s = c % kScanStages;
        const uint32_t bytes = (uint32_t)rows_of(c) * RB;
        mbar_expect_tx(smem_u32(s_bar + s), bytes);
        bulk_g2s(smem_u32(s_rows + s * kChunkBytes), kbase + (int64_t)c * ROWS * RB, bytes, smem_u32(s_bar + s));
    };
    if (tid == 0) {
        for (int s = 0; s < kScanStages; s++) mbar_init(smem_u32(s_bar + s), 1);
        fence_mbar_init();
        for (int c = 0; c < nchunks && c < kScanStages; c++) issue(c);
    }
    for (int i = tid; i < kHistBins / 2; i += kScanThreads) s_hist[i] = 0;
    load_qsum<DI>(qI, qi, HI, s_q);
    __syncthreads();
    const int lane = tid & 31, warp = tid >> 5;
    const int cg = lane % LPR, sub = lane / LPR;
    float qv[8];
#pragma unroll
    for (int x = 0; x < 8; x++) qv[x] = s_q[cg * 8 + x];
    uint32_t *keys = w.keys + qg * w.key_stride + r_begin;
    // Warp `warp` scores the rows wbase .. wbase + ROWS_W - 1 of every chunk,
    // RPW rows per step (LPR lanes per row, 8 elements per lane), all ITERS
    // steps' loads and products first.  A transposing butterfly then sums
    // each row over its LPR lanes and leaves whole row sums spread over the
    // lanes: lane L ends with VF of them, those of steps j + it_off(L),
    // j < VF; when LPR > ITERS, DUP lanes hold each sum and only the first
    // of them emits it.
    constexpr int ROWS_W = ROWS / NWARP;
    constexpr int ITERS = ROWS_W / RPW;
    constexpr int VF = ITERS >= LPR ? ITERS / LPR : 1;
    constexpr int DUP = LPR > ITERS ? LPR / ITERS : 1;
    static_assert(ROWS % NWARP == 0 && ROWS_W % RPW == 0 && (ITERS & (ITERS - 1)) == 0, "scan tiling");
    const int wbase = warp * ROWS_W;
    int it_off = 0;
#pragma unroll
    for (int m = LPR / 2, v = ITERS; m >= 1; m >>= 1)
        if (v > 1) {
            if (lane & m) it_off += v / 2;
            v /= 2;
        }
    const bool emits = (lane & (DUP - 1)) == 0;
    auto row_of = [&](int j) { return wbase + (j + it_off) * RPW + sub; };
    // FP8: the scales of this lane's VF rows, loaded one chunk ahead
    float sc_cur[VF], sc_nxt[VF];
    auto load_scales = [&](int c, float (&sc)[VF]) {
        const int rows = rows_of(c);
#pragma unroll
        for (int j = 0; j < VF; j++) {
            const int row = row_of(j);
            sc[j] = row < rows ? __ldg(sbase + (int64_t)c * ROWS + row) : 0.f;
        }
    };
    if constexpr (FP8) load_scales(0, sc_cur);
    for (int c = 0; c < nchunks; c++) {
        const int s = c % kScanStages;
        if constexpr (FP8) {
            if (c + 1 < nchunks) load_scales(c + 1, sc_nxt);
        }
        // each thread's own wait makes the stage's bytes visible to it; a
        // wait that gave up is acted on at the barrier that ends the chunk
        const bool landed = mbar_wait(smem_u32(s_bar + s), (uint32_t)((c / kScanStages) & 1));
        const int rows = rows_of(c);
        const uint8_t *src = s_rows + s * kChunkBytes;
        float a[ITERS];
#pragma unroll
        for (int it = 0; it < ITERS; it++) {
            const int row = wbase + it * RPW + sub;
            const bool in = row < rows;
            float acc = 0.f;
            if constexpr (FP8) {
                // 8 codes per lane; E4M3 -> f16 is exact
                const uint2 v = in ? *reinterpret_cast<const uint2 *>(src + row * RB + cg * 8) : make_uint2(0, 0);
                const uint32_t wd[2] = {v.x, v.y};
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)(wd[k >> 1] >> (16 * (k & 1)));
                    const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
                    acc = fmaf(qv[2 * k], f.x, acc);
                    acc = fmaf(qv[2 * k + 1], f.y, acc);
                }
            } else {
                const uint4 v = in ? *reinterpret_cast<const uint4 *>(src + row * RB + cg * 16) : make_uint4(0, 0, 0, 0);
                const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    acc = fmaf(qv[2 * k], bf16_lo(wd[k]), acc);
                    acc = fmaf(qv[2 * k + 1], bf16_hi(wd[k]), acc);
                }
            }
            a[it] = acc;
        }
        row_butterfly<ITERS, LPR / 2>(a, lane);
        uint32_t *kc = keys + (int64_t)c * ROWS;
#pragma unroll
        for (int j = 0; j < VF; j++) {
            const int row = row_of(j);
            const uint32_t key = score_key(FP8 ? a[j] * sc_cur[j] : a[j]);
            if (emits && row < rows) {
                kc[row] = key;
                const uint32_t bin = key >> (32 - kHistBits);
                atomicAdd(&s_hist[bin >> 1], (bin & 1u) ? 0x10000u : 1u);
            }
        }
        if constexpr (FP8) {
#pragma unroll
            for (int j = 0; j < VF; j++) sc_cur[j] = sc_nxt[j];
        }
        // stage s has been read by every thread
        if (__syncthreads_or(!landed)) {
            // the histogram stays incomplete: the select kernel sees a count
            // mismatch and pads the row
            if (tid == 0) set_error(err, CSA_ERR_TIMEOUT);
            griddep_wait();
            return;
        }
        if (tid == 0 && c + kScanStages < nchunks) issue(c + kScanStages);
        // the select kernel may launch once every CTA has scored its first
        // chunk (it waits for this grid); launched earlier, its waiting CTAs
        // hold SMs that the branch started beside the select wants
        if (c == 0) griddep_launch();
    }
    uint32_t *ghist = w.hist + qg * kHistBins;
    for (int i = tid; i < kHistBins / 2; i += kScanThreads) {
        const uint32_t pair = s_hist[i];
        if (pair & 0xffffu) atomicAdd(ghist + 2 * i, pair & 0xffffu);
        if (pair >> 16) atomicAdd(ghist + 2 * i + 1, pair >> 16);
    }
    // Launched behind another kernel (IndexArgs::pdl), this grid reads nothing
    // that kernel writes, but completes only after it: whatever waits for this
    // grid may rely on the earlier one too.
    griddep_wait();
}

// Shared memory of one select CTA.
template <int NT>
struct SelSmem {
    uint32_t cand[kSelCandCta];   // this CTA's keys in the boundary bin
    uint32_t ncand;               // read by the peers
    uint32_t hist[2][256];        // fallback refinement histograms (read by the peers)
    uint32_t tot[256];
    uint32_t cnt[2];              // this CTA's (greater, equal) counts (read by the peers)
    uint32_t off[2];
    uint32_t coff[kSelClusterMax + 1];
    uint32_t w[2 * (NT / 32) + 1];
    uint32_t digit, above, bin;
};

// The select of one query by a cluster of kSelCluster CTAs (see the kernels
// below).  On entry: big (4096 words of shared memory) holds the query's
// summed histogram (it later holds the cluster's candidates),
// ss.ncand is zero and a __syncthreads() has passed; thread t of cluster rank
// r holds the keys seg0 .. seg0 + m - 1 of the row in key[0 .. m).  A
// non-null ghist (the global histogram) is returned to zero.
template <int NT, int KPT, int CL>
__device__ __forceinline__ void select_core(SelSmem<NT> &ss, uint32_t *big, const uint32_t (&key)[KPT], int m, int64_t seg0,
                                            uint32_t rank, int64_t n, int top_k, bool bad, uint32_t *ghist,
                                            int32_t *idx_row, float *sc_row, int *err)
{
    constexpr int BPT = kHistBins / NT;                 // top-level bins per thread
    static_assert(KPT % 4 == 0 && BPT % 4 == 0 && NT >= 256 && kHistBins % CL == 0, "select tiling");
    static_assert(kSelCandTotal <= kHistBins, "the candidate list reuses the histogram stage");
    static_assert(NT * KPT < 65536, "per-CTA counts are packed in 16 bits");
    const int tid = threadIdx.x;
    // thread t takes bins 4095 - BPT t - i, i < BPT (walked from the top bin down)
    uint32_t hc[BPT], hsum = 0;
#pragma unroll
    for (int j = 0; j < BPT / 4; j++) {
        const uint4 v = reinterpret_cast<const uint4 *>(big)[(kHistBins - BPT * (tid + 1)) / 4 + j];
        hc[BPT - 1 - 4 * j] = v.x;
        hc[BPT - 2 - 4 * j] = v.y;
        hc[BPT - 3 - 4 * j] = v.z;
        hc[BPT - 4 - 4 * j] = v.w;
    }
#pragma unroll
    for (int i = 0; i < BPT; i++) hsum += hc[i];
    const uint32_t k_eff = (uint32_t)(n < top_k ? n : top_k);
    // level 1: the 12-bit bin that holds the k-th largest key
    uint32_t tot;
    const uint32_t excl = block_scan<NT>(hsum, ss.w, tot);
    if (k_eff > 0 && excl < k_eff && k_eff <= excl + hsum) {
        uint32_t acc = excl;
#pragma unroll
        for (int i = 0; i < BPT; i++) {
            if (acc + hc[i] >= k_eff) {
                ss.digit = (uint32_t)(kHistBins - 1 - BPT * tid - i);
                ss.above = acc;
                ss.bin = hc[i];
                break;
            }
            acc += hc[i];
        }
    }
    __syncthreads();
    const bool partial = !bad && tot == (uint32_t)n && k_eff < (uint32_t)n;   // the boundary bin is split
    const uint32_t b1 = ss.digit;
    // this CTA's members of the boundary bin
    if (partial) {
#pragma unroll
        for (int i = 0; i < KPT; i++) {
            if (i < m && (key[i] >> 20) == b1) {
                const uint32_t slot = atomicAdd(&ss.ncand, 1u);
                if (slot < (uint32_t)kSelCandCta) ss.cand[slot] = key[i];
            }
        }
    }
    cluster_sync();   // the histogram has been read everywhere; candidate counts are published
    if (ghist)
        for (int i = (int)rank * (kHistBins / CL) + tid; i < (int)(rank + 1) * (kHistBins / CL); i += NT) ghist[i] = 0;
    if (bad || tot != (uint32_t)n) {   // a layout error, or a chunk that did not land (reported by the scan)
        if (bad && rank == 0 && tid == 0) set_error(err, CSA_ERR_DEVICE);
        if (rank == 0) write_row_padding(idx_row, sc_row, 0, top_k);
        cluster_sync();   // no CTA leaves while a peer may still read its counts
        return;
    }
    // the k-th key kstar: keys above it are taken, keys equal to it lowest index first
    uint32_t kstar = 0, need_eq = 0xffffffffu;   // default: every key (kstar = 0 is at or below all of them)
    if (partial) {
        uint32_t remaining = k_eff - ss.above;
        if (tid < 32) {   // lane r reads rank r's count; a warp scan gives the offsets
            const uint32_t c = tid < CL ? ld_cluster_u32(cluster_map(smem_u32(&ss.ncand), (uint32_t)tid)) : 0u;
            uint32_t incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += v;
            }
            if (tid <= CL) ss.coff[tid] = incl - c;
        }
        __syncthreads();
        bool fits = ss.coff[CL] <= (uint32_t)kSelCandTotal;
        for (int r = 0; r < CL; r++) fits = fits && ss.coff[r + 1] - ss.coff[r] <= (uint32_t)kSelCandCta;
        uint32_t prefix = b1 << 20, pmask = 0xfff00000u;
        bool whole = ss.bin == remaining;   // the boundary bin is taken whole
        if (!whole && fits) {
            // gather the cluster's boundary-bin keys, then refine them here
            // 8 + 8 + 4 bits at a time (every CTA reaches the same answer)
            const uint32_t total = ss.coff[CL];
            uint32_t *all = big;
            for (uint32_t i = tid; i < total; i += NT) {
                int r = 0;
                while (i >= ss.coff[r + 1]) r++;
                all[i] = ld_cluster_u32(cluster_map(smem_u32(ss.cand + (i - ss.coff[r])), (uint32_t)r));
            }
#pragma unroll 1
            for (int level = 0; level < 3 && !whole; level++) {
                const int sh = level == 0 ? 12 : (level == 1 ? 4 : 0);
                const uint32_t dm = level == 2 ? 0xfu : 0xffu;
                for (int i = tid; i < 256; i += NT) ss.tot[i] = 0;
                __syncthreads();
                for (uint32_t i = tid; i < total; i += NT) {
                    const uint32_t k = all[i];
                    if ((k & pmask) == prefix) atomicAdd(&ss.tot[(k >> sh) & dm], 1u);
                }
                __syncthreads();
                if (tid < 32) find_digit_256(ss.tot, remaining, &ss.digit, &ss.above);
                __syncthreads();
                remaining -= ss.above;
                prefix |= ss.digit << sh;
                pmask |= dm << sh;
                whole = ss.tot[ss.digit] == remaining;
                __syncthreads();   // ss.digit, ss.above and ss.tot are rewritten by the next level
            }
        } else if (!whole) {
            // many members (heavy ties): the same refinement over the keys in
            // registers, the CTAs' histograms summed through distributed shared memory
#pragma unroll 1
            for (int level = 0; level < 3 && !whole; level++) {
                const int sh = level == 0 ? 12 : (level == 1 ? 4 : 0);
                const uint32_t dm = level == 2 ? 0xfu : 0xffu;
                uint32_t *h = ss.hist[level & 1];
                for (int i = tid; i < 256; i += NT) h[i] = 0;
                __syncthreads();
#pragma unroll
                for (int i = 0; i < KPT; i++)
                    if (i < m && (key[i] & pmask) == prefix) atomicAdd(&h[(key[i] >> sh) & dm], 1u);
                cluster_sync();
                if (tid < 256) {
                    const uint32_t a = smem_u32(h + tid);
                    uint32_t t = 0;
#pragma unroll
                    for (int r = 0; r < CL; r++) t += ld_cluster_u32(cluster_map(a, (uint32_t)r));
                    ss.tot[tid] = t;
                }
                __syncthreads();
                if (tid < 32) find_digit_256(ss.tot, remaining, &ss.digit, &ss.above);
                __syncthreads();
                remaining -= ss.above;
                prefix |= ss.digit << sh;
                pmask |= dm << sh;
                whole = ss.tot[ss.digit] == remaining;
                __syncthreads();   // ss.digit, ss.above and ss.tot are rewritten by the next level
            }
        }
        // whole: every key at or above `prefix` (its lower bits zero) is taken
        kstar = prefix;
        need_eq = whole ? 0xffffffffu : remaining;
    }
    // ordered emission: a thread's keys are contiguous in index order, and the
    // CTAs of the cluster hold consecutive segments
    uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
    for (int i = 0; i < KPT; i++) {
        n_gt += (i < m && key[i] > kstar) ? 1u : 0u;
        n_eq += (i < m && key[i] == kstar) ? 1u : 0u;
    }
    uint32_t t_both;   // (greater, equal) counts packed 16 + 16 bits: at most NT * KPT <= 65536 keys per CTA
    const uint32_t both_before = block_scan<NT>((n_eq << 16) | n_gt, ss.w, t_both);
    const uint32_t gt_before = both_before & 0xffffu, eq_before = both_before >> 16;
    if (tid == 0) {
        ss.cnt[0] = t_both & 0xffffu;
        ss.cnt[1] = t_both >> 16;
    }
    cluster_sync();
    if (tid < 32) {   // lane r < rank reads rank r's counts
        uint32_t g = 0, e = 0;
        if ((uint32_t)tid < rank) {
            g = ld_cluster_u32(cluster_map(smem_u32(ss.cnt), (uint32_t)tid));
            e = ld_cluster_u32(cluster_map(smem_u32(ss.cnt + 1), (uint32_t)tid));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, o);
            e += __shfl_xor_sync(0xffffffffu, e, o);
        }
        if (tid == 0) {
            ss.off[0] = g;
            ss.off[1] = e;
        }
    }
    cluster_arrive();   // this CTA reads no peer from here on (waited for at the end)
    // The attention after this kernel may launch now (it waits for this grid
    // on the device).  Triggered this late so that its CTAs do not sit on SMs
    // the concurrent dense branch could use.
    griddep_launch();
    __syncthreads();
    const uint32_t eq0 = ss.off[1] + eq_before;
    uint32_t pos = ss.off[0] + gt_before + (eq0 < need_eq ? eq0 : need_eq);
    uint32_t eq_rank = eq0;
#pragma unroll
    for (int i = 0; i < KPT; i++) {
        if (i >= m) continue;
        bool take = key[i] > kstar;
        if (key[i] == kstar) take = eq_rank++ < need_eq;
        if (take) {
            if (pos < (uint32_t)top_k) {
                idx_row[pos] = (int32_t)(seg0 + i);
                if (sc_row) sc_row[pos] = key_score(key[i]);
            }
            pos++;
        }
    }
    if (rank == 0) write_row_padding(idx_row, sc_row, (int)k_eff, top_k);
    if (rank == CL - 1 && tid == NT - 1 && pos != k_eff) set_error(err, CSA_ERR_DEVICE);
    cluster_wait();   // the peers have read this CTA's counts and candidates
}

// Rows of 16385-32768 entries (256 threads, 16 keys each) come in large
// batches: four CTAs per SM (64 registers a thread) let a batch's clusters
// share the GPU in fewer waves.
template <int NT, int KPT, int CL>
__global__ void __launch_bounds__(NT, (NT == 256 && KPT == 16) ? 4 : 1)
index_select_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                    const int64_t *__restrict__ cu_csa, int64_t q_begin, int ratio, int top_k, WsD w,
                    int32_t *__restrict__ idx_out, float *__restrict__ score_out, int *err)
{
    __shared__ __align__(16) SelSmem<NT> ss;
    __shared__ __align__(16) uint32_t s_big[kHistBins];

    const int tid = threadIdx.x;
    const uint32_t rank = cluster_rank();
    const int64_t qg = blockIdx.y;
    const int64_t qi = q_begin + qg;
    const QueryPos p = query_pos(cu_kv, cu_q, cu_csa, batch, qi);   // layout arrays: inputs of the call
    if (tid == 0) ss.ncand = 0;
    griddep_wait();   // every chunk's keys and histogram counts are in place
    const int64_t n = (p.t + 1) / ratio;
    int32_t *idx_row = idx_out + qi * top_k;
    float *sc_row = score_out ? score_out + qi * top_k : nullptr;
    uint32_t *ghist = w.hist + qg * kHistBins;
    // every test below gives the same answer in all CTAs of the cluster
    const bool bad = !entry_count_ok(cu_csa, p, ratio) || n > w.key_stride || n > (int64_t)CL * NT * KPT;

    // one round trip: this thread's key segment and the histogram (coalesced, into shared memory)
    const int64_t seg0 = ((int64_t)rank * NT + tid) * KPT;
    const int m = bad ? 0 : (int)(n - seg0 < 0 ? 0 : (n - seg0 < KPT ? n - seg0 : KPT));   // valid keys here
    const uint32_t *krow = w.keys + qg * w.key_stride;
    uint32_t key[KPT];
#pragma unroll
    for (int i = 0; i < KPT; i += 4) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (i < m) v = __ldcg(reinterpret_cast<const uint4 *>(krow + seg0 + i));
        key[i] = v.x;
        key[i + 1] = v.y;
        key[i + 2] = v.z;
        key[i + 3] = v.w;
    }
    for (int i = tid; i < kHistBins / 4; i += NT)
        reinterpret_cast<uint4 *>(s_big)[i] = bad ? make_uint4(0, 0, 0, 0) : __ldcg(reinterpret_cast<const uint4 *>(ghist) + i);
    __syncthreads();
    select_core<NT, KPT, CL>(ss, s_big, key, m, seg0, rank, n, top_k, bad, ghist, idx_row, sc_row, err);
}

constexpr int64_t kSelMaxN = (int64_t)kSelCluster * 1024 * 32;   // longest row the select cluster holds (entries)
constexpr int64_t kCompressBehindScan = 4096;   // scanned keys per SM that hide a fused compression

bool use_cta_path(const IndexArgs &a)
{
    const int64_t max_n = a.max_kv_len / a.ratio;
    return max_n <= kCtaMaxN && a.total_q >= 1024;
}

int64_t group_size(const IndexArgs &a)
{
    const int64_t max_n = a.max_kv_len / a.ratio;
    const int64_t per_q = wsd_bytes_per_query(max_n, a.top_k);
    int64_t g = kGroupBudget / per_q;
    if (g < 1) g = 1;
    if (g > 65535) g = 65535;   // queries ride on grid.y
    return g < a.total_q ? g : a.total_q;
}

int device_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

// The select cluster for rows of up to max_n entries: kSelCluster CTAs of NT
// threads holding KPT keys each.
cudaError_t launch_select(const IndexArgs &a, int64_t max_n, int64_t q0, int64_t nq, const WsD &w, cudaStream_t st)
{
    auto go = [&](auto kern, int nt, int cl) {
        return launch_kernel_cluster("index_select", kern, dim3((unsigned)cl, (unsigned)nq), dim3(nt), 0, st, true,
                                     (unsigned)cl, a.batch, a.cu_kv, a.cu_q, a.cu_csa, q0, a.ratio, a.top_k, w,
                                     a.idx_out, a.score_out, a.err);
    };
    if (max_n <= kSelCluster * 256 * 8) return go(index_select_kernel<256, 8, kSelCluster>, 256, kSelCluster);
    if (max_n <= kSelCluster * 256 * 16) return go(index_select_kernel<256, 16, kSelCluster>, 256, kSelCluster);
    if (max_n <= kSelCluster * 512 * 32) return go(index_select_kernel<512, 32, kSelCluster>, 512, kSelCluster);
    // the longest rows: 16 CTAs per query, half the keys per thread
    return go(index_select_kernel<1024, 16, kSelClusterMax>, 1024, kSelClusterMax);
}

template <int DI>
cudaError_t launch_index_t(const IndexArgs &a_in, cudaStream_t st)
{
    IndexArgs a = a_in;
    if (a.total_q <= 0) return cudaSuccess;
    const int64_t max_n = a.max_kv_len / a.ratio;
    // scan_done: after the last key scan of the multi-kernel paths; the
    // single-kernel paths mark it up front (their kernel holds the GPU to the end)
    auto mark = [&]() -> cudaError_t { return a.scan_done ? cudaEventRecord(a.scan_done, st) : cudaSuccess; };
    const bool fp8 = a.fp8;   // FP8 keys: the chunk scan and the select only
    const bool single = !fp8 && (index_tc_applicable(a) || index_block_applicable(a) || use_cta_path(a));
    // A compression of the same call runs ahead of the indexer, except behind a
    // chunk scan long enough to hide it (at least kCompressBehindScan keys per
    // SM: measured, ragged decode 98.3 -> 94.7 us and 1M decode 69.0 -> 66.2 us,
    // while a 64K decode's 11 us scan cannot hide it: 34.8 -> 36.9 us); there it
    // starts after the first key scan, whose CTAs then hold every SM from the start.
    const CompressArgs *comp = a.compress;
    a.compress = nullptr;
    const bool behind_scan = !single && max_n <= kSelMaxN &&
                             a.total_q * max_n >= kCompressBehindScan * (int64_t)device_sms();
    if (comp && !behind_scan) {
        CompressArgs c = *comp;
        c.pdl = false;
        cudaError_t e = launch_compress(c, st);
        if (e != cudaSuccess) return e;
        a.pdl = true;
        comp = nullptr;
    }
    if (single) {
        cudaError_t e = mark();
        if (e != cudaSuccess) return e;
    }
    if (!fp8 && index_tc_applicable(a)) return launch_index_tc(a, st);
    if (!fp8 && index_block_applicable(a)) return launch_index_block(a, st);
    if (!fp8 && use_cta_path(a)) {
        const int64_t nsm = max_n < 1 ? 1 : max_n;
        const size_t smem = (size_t)nsm * 4;
        for (int64_t q0 = 0; q0 < a.total_q; q0 += 1 << 30) {
            const int64_t nq = a.total_q - q0 < (1 << 30) ? a.total_q - q0 : (1 << 30);
            cudaError_t e = launch_kernel("index_topk_cta", index_topk_cta_kernel<DI>, dim3((unsigned)nq),
                                          dim3(kCtaThreads), smem, st, false, a.batch, a.cu_kv, a.cu_q, a.cu_csa, q0,
                                          a.q_idx, a.k_idx, a.n_heads_idx, a.ratio, a.top_k, (int)nsm,
                                          a.idx_out, a.score_out, a.err);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    const int64_t gq = group_size(a);
    const int64_t nchunks = (max_n <= 0 ? 1 : (max_n + kScanChunk - 1) / kScanChunk);
    WsD w = carve_wsd(a.ws, gq, max_n < 1 ? 1 : max_n, a.top_k);
    if (max_n <= kSelMaxN) {
        const int ROWS = kChunkBytes / (fp8 ? DI : 2 * DI);
        const int64_t nch = max_n <= 0 ? 1 : (max_n + ROWS - 1) / ROWS;
        // chunks per CTA: the group's chunks over about two CTAs per SM
        const int64_t slots = 2 * (int64_t)device_sms();
        for (int64_t q0 = 0; q0 < a.total_q; q0 += gq) {
            const int64_t nq = a.total_q - q0 < gq ? a.total_q - q0 : gq;
            int64_t cpc = (nq * nch + slots - 1) / slots;
            if (cpc > 65535 / ROWS) cpc = 65535 / ROWS;   // the scan's 16-bit per-CTA bin counts
            if (cpc < 1) cpc = 1;
            if (cpc > nch) cpc = nch;
            const int64_t gx = (nch + cpc - 1) / cpc;
            cudaError_t e =
                fp8 ? launch_kernel("index_scan", index_chunk_scan_kernel<DI, true>, dim3((unsigned)gx, (unsigned)nq),
                                        dim3(kScanThreads), (size_t)kScanStages * kChunkBytes, st, a.pdl, a.batch,
                                        a.cu_kv, a.cu_q, a.cu_csa, q0, a.q_idx, (const void *)a.k_fp8, a.k_scale,
                                        a.n_heads_idx, a.ratio, (int)cpc, w, a.err)
                        : launch_kernel("index_scan", index_chunk_scan_kernel<DI, false>, dim3((unsigned)gx, (unsigned)nq),
                                        dim3(kScanThreads), (size_t)kScanStages * kChunkBytes, st, a.pdl, a.batch,
                                        a.cu_kv, a.cu_q, a.cu_csa, q0, a.q_idx, (const void *)a.k_idx, a.k_scale,
                                        a.n_heads_idx, a.ratio, (int)cpc, w, a.err);
            if (e == cudaSuccess && comp) {
                // the compression overlaps the key scan (it starts once every scan CTA
                // has scored its first chunk) and completes only after it
                CompressArgs c = *comp;
                c.pdl = true;
                e = launch_compress(c, st);
                comp = nullptr;
            }
            if (e == cudaSuccess && q0 + nq >= a.total_q) e = mark();
            if (e != cudaSuccess) return e;
            e = launch_select(a, max_n, q0, nq, w, st);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    if (fp8) return cudaErrorInvalidValue;   // rows longer than index_fp8_max_n(): refused by the caller
    for (int64_t q0 = 0; q0 < a.total_q; q0 += gq) {
        const int64_t nq = a.total_q - q0 < gq ? a.total_q - q0 : gq;
        dim3 grid((unsigned)nchunks, (unsigned)nq);
        cudaError_t e = launch_kernel("index_scan", index_scan_kernel<DI>, grid, dim3(kScanThreads), 0, st, false,
                                      a.batch, a.cu_kv, a.cu_q, a.cu_csa, q0, a.q_idx, a.k_idx, a.n_heads_idx,
                                      a.ratio, a.top_k, w, a.idx_out, a.score_out, a.err);
        if (e == cudaSuccess && q0 + nq >= a.total_q) e = mark();
        if (e != cudaSuccess) return e;
        e = launch_kernel("index_filter", index_filter_kernel, grid, dim3(kScanThreads), 0, st, true, a.batch, a.cu_kv,
                          a.cu_q, a.cu_csa, q0, a.ratio, a.top_k, w, a.idx_out, a.score_out, a.err);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

bool index_supported(int n_heads_idx, int d_idx, int top_k)
{
    return n_heads_idx >= 1 && n_heads_idx <= 16 && (d_idx == 32 || d_idx == 64 || d_idx == 128) && top_k >= 1 &&
           top_k <= kMaxTopK;
}

size_t index_workspace_bytes(const IndexArgs &a)
{
    if (a.total_q <= 0) return 0;
    if (index_tc_applicable(a)) return index_tc_ws_bytes(a);
    if (index_block_applicable(a)) return index_block_ws_bytes(a);
    if (use_cta_path(a)) return 0;
    const int64_t max_n = a.max_kv_len / a.ratio;
    return (size_t)wsd_total_bytes(group_size(a), max_n < 1 ? 1 : max_n, a.top_k);
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) indexer keys: one warp per key row.  Lane l holds values
// l*V .. l*V + V - 1 (V = d_idx / 32); the row's absolute maximum a gives
// inv = 448 / a and scale = a / 448 (IEEE fp32), each value k * inv is
// converted to E4M3 rounding to nearest even and saturating at +-448.
// ---------------------------------------------------------------------------
// One key row by one warp (every lane calls it with the same row).
template <int DI>
__device__ __forceinline__ void quantize_row(const uint16_t *__restrict__ k_idx, int64_t row, uint8_t *__restrict__ k_fp8,
                                             float *__restrict__ k_scale)
{
    constexpr int V = DI / 32;
    static_assert(DI % 32 == 0 && V >= 1 && V <= 4, "row width");
    const int lane = threadIdx.x & 31;
    const uint16_t *src = k_idx + row * DI + lane * V;
    float v[V];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < V; i++) {
        v[i] = __uint_as_float((uint32_t)__ldg(src + i) << 16);
        amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
    uint8_t code[V];
#pragma unroll
    for (int i = 0; i < V; i++)
        code[i] = amax > 0.f ? (uint8_t)__nv_cvt_float_to_fp8(__fmul_rn(v[i], inv), __NV_SATFINITE, __NV_E4M3)
                             : (uint8_t)0;
    uint8_t *dst = k_fp8 + row * DI + lane * V;
#pragma unroll
    for (int i = 0; i < V; i++) dst[i] = code[i];
    if (lane == 0) k_scale[row] = __fdiv_rn(amax, 448.f);
}

// Every row of the key array.
template <int DI>
__global__ void __launch_bounds__(256)
quantize_index_keys_kernel(const uint16_t *__restrict__ k_idx, int64_t rows, uint8_t *__restrict__ k_fp8,
                           float *__restrict__ k_scale)
{
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    quantize_row<DI>(k_idx, row, k_fp8, k_scale);
}

// Only the rows of the entries that the layout's query positions close: the
// query at position t closes entry (t + 1) / ratio - 1 of its sequence when
// (t + 1) is a multiple of ratio, and no other query closes that entry.  One
// warp per query.
template <int DI>
__global__ void __launch_bounds__(256)
quantize_closed_keys_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                            const int64_t *__restrict__ cu_csa, int64_t total_q, int ratio,
                            const uint16_t *__restrict__ k_idx, uint8_t *__restrict__ k_fp8,
                            float *__restrict__ k_scale, int *err)
{
    const int64_t qi = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (qi >= total_q) return;
    const QueryPos p = query_pos(cu_kv, cu_q, cu_csa, batch, qi);
    if (!entry_count_ok(cu_csa, p, ratio)) {
        if ((threadIdx.x & 31) == 0) set_error(err, CSA_ERR_DEVICE);
        return;
    }
    if ((p.t + 1) % ratio != 0) return;
    quantize_row<DI>(k_idx, p.e0 + (p.t + 1) / ratio - 1, k_fp8, k_scale);
}

cudaError_t launch_quantize_index_keys(const uint16_t *k_idx, int64_t rows, int d_idx, uint8_t *k_fp8,
                                       float *k_scale, cudaStream_t st)
{
    if (rows <= 0) return cudaSuccess;
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)blocks);
    switch (d_idx) {
    case 32: return launch_kernel("quantize_index_keys", quantize_index_keys_kernel<32>, grid, dim3(256), 0, st, false, k_idx, rows, k_fp8, k_scale);
    case 64: return launch_kernel("quantize_index_keys", quantize_index_keys_kernel<64>, grid, dim3(256), 0, st, false, k_idx, rows, k_fp8, k_scale);
    case 128: return launch_kernel("quantize_index_keys", quantize_index_keys_kernel<128>, grid, dim3(256), 0, st, false, k_idx, rows, k_fp8, k_scale);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_quantize_closed_keys(int batch, const int64_t *cu_kv, const int64_t *cu_q, const int64_t *cu_csa,
                                        int64_t total_q, int ratio, const uint16_t *k_idx, int d_idx, uint8_t *k_fp8,
                                        float *k_scale, int *err, cudaStream_t st)
{
    if (total_q <= 0) return cudaSuccess;
    const int64_t blocks = (total_q + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)blocks);
    switch (d_idx) {
    case 32: return launch_kernel("quantize_closed_keys", quantize_closed_keys_kernel<32>, grid, dim3(256), 0, st, false, batch, cu_kv, cu_q, cu_csa, total_q, ratio, k_idx, k_fp8, k_scale, err);
    case 64: return launch_kernel("quantize_closed_keys", quantize_closed_keys_kernel<64>, grid, dim3(256), 0, st, false, batch, cu_kv, cu_q, cu_csa, total_q, ratio, k_idx, k_fp8, k_scale, err);
    case 128: return launch_kernel("quantize_closed_keys", quantize_closed_keys_kernel<128>, grid, dim3(256), 0, st, false, batch, cu_kv, cu_q, cu_csa, total_q, ratio, k_idx, k_fp8, k_scale, err);
    default: return cudaErrorInvalidValue;
    }
}

int64_t index_fp8_max_n() { return kSelMaxN; }

size_t index_fp8_workspace_bytes(const IndexArgs &a)
{
    if (a.total_q <= 0) return 0;
    const int64_t max_n = a.max_kv_len / a.ratio;
    return (size_t)wsd_total_bytes(group_size(a), max_n < 1 ? 1 : max_n, a.top_k);
}

cudaError_t launch_index_topk(const IndexArgs &a, cudaStream_t st)
{
    switch (a.d_idx) {
    case 32: return launch_index_t<32>(a, st);
    case 64: return launch_index_t<64>(a, st);
    case 128: return launch_index_t<128>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------
// Library-owned scratch for callers that cannot allocate device memory.
//
// The multi-CTA path needs a workspace (key rows, histograms, counters and
// candidate lists).  For callers that cannot hand one over, this file-scope
// device array stands in for it.  Every device that loads this code holds
// the array until the process exits, and every call shares it: calls that
// overlap on the GPU race on it.  Its address is looked up once per device,
// with that device current (host code cannot use the symbol itself: on the
// host it names a stand-in, not device memory).
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_index_static_scratch[kIndexStaticScratchBytes];

namespace {
constexpr int kMaxStaticDevices = 64;
void *g_static_ptr[kMaxStaticDevices];
std::mutex g_static_mu;
}  // namespace

cudaError_t index_static_scratch(void **ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxStaticDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_index_static_scratch);
        if (e != cudaSuccess) return e;
        g_static_ptr[dev] = p;
    }
    *ptr = g_static_ptr[dev];
    return cudaSuccess;
}

size_t index_static_need_bytes(const IndexArgs &a)
{
    if (a.total_q > 0 && index_tc_applicable(a)) return index_tc_min_ws_bytes();
    if (a.total_q > 0 && index_block_applicable(a)) return index_block_min_ws_bytes();
    return index_workspace_bytes(a);
}

size_t index_static_zero_bytes(const IndexArgs &a)
{
    if (a.total_q <= 0 || index_tc_applicable(a) || index_block_applicable(a) || use_cta_path(a)) return 0;
    const int64_t gq = group_size(a);
    return (size_t)(align_up(gq * kHistBins * 4, 256) + align_up(gq * kMetaWords * 4, 256));
}

}  // namespace csa
