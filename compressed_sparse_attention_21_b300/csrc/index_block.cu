// Lightning indexer + top-k for prefill-sized batches ("DeepSeek-V4 core
// architecture", §2.2 CSA step 2: a light scorer rates each query against
// every compressed entry and only the top-k entries are kept).
//
// The per-query scan re-reads a sequence's indexer keys once per query; here
// a persistent CTA takes 16 consecutive queries of a sequence at a time and
// streams the sequence's keys through shared memory once for all 16:
//
//  1. Scores on the tensor cores.  The head-summed query (fp32) is split into
//     three bf16 terms (hi + mid + lo, exact to 2^-27 relative) and
//     s = sum_terms term . k is accumulated in fp32 by mma.m16n8k16 (16
//     queries x 8 entries per product, products exact).  This is the fp32
//     score of the definition up to fp32 rounding order.
//  2. A threshold per query from 256 evenly spaced entries: the sampled score
//     expected to have about 2k entries above it.  While the keys stream by,
//     only entries at or above the threshold are kept as candidates.
//  3. Exact selection among the candidates: the k-th largest key by a 4 x 8-bit
//     radix select, then every kept entry finds its output slot from prefix
//     counts over bitmaps of the entries above and equal to it (index order,
//     ties to the lower index).
//  A query whose candidates turn out fewer than min(k, n) or more than the
//  buffer holds (a sample that misjudged the distribution, many equal
//  scores) is selected exactly from all of its scores instead.  The result
//  never depends on the sample; only the amount of work does.
#include "common.cuh"
#include "launch.h"
#include "prefill_select.cuh"

namespace csa {

namespace {

constexpr int kBQ = 16;              // queries per block (M of one m16n8k16 tile)
constexpr size_t kBSlotBytes = (size_t)kBQ * kBCap * 8;   // candidate slot of one persistent CTA

template <int DI>
struct BCfg {
    static constexpr int RB = 2 * DI;            // bytes of a key row
    static constexpr int PRB = RB + 16;          // padded row stride: ldmatrix without bank conflicts
    static constexpr int CPR = RB / 16;          // 16-byte chunks per row
    static constexpr uint32_t buf_bytes = kBRows * PRB;
    // chunks in the streaming ring (all but one in flight while one is scored)
    static constexpr int NB = DI == 32 ? 6 : (DI == 64 ? 5 : 2);
    // shared-memory layout (bytes)
    static constexpr uint32_t off_buf = 0;                                   // NB chunk buffers
    static constexpr uint32_t off_qs = off_buf + NB * buf_bytes;             // [16][DI] fp32 head sums
    static constexpr uint32_t off_skey = off_qs + kBQ * DI * 4;              // [16][256] sampled keys
    static constexpr uint32_t off_gt = off_skey + kBQ * kBSample * 4;        // bitmaps and their prefixes
    static constexpr uint32_t off_eq = off_gt + kBWords * 4;
    static constexpr uint32_t off_pre = off_eq + kBWords * 4;                // packed (gt << 16 | eq) prefix
    static constexpr uint32_t off_end = off_pre + kBWords * 4;
    static constexpr size_t smem = off_end;
    // per-warp selection scratch, in the ring once the keys have streamed by:
    // a 256-bin histogram, the taken-entry bitmap and its 16-bit word prefixes
    static constexpr uint32_t warp_scratch = 256 * 4 + kBWords * 4 + kBWords * 2;
    static_assert(kBQ * warp_scratch <= NB * buf_bytes, "selection scratch fits the ring");
    static_assert(kBQ * 256 * 4 <= buf_bytes, "sampling histograms fit one chunk buffer");
    static_assert(smem <= 232448, "shared memory per CTA");
};

// m16n8k16 bf16 fragments of the 16 x DI head-summed queries, split in three
// bf16 terms: a[ks][term][4].
template <int DI>
__device__ __forceinline__ void load_a_frags(const float *qs, uint32_t (&a)[DI / 16][3][4])
{
    const int lane = threadIdx.x & 31, g = lane >> 2, c4 = lane & 3;
#pragma unroll
    for (int ks = 0; ks < DI / 16; ks++) {
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int row = g + (r & 1) * 8;
            const int col = ks * 16 + 2 * c4 + (r >> 1) * 8;
            float x0 = qs[row * DI + col], x1 = qs[row * DI + col + 1];
#pragma unroll
            for (int term = 0; term < 3; term++) {
                const uint32_t p = pack_bf16x2(x0, x1);
                a[ks][term][r] = p;
                x0 -= bf16_lo(p);
                x1 -= bf16_hi(p);
            }
        }
    }
}

// Scores of the 16 queries against the 16 entries this warp owns in a chunk
// buffer (rows 16 w .. 16 w + 15): s[tile][4] in C-fragment order.
template <int DI>
__device__ __forceinline__ void warp_scores(uint32_t buf, const uint32_t (&a)[DI / 16][3][4], float (&s)[2][4])
{
    using C = BCfg<DI>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int t = 0; t < 2; t++) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
    const int row = warp * 16 + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
    for (int ks = 0; ks < DI / 16; ks++) {
        uint32_t b0, b1, b2, b3;
        const int ch = ks * 2 + ((lane >> 3) & 1);
        ldmatrix_x4(buf + row * C::PRB + ch * 16, b0, b1, b2, b3);
#pragma unroll
        for (int term = 0; term < 3; term++) {
            mma_bf16_16816(s[0], a[ks][term], b0, b1);
            mma_bf16_16816(s[1], a[ks][term], b2, b3);
        }
    }
}

// Copy key rows into a padded chunk buffer; row r of the buffer takes entry
// row src_row(r) of the sequence, or zeros when src_row(r) < 0.
template <int DI, typename RowOf>
__device__ __forceinline__ void load_rows(uint32_t buf, const uint16_t *kseq, RowOf src_row, const uint16_t *safe)
{
    using C = BCfg<DI>;
    for (int i = threadIdx.x; i < kBRows * C::CPR; i += kBT) {
        const int r = i / C::CPR, c = i % C::CPR;
        const int64_t e = src_row(r);
        cp_async_16(buf + r * C::PRB + c * 16, e >= 0 ? (const void *)(kseq + e * DI + c * 8) : (const void *)safe,
                    e >= 0 ? 16 : 0);
    }
}

template <int DI>
__global__ void __launch_bounds__(kBT, 1)
index_block_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                   const int64_t *__restrict__ cu_csa, int64_t total_q, const uint16_t *__restrict__ qI,
                   const uint16_t *__restrict__ kI, int HI, int ratio, int top_k, uint64_t *__restrict__ cand_ws,
                   int32_t *__restrict__ idx_out, float *__restrict__ score_out, int *err)
{
    using C = BCfg<DI>;
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ BlockQ s_q[kBQ];
    __shared__ uint32_t s_tau[kBQ], s_cnt[kBQ];
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_w[2 * (kBT / 32) + 1];
    __shared__ uint32_t s_dig[2];
    __shared__ int s_need_sample;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c4 = lane & 3;
    __shared__ uint32_t s_wdig[kBQ][2];
    __shared__ int s_fall[kBQ];
    const uint32_t sbase = smem_u32(sm);
    const uint32_t buf0 = sbase + C::off_buf;
    auto bufn = [&](int i) { return buf0 + (uint32_t)i * C::buf_bytes; };
    float *qs = reinterpret_cast<float *>(sm + C::off_qs);
    uint32_t *skey = reinterpret_cast<uint32_t *>(sm + C::off_skey);
    uint64_t *cand = cand_ws + (int64_t)blockIdx.x * kBQ * kBCap;
    const int64_t nblocks = (total_q + kBQ - 1) / kBQ;

    for (int64_t blk = blockIdx.x; blk < nblocks; blk += gridDim.x) {
        const int64_t q0 = blk * kBQ;
        const int nqb = (int)(total_q - q0 < kBQ ? total_q - q0 : kBQ);
        // ---- the block's queries ----
        if (warp < kBQ) {
            const int64_t qi = q0 + (warp < nqb ? warp : 0);
            const QueryPos p = query_pos(cu_kv, cu_q, cu_csa, batch, qi);
            if (lane == 0) {
                BlockQ r;
                r.b = p.b;
                r.n = (int)((p.t + 1) / ratio);
                r.e0 = p.e0;
                r.ok = warp < nqb && p.ne == p.L / ratio && p.t >= 0 && p.t < p.L && r.n <= kBMaxN;
                s_q[warp] = r;
            }
        }
        for (int i = tid; i < kBQ * DI; i += kBT) {
            const int qq = i / DI, d = i % DI;
            float acc = 0.f;
            if (qq < nqb)
                for (int h = 0; h < HI; h++) acc += bf16_lo(__ldg(qI + ((q0 + qq) * HI + h) * DI + d));
            qs[i] = acc;
        }
        __syncthreads();
        uint32_t afr[DI / 16][3][4];
        load_a_frags<DI>(qs, afr);

        // ---- one pass per sequence present in the block (nearly always one) ----
        for (int ga = 0; ga < nqb;) {
            int gz = ga + 1;
            while (gz < nqb && s_q[gz].b == s_q[ga].b) gz++;
            int n_max = 0;
            for (int i = ga; i < gz; i++)
                if (s_q[i].ok && s_q[i].n > n_max) n_max = s_q[i].n;
            const int64_t e0 = s_q[ga].e0;
            const uint16_t *kseq = kI + e0 * DI;
            // thresholds: keep everything when the row fits the candidate buffer
            if (tid < kBQ) {
                s_tau[tid] = 0u;
                s_cnt[tid] = 0u;
            }
            if (tid == 0) {
                int need = 0;
                for (int i = ga; i < gz; i++) need |= (s_q[i].ok && s_q[i].n > kBCap);
                s_need_sample = need;
            }
            __syncthreads();
            if (s_need_sample) {
                // sampled rows j_s = s * n_max / 256 of the sequence
                load_rows<DI>(buf0, kseq, [&](int r) -> int64_t { return (int64_t)r * n_max / kBSample; }, kI);
                cp_async_commit();
                cp_async_wait<0>();
                __syncthreads();
                float sc[2][4];
                warp_scores<DI>(buf0, afr, sc);
#pragma unroll
                for (int t = 0; t < 2; t++)
#pragma unroll
                    for (int r = 0; r < 4; r++) {
                        const int qq = g + (r >> 1) * 8;
                        const int s_i = warp * 16 + t * 8 + 2 * c4 + (r & 1);
                        const int64_t j = (int64_t)s_i * n_max / kBSample;
                        const bool v = qq >= ga && qq < gz && s_q[qq].ok && j < s_q[qq].n;
                        skey[qq * kBSample + s_i] = v ? score_key(sc[t][r]) : 0u;
                    }
                __syncthreads();
                // the m-th largest sampled key of each query, one warp per query
                // (the histograms use the second chunk buffer, idle here)
                {
                    const int qq = warp;
                    const BlockQ &Q = s_q[qq];
                    if (qq >= ga && qq < gz && Q.ok && Q.n > kBCap) {
                        int m = (int)(((int64_t)kBSample * 2 * top_k + Q.n - 1) / Q.n);
                        if (m < 1) m = 1;
                        if (m <= kBSample) {
                            const uint32_t *kk = skey + qq * kBSample;
                            uint32_t *hist = reinterpret_cast<uint32_t *>(sm + C::off_buf + C::buf_bytes) + qq * 256;
                            uint32_t tau, need;
                            warp_radix_select([&](int i, uint32_t &key) { key = kk[i]; }, kBSample, (uint32_t)m, hist,
                                              s_wdig[qq], &tau, &need);
                            if (lane == 0) s_tau[qq] = tau;
                        }
                    }
                }
                __syncthreads();
            }
            // ---- stream the keys, keep candidates ----
            const int nchunks = (n_max + kBRows - 1) / kBRows;
            constexpr int NB = C::NB;
            auto load_chunk = [&](int c) {
                const int base = c * kBRows;
                load_rows<DI>(bufn(c % NB), kseq, [&](int r) -> int64_t { return base + r < n_max ? base + r : -1; },
                              kI);
            };
            // ring of NB chunk buffers: chunks c + 1 .. c + NB - 1 load while chunk c is scored
            for (int c = 0; c < NB - 1; c++) {
                if (c < nchunks) load_chunk(c);
                cp_async_commit();
            }
            for (int c = 0; c < nchunks; c++) {
                if (c + NB - 1 < nchunks) load_chunk(c + NB - 1);   // the buffer chunk c - 1 left
                cp_async_commit();
                cp_async_wait<NB - 1>();
                __syncthreads();
                float sc[2][4];
                warp_scores<DI>(bufn(c % NB), afr, sc);
#pragma unroll
                for (int t = 0; t < 2; t++)
#pragma unroll
                    for (int r = 0; r < 4; r++) {
                        const int qq = g + (r >> 1) * 8;
                        const int e = c * kBRows + warp * 16 + t * 8 + 2 * c4 + (r & 1);
                        if (qq < ga || qq >= gz || !s_q[qq].ok || e >= s_q[qq].n) continue;
                        const uint32_t key = score_key(sc[t][r]);
                        if (key >= s_tau[qq]) {
                            const uint32_t pos = atomicAdd(&s_cnt[qq], 1u);
                            if (pos < (uint32_t)kBCap) cand[qq * kBCap + pos] = ((uint64_t)key << 32) | (uint32_t)e;
                        }
                    }
                __syncthreads();
            }
            cp_async_wait<0>();
            __syncthreads();
            // ---- exact selection: one warp per query (the ring is free now) ----
            {
                const int qq = warp;
                int fall = 0;
                if (qq >= ga && qq < gz) {
                    const BlockQ Q = s_q[qq];
                    const int64_t qi = q0 + qq;
                    int32_t *idx_row = idx_out + qi * top_k;
                    float *sc_row = score_out ? score_out + qi * top_k : nullptr;
                    if (!Q.ok) {
                        if (lane == 0) set_error(err, CSA_ERR_DEVICE);
                        for (int i = lane; i < top_k; i += 32) {
                            idx_row[i] = -1;
                            if (sc_row) sc_row[i] = -INFINITY;
                        }
                    } else {
                        const uint32_t cnt = s_cnt[qq];
                        const uint32_t k_eff = (uint32_t)(Q.n < top_k ? Q.n : top_k);
                        if (k_eff == 0) {
                            for (int i = lane; i < top_k; i += 32) {
                                idx_row[i] = -1;
                                if (sc_row) sc_row[i] = -INFINITY;
                            }
                        } else if (cnt >= k_eff && cnt <= (uint32_t)kBCap) {
                            const uint64_t *qc = cand + qq * kBCap;
                            fall = warp_select_write<8>([&](int i) { return __ldcg(qc + i); }, (int)cnt, Q.n, top_k,
                                                     sm + C::off_buf + qq * C::warp_scratch, s_wdig[qq], idx_row,
                                                     sc_row) ? 0 : 1;   // 1: ties at the k-th key
                        } else {
                            fall = 2;   // the sample misjudged the row: every score again
                        }
                    }
                }
                if (lane == 0) s_fall[qq] = fall;
            }
            __syncthreads();
            // ---- the rare queries the warps left: the whole block, one query at a time ----
            // first the ties at the k-th key (they select among their own candidates),
            // then the rows the sample misjudged (they use the CTA's whole candidate
            // slot as scratch for their keys)
            for (int pass = 1; pass <= 2; pass++)
            for (int qq = ga; qq < gz; qq++) {
                const int fall = s_fall[qq];
                if (fall != pass) continue;
                const BlockQ Q = s_q[qq];
                const int64_t qi = q0 + qq;
                int32_t *idx_row = idx_out + qi * top_k;
                float *sc_row = score_out ? score_out + qi * top_k : nullptr;
                const uint32_t cnt = s_cnt[qq];
                if (fall == 1) {
                    constexpr int KPT = kBCap / kBT;
                    uint64_t cv[KPT];
#pragma unroll
                    for (int i = 0; i < KPT; i++) {
                        const uint32_t c = tid + i * kBT;
                        cv[i] = c < cnt ? __ldcg(cand + (int64_t)qq * kBCap + c) : ~0ull;
                    }
                    auto src = [&](int i, uint32_t &key, int32_t &ent) -> bool {
                        uint64_t v = 0;
#pragma unroll
                        for (int j = 0; j < KPT; j++)
                            if (j == i) v = cv[j];
                        key = (uint32_t)(v >> 32);
                        ent = (int32_t)(uint32_t)v;
                        return v != ~0ull;
                    };
                    select_write<KPT>(src, Q.n, top_k, sm + C::off_gt, sm + C::off_eq, sm + C::off_pre, s_hist, s_w, s_dig, idx_row, sc_row);
                } else {
                    // exact fallback: every key of this query, computed once (fp32) into the slot
                    uint32_t *fkeys = reinterpret_cast<uint32_t *>(cand);
                    const float *qv = qs + qq * DI;
                    const int n = Q.n;
                    for (int e = tid; e < n; e += kBT) {
                        const uint16_t *kr = kseq + (int64_t)e * DI;
                        float acc = 0.f;
                        for (int d = 0; d < DI; d += 2) {
                            const uint32_t w2 = __ldg(reinterpret_cast<const uint32_t *>(kr + d));
                            acc = fmaf(qv[d], bf16_lo(w2), acc);
                            acc = fmaf(qv[d + 1], bf16_hi(w2), acc);
                        }
                        fkeys[e] = score_key(acc);
                    }
                    __syncthreads();
                    auto src = [&](int i, uint32_t &key, int32_t &ent) -> bool {
                        const int e = i * kBT + tid;   // a warp's loads are consecutive words
                        ent = e;
                        if (e >= n) return false;
                        key = __ldcg(fkeys + e);
                        return true;
                    };
                    select_write<kBFallKeys>(src, n, top_k, sm + C::off_gt, sm + C::off_eq, sm + C::off_pre, s_hist, s_w, s_dig, idx_row, sc_row);
                }
            }
            ga = gz;
            __syncthreads();
        }
        __syncthreads();
    }
}

int g_sms_cache[64];

int device_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!g_sms_cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sms_cache[dev] = n;
    }
    return g_sms_cache[dev];
}

template <int DI>
cudaError_t launch_block_t(const IndexArgs &a, cudaStream_t st)
{
    using C = BCfg<DI>;
    const int64_t nblocks = (a.total_q + kBQ - 1) / kBQ;
    const int64_t sms = device_sms();
    // one candidate slot per CTA: as many persistent CTAs as the workspace holds
    int64_t grid = nblocks < sms ? nblocks : sms;
    const int64_t slots = (int64_t)(a.ws_bytes / kBSlotBytes);
    if (grid > slots) grid = slots;
    if (grid < 1) return cudaErrorInvalidValue;
    return launch_kernel("index_block", index_block_kernel<DI>, dim3((unsigned)grid), dim3(kBT), C::smem, st, false, a.batch,
                         a.cu_kv, a.cu_q, a.cu_csa, a.total_q, a.q_idx, a.k_idx, a.n_heads_idx, a.ratio, a.top_k,
                         reinterpret_cast<uint64_t *>(a.ws), a.idx_out, a.score_out, a.err);
}

}  // namespace

bool index_block_applicable(const IndexArgs &a)
{
    const int64_t max_n = a.max_kv_len / a.ratio;
    return a.total_q >= 1024 && max_n <= kBMaxN && a.top_k <= kBMaxK &&
           (a.d_idx == 32 || a.d_idx == 64 || a.d_idx == 128);
}

size_t index_block_ws_bytes(const IndexArgs &a)
{
    const int64_t nblocks = (a.total_q + kBQ - 1) / kBQ;
    const int64_t sms = device_sms();
    const int64_t grid = nblocks < sms ? nblocks : sms;
    return (size_t)grid * kBSlotBytes;
}

size_t index_block_min_ws_bytes() { return kBSlotBytes; }

cudaError_t launch_index_block(const IndexArgs &a, cudaStream_t st)
{
    if (a.total_q <= 0) return cudaSuccess;
    switch (a.d_idx) {
    case 32: return launch_block_t<32>(a, st);
    case 64: return launch_block_t<64>(a, st);
    case 128: return launch_block_t<128>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace csa
