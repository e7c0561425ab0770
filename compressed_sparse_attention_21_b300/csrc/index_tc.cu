// Lightning indexer + top-k for prefill-sized batches with d_I = 64, scores
// on the fifth-generation tensor cores ("DeepSeek-V4 core architecture",
// §2.2 CSA step 2: a light scorer rates each query against every compressed
// entry and only the top-k entries are kept).
//
// A persistent CTA takes 128 consecutive queries of the batch at a time (one
// pass per sequence present among them) and streams that sequence's indexer
// keys through shared memory once for all 128:
//
//  1. Scores.  The head-summed query (fp32) is split into three bf16 terms
//     (hi + mid + lo, exact to 2^-27 relative) that sit in shared memory as
//     the A operand, M = 128 queries x K = 64; each 256-key chunk (TMA, 128-
//     byte swizzled) is the B operand, N = 256.  Twelve tcgen05.mma (3 terms
//     x 4 k-steps of 16) accumulate S = sum_terms term . k in fp32 in tensor
//     memory: the fp32 score of the definition up to fp32 rounding order.
//     Two S buffers (2 x 256 columns) let the next chunk's products run while
//     the current one is read.
//  2. A threshold per query from 256 evenly spaced entries (scored in fp32 on
//     the CUDA cores): the sampled key expected to have about 2k entries above
//     it, found by a warp radix select.  Rows that fit the candidate buffer
//     keep every entry.
//  3. Twelve filter warps read the scores from tensor memory (a thread owns
//     one query row and a third of the chunk's columns) and append the keys
//     at or above the threshold, with their entry index, to the query's
//     candidate list in the workspace.
//  4. Exact selection among the candidates, one warp per query (the
//     selection shared with index_block.cu); ties at the k-th key and rows the
//     sample misjudged go to the block-wide exact selection.
// Warp roles while streaming: warp 0 lane 0 issues the TMA loads, warp 1
// lane 0 the MMAs (warp 1 owns the tensor memory), warps 4-15 filter.  Every
// wait is bounded: one that runs out reports CSA_ERR_TIMEOUT and the CTA stops.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "prefill_select.cuh"
#include "tc.cuh"
#include "tma.h"

namespace csa {

namespace {

constexpr int kTQ = 128;                  // queries per block (MMA M)
constexpr int kTR = 256;                  // keys per chunk (MMA N)
constexpr int kTDI = 64;                  // indexer key width handled here
constexpr int kTStages = 4;               // key chunks in flight
constexpr int kTFilterWarps = 12;         // warps 4 .. 15
constexpr uint32_t kTRowB = kTDI * 2;     // one key or query-term row: 128 bytes
constexpr uint32_t kTAB = kTQ * kTRowB;   // one query term: 16 KiB
constexpr uint32_t kTChunkB = kTR * kTRowB;   // one key chunk: 32 KiB
// dynamic shared memory (bytes from a 1024-aligned base)
constexpr uint32_t T_OFF_A = 0;                                   // 3 query terms (SW128, K-major)
constexpr uint32_t T_OFF_B = T_OFF_A + 3 * kTAB;                  // kTStages key chunks (SW128, K-major)
constexpr uint32_t T_OFF_QS = T_OFF_B + kTStages * kTChunkB;      // [128][64] fp32 head sums
constexpr uint32_t T_OFF_BAR = T_OFF_QS + kTQ * kTDI * 4;
constexpr uint32_t T_OFF_END = T_OFF_BAR + 16 * 8;
constexpr uint32_t kTSmem = T_OFF_END + 1024;                     // + alignment slack
// while sampling, the chunk stages hold the sampled rows (padded stride: no
// bank conflicts), the warps' histograms and half of the block's sampled keys
constexpr uint32_t kTSampStride = kTRowB + 16;
constexpr uint32_t T_SMP_ROWS = T_OFF_B;
constexpr uint32_t T_SMP_HIST = T_SMP_ROWS + kBSample * kTSampStride;
constexpr uint32_t T_SMP_KEYS = T_SMP_HIST + 16 * 256 * 4;
// after streaming, the chunk stages hold the selecting warps' scratch and,
// behind it, the bitmaps of the block-wide selection
constexpr uint32_t kTWarpScratch = 256 * 4 + kBWords * 4 + kBWords * 2;
constexpr uint32_t T_OFF_GT = T_OFF_B + 16 * kTWarpScratch;
constexpr uint32_t T_OFF_EQ = T_OFF_GT + kBWords * 4;
constexpr uint32_t T_OFF_PRE = T_OFF_EQ + kBWords * 4;
static_assert(T_OFF_PRE + kBWords * 4 <= T_OFF_B + kTStages * kTChunkB, "selection bitmaps fit the stages");
static_assert(T_SMP_KEYS + (kTQ / 2) * kBSample * 4 <= T_OFF_B + kTStages * kTChunkB, "sampling fits the stages");
static_assert(16 * kTWarpScratch <= kTStages * kTChunkB, "selection scratch fits the stages");
static_assert(kTSmem + 6 * 1024 <= 232448, "shared memory per CTA (dynamic + static)");
constexpr size_t kTSlotBytes = (size_t)kTQ * kBCap * 8;            // candidates of one persistent CTA
constexpr uint32_t kTTmemCols = 512;                               // two S buffers of 256 columns

// mbarriers
constexpr int TB_KFULL = 0, TB_KFREE = 4, TB_SFULL = 8, TB_SFREE = 10, TB_FIN = 12;

__global__ void __launch_bounds__(kBT, 1)
index_tc_kernel(const __grid_constant__ CUtensorMap map_k, int batch, const int64_t *__restrict__ cu_kv,
                const int64_t *__restrict__ cu_q, const int64_t *__restrict__ cu_csa, int64_t total_q,
                const uint16_t *__restrict__ qI, const uint16_t *__restrict__ kI, int HI, int ratio, int top_k,
                uint64_t *__restrict__ cand_ws, int32_t *__restrict__ idx_out, float *__restrict__ score_out,
                int *err)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ BlockQ s_q[kTQ];
    __shared__ uint32_t s_tau[kTQ], s_cnt[kTQ];
    __shared__ int s_fall[kTQ];
    __shared__ uint32_t s_wdig[16][2];
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_w[2 * (kBT / 32) + 1];
    __shared__ uint32_t s_dig[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_stop;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;            // swizzled operands need 1024-byte alignment
    uint8_t *sm = smem_raw + (sb - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *qs = reinterpret_cast<float *>(sm + T_OFF_QS);
    uint64_t *cand = cand_ws + (int64_t)blockIdx.x * kTQ * kBCap;
    auto bar = [&](int i) { return sb + T_OFF_BAR + 8u * (uint32_t)i; };

    if (tid == 0) {
        for (int s = 0; s < kTStages; s++) {
            mbar_init(bar(TB_KFULL + s), 1);
            mbar_init(bar(TB_KFREE + s), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(bar(TB_SFULL + b), 1);
            mbar_init(bar(TB_SFREE + b), kTFilterWarps * 32);
        }
        mbar_init(bar(TB_FIN), 1);
        fence_mbar_init();
        s_stop = 0;
    }
    if (warp == 1) tc::tmem_alloc(smem_u32(&s_tmem), kTTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;

    const int64_t nblocks = (total_q + kTQ - 1) / kTQ;
    uint32_t G = 0;   // key chunks streamed so far by this CTA (every thread counts them)
    bool stop = false;

    for (int64_t blk = blockIdx.x; blk < nblocks && !stop; blk += gridDim.x) {
        const int64_t q0 = blk * kTQ;
        const int nqb = (int)(total_q - q0 < kTQ ? total_q - q0 : kTQ);
        // ---- the block's queries ----
        for (int j = warp; j < kTQ; j += kBT / 32) {
            const int64_t qi = q0 + (j < nqb ? j : 0);
            const QueryPos p = query_pos(cu_kv, cu_q, cu_csa, batch, qi);
            if (lane == 0) {
                BlockQ r;
                r.b = p.b;
                r.n = (int)((p.t + 1) / ratio);
                r.e0 = p.e0;
                r.ok = j < nqb && p.ne == p.L / ratio && p.t >= 0 && p.t < p.L && r.n <= kBMaxN;
                s_q[j] = r;
            }
        }
        for (int i = tid; i < kTQ * kTDI; i += kBT) {
            const int qq = i / kTDI, d = i % kTDI;
            float acc = 0.f;
            if (qq < nqb)
                for (int h = 0; h < HI; h++) acc += bf16_lo(__ldg(qI + ((q0 + qq) * HI + h) * kTDI + d));
            qs[i] = acc;
        }
        __syncthreads();
        // the three bf16 terms of the head sums, 128-byte swizzled rows (16-byte chunk c of row r at c ^ (r & 7))
        for (int i = tid; i < kTQ * (kTDI / 2); i += kBT) {
            const int qq = i / (kTDI / 2), d = 2 * (i % (kTDI / 2));
            float x0 = qs[qq * kTDI + d], x1 = qs[qq * kTDI + d + 1];
            const uint32_t off = (uint32_t)qq * kTRowB + (((uint32_t)(d >> 3) ^ (uint32_t)(qq & 7)) << 4) + (d & 7) * 2;
#pragma unroll
            for (int term = 0; term < 3; term++) {
                const uint32_t pk = pack_bf16x2(x0, x1);
                *reinterpret_cast<uint32_t *>(sm + T_OFF_A + term * kTAB + off) = pk;
                x0 -= bf16_lo(pk);
                x1 -= bf16_hi(pk);
            }
        }
        tc::fence_proxy_async();
        __syncthreads();
        tc::fence_after_sync();

        // ---- one pass per sequence present in the block ----
        for (int ga = 0; ga < nqb && !stop;) {
            int gz = ga + 1;
            while (gz < nqb && s_q[gz].b == s_q[ga].b) gz++;
            int n_max = 0;
            bool need_sample = false;
            for (int i = ga; i < gz; i++)
                if (s_q[i].ok) {
                    n_max = s_q[i].n > n_max ? s_q[i].n : n_max;
                    need_sample |= s_q[i].n > kBCap;
                }
            const int64_t e0 = s_q[ga].e0;
            const uint16_t *kseq = kI + e0 * kTDI;
            if (tid < kTQ) {
                s_tau[tid] = 0u;
                s_cnt[tid] = 0u;
            }
            __syncthreads();
            if (need_sample) {
                // sampled rows j_s = s * n_max / 256 of the sequence, scored in fp32
                for (int i = tid; i < kBSample * 8; i += kBT) {
                    const int r = i >> 3, c = i & 7;
                    const int64_t j = (int64_t)r * n_max / kBSample;
                    *reinterpret_cast<uint4 *>(sm + T_SMP_ROWS + r * kTSampStride + c * 16) =
                        __ldg(reinterpret_cast<const uint4 *>(kseq + j * kTDI) + c);
                }
                __syncthreads();
                uint32_t *skeys = reinterpret_cast<uint32_t *>(sm + T_SMP_KEYS);
                for (int half = 0; half < 2; half++) {
                    // 8 threads per query; at each step they read 8 consecutive sampled rows
                    // (the padded stride puts them in distinct banks)
                    const int qq = 64 * half + (tid >> 3);
                    const bool qv_ok = qq >= ga && qq < gz && s_q[qq].ok;
                    const int nq = s_q[qq].n;
                    float qv[kTDI];
#pragma unroll
                    for (int d = 0; d < kTDI; d++) qv[d] = qs[qq * kTDI + d];
                    for (int i = 0; i < kBSample / 8; i++) {
                        const int s = 8 * i + (tid & 7);
                        const uint32_t *row = reinterpret_cast<const uint32_t *>(sm + T_SMP_ROWS + s * kTSampStride);
                        float acc = 0.f;
#pragma unroll
                        for (int d2 = 0; d2 < kTDI / 2; d2++) {
                            const uint32_t w2 = row[d2];
                            acc = fmaf(qv[2 * d2], bf16_lo(w2), acc);
                            acc = fmaf(qv[2 * d2 + 1], bf16_hi(w2), acc);
                        }
                        const int64_t j = (int64_t)s * n_max / kBSample;
                        skeys[(qq - 64 * half) * kBSample + s] = (qv_ok && j < nq) ? score_key(acc) : 0u;
                    }
                    __syncthreads();
                    // the threshold of each query: warp w takes queries 64 half + w + 16 i
                    uint32_t *whist = reinterpret_cast<uint32_t *>(sm + T_SMP_HIST) + warp * 256;
                    for (int i = 0; i < 4; i++) {
                        const int q = 64 * half + warp + 16 * i;
                        if (q < ga || q >= gz || !s_q[q].ok || s_q[q].n <= kBCap) continue;
                        int m = (int)(((int64_t)kBSample * 2 * top_k + s_q[q].n - 1) / s_q[q].n);
                        if (m < 1) m = 1;
                        if (m > kBSample) continue;
                        const uint32_t *kk = skeys + (q - 64 * half) * kBSample;
                        uint32_t tau, need;
                        warp_radix_select([&](int ii, uint32_t &key) { key = kk[ii]; }, kBSample, (uint32_t)m, whist,
                                          s_wdig[warp], &tau, &need);
                        if (lane == 0) s_tau[q] = tau;
                    }
                    __syncthreads();
                }
                tc::fence_proxy_async();   // the stages' generic writes before the key chunks' bulk loads
                __syncthreads();
            }

            // ---- stream the keys: TMA producer, MMA issuer, filters ----
            const int nch = (n_max + kTR - 1) / kTR;
            bool fail = false;
            if (warp == 0) {
                if (lane == 0) {
                    const uint64_t once = tc::policy_evict_first();
                    for (int c = 0; c < nch && !fail; c++) {
                        const uint32_t g = G + (uint32_t)c;
                        const int s = (int)(g % kTStages);
                        if (g >= kTStages && !mbar_wait(bar(TB_KFREE + s), ((g - kTStages) / kTStages) & 1u)) {
                            fail = true;
                            break;
                        }
                        mbar_expect_tx(bar(TB_KFULL + s), kTChunkB);
                        tc::tma_tile2d(sb + T_OFF_B + s * kTChunkB, &map_k, 0, (int)(e0 + (int64_t)c * kTR),
                                       bar(TB_KFULL + s), once);
                    }
                }
                __syncwarp();
            } else if (warp == 1) {
                if (lane == 0) {
                    constexpr uint32_t idesc = tc::idesc_bf16_f32(kTQ, kTR, false, false);
                    const uint64_t a0 = tc::sdesc_sw128(sb + T_OFF_A, 16, 1024);
                    const uint64_t b0 = tc::sdesc_sw128(sb + T_OFF_B, 16, 1024);
                    for (int c = 0; c < nch && !fail; c++) {
                        const uint32_t g = G + (uint32_t)c;
                        const int s = (int)(g % kTStages), b = (int)(g & 1u);
                        if (!mbar_wait(bar(TB_KFULL + s), (g / kTStages) & 1u) ||
                            (g >= 2 && !mbar_wait(bar(TB_SFREE + b), ((g - 2) >> 1) & 1u))) {
                            fail = true;
                            break;
                        }
                        tc::fence_after_sync();
#pragma unroll
                        for (int term = 0; term < 3; term++)
#pragma unroll
                            for (int ks = 0; ks < kTDI / 16; ks++)
                                // descriptors advance by adding (byte offset >> 4) to the address field
                                tc::mma_ss(tmem + 256u * (uint32_t)b, a0 + (uint64_t)((term * kTAB + ks * 32) >> 4),
                                           b0 + (uint64_t)((s * kTChunkB + ks * 32) >> 4), idesc, (term | ks) != 0);
                        tc::mma_commit(bar(TB_KFREE + s));
                        tc::mma_commit(bar(TB_SFULL + b));
                    }
                }
                __syncwarp();
            } else if (warp >= 4) {
                // filter: thread (quarter qr, lane) owns query 32 qr + lane and a third of each chunk's columns
                const int qr = warp & 3, part = (warp - 4) >> 2;
                const int q = 32 * qr + lane;
                const int g0 = 3 * part, g1 = g0 + 3 < 8 ? g0 + 3 : 8;
                const bool q_ok = q >= ga && q < gz && s_q[q].ok;
                const int nq = s_q[q].n;
                const uint32_t tau = s_tau[q];
                uint64_t *qcand = cand + (int64_t)q * kBCap;
                const uint32_t lane_base = (uint32_t)(qr * 32) << 16;
                for (int c = 0; c < nch; c++) {
                    const uint32_t g = G + (uint32_t)c;
                    const int b = (int)(g & 1u);
                    // the warp leaves together (the tensor-memory loads below are warp-wide)
                    if (__any_sync(0xffffffffu, !mbar_wait(bar(TB_SFULL + b), (g >> 1) & 1u))) {
                        fail = true;
                        break;
                    }
                    tc::fence_after_sync();
                    // one 32-column group at a time; the S buffer is released after the last read
                    for (int gi = g0; gi < g1; gi++) {
                        float v[32];
                        tc::tmem_ld32(tmem + lane_base + 256u * (uint32_t)b + 32u * (uint32_t)gi, v);
                        tc::tmem_wait_ld();
                        if (gi == g1 - 1) {
                            tc::fence_before_sync();
                            mbar_arrive(bar(TB_SFREE + b));
                        }
                        if (q_ok) {
                            const int ebase = c * kTR + 32 * gi;
#pragma unroll
                            for (int j = 0; j < 32; j++) {
                                const uint32_t key = score_key(v[j]);
                                if (ebase + j < nq && key >= tau) {
                                    const uint32_t pos = atomicAdd(&s_cnt[q], 1u);
                                    if (pos < (uint32_t)kBCap)
                                        qcand[pos] = ((uint64_t)key << 32) | (uint32_t)(ebase + j);
                                }
                            }
                        }
                    }
                }
            }
            G += (uint32_t)nch;
            if (fail) s_stop = 1;
            __syncthreads();   // candidates complete; the stages and S buffers are idle
            if (s_stop) {
                if (tid == 0) set_error(err, CSA_ERR_TIMEOUT);
                stop = true;
                break;
            }

            // ---- exact selection: one warp per query (the stages are free now) ----
            for (int qq = ga + warp; qq < gz; qq += kBT / 32) {
                const BlockQ Q = s_q[qq];
                const int64_t qi = q0 + qq;
                int32_t *idx_row = idx_out + qi * top_k;
                float *sc_row = score_out ? score_out + qi * top_k : nullptr;
                int fall = 0;
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
                        fall = warp_select_write(cand + (int64_t)qq * kBCap, (int)cnt, Q.n, top_k,
                                                 sm + T_OFF_B + warp * kTWarpScratch, s_wdig[warp], idx_row, sc_row)
                                   ? 0
                                   : 1;   // 1: ties at the k-th key
                    } else {
                        fall = 2;         // the sample misjudged the row: every score again
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
                    select_write<KPT>(src, Q.n, top_k, sm + T_OFF_GT, sm + T_OFF_EQ, sm + T_OFF_PRE, s_hist, s_w, s_dig, idx_row, sc_row);
                } else {
                    // exact fallback: every key of this query, computed once (fp32) into the slot
                    uint32_t *fkeys = reinterpret_cast<uint32_t *>(cand);
                    const float *qv = qs + qq * kTDI;
                    const int n = Q.n;
                    for (int e = tid; e < n; e += kBT) {
                        const uint16_t *kr = kseq + (int64_t)e * kTDI;
                        float acc = 0.f;
                        for (int d = 0; d < kTDI; d += 2) {
                            const uint32_t w2 = __ldg(reinterpret_cast<const uint32_t *>(kr + d));
                            acc = fmaf(qv[d], bf16_lo(w2), acc);
                            acc = fmaf(qv[d + 1], bf16_hi(w2), acc);
                        }
                        fkeys[e] = score_key(acc);
                    }
                    __syncthreads();
                    auto src = [&](int i, uint32_t &key, int32_t &ent) -> bool {
                        const int e = tid * kBFallKeys + i;
                        ent = e;
                        if (e >= n) return false;
                        key = __ldcg(fkeys + e);
                        return true;
                    };
                    select_write<kBFallKeys>(src, n, top_k, sm + T_OFF_GT, sm + T_OFF_EQ, sm + T_OFF_PRE, s_hist, s_w, s_dig, idx_row, sc_row);
                }
            }
            tc::fence_proxy_async();   // the selection scratch (generic writes) before later bulk loads
            __syncthreads();
            ga = gz;
        }
    }
    // every product is complete before the tensor memory is released
    if (warp == 1) {
        if (lane == 0) {
            tc::mma_commit(bar(TB_FIN));
            if (!mbar_wait(bar(TB_FIN), 0)) set_error(err, CSA_ERR_TIMEOUT);
        }
        __syncwarp();
    }
    // no key chunk may still be landing when the CTA ends
    if (warp == 0 && lane == 0 && stop) {
        for (uint32_t g = G >= kTStages ? G - kTStages : 0; g < G; g++)
            mbar_wait(bar(TB_KFULL + (int)(g % kTStages)), (g / kTStages) & 1u);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, kTTmemCols);
}

int g_tc_sms[64];

int tc_device_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!g_tc_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_tc_sms[dev] = n;
    }
    return g_tc_sms[dev];
}

}  // namespace

bool index_tc_applicable(const IndexArgs &a)
{
    const int64_t max_n = a.max_kv_len / a.ratio;
    return !a.fp8 && a.d_idx == kTDI && a.total_q >= 1024 && max_n <= kBMaxN && a.top_k <= kBMaxK &&
           a.total_csa + kTR < 0x7fffffffLL && tma_available();
}

size_t index_tc_ws_bytes(const IndexArgs &a)
{
    const int64_t nblocks = (a.total_q + kTQ - 1) / kTQ;
    const int64_t sms = tc_device_sms();
    const int64_t grid = nblocks < sms ? nblocks : sms;
    return (size_t)grid * kTSlotBytes;
}

size_t index_tc_min_ws_bytes() { return kTSlotBytes; }

cudaError_t launch_index_tc(const IndexArgs &a, cudaStream_t st)
{
    if (a.total_q <= 0) return cudaSuccess;
    const int64_t nblocks = (a.total_q + kTQ - 1) / kTQ;
    int64_t grid = nblocks < tc_device_sms() ? nblocks : tc_device_sms();
    const int64_t slots = (int64_t)(a.ws_bytes / kTSlotBytes);   // one candidate slot per persistent CTA
    if (grid > slots) grid = slots;
    if (grid < 1) return cudaErrorInvalidValue;
    CUtensorMap m_k;
    // with no entries at all the map still needs a valid base: no chunk is loaded then
    const void *kbase = a.total_csa > 0 ? (const void *)a.k_idx : (const void *)a.q_idx;
    const int64_t krows = a.total_csa > 0 ? a.total_csa : 1;
    cudaError_t e = tma_map_bf16(&m_k, kbase, krows, kTDI, kTDI, kTR);
    if (e != cudaSuccess) return e;
    return launch_kernel("index_tc", index_tc_kernel, dim3((unsigned)grid), dim3(kBT), kTSmem, st, false, m_k,
                         a.batch, a.cu_kv, a.cu_q, a.cu_csa, a.total_q, a.q_idx, a.k_idx, a.n_heads_idx, a.ratio,
                         a.top_k, reinterpret_cast<uint64_t *>(a.ws), a.idx_out, a.score_out, a.err);
}

}  // namespace csa
