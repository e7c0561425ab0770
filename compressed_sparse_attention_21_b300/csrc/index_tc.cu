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
//     at or above the threshold, with their entry index, to their own
//     sub-list of the query's candidates in the workspace: no shared counter,
//     and each sub-list stays in entry order.
//  4. Exact selection among the candidates by four groups of four warps, one
//     query per group at a time: the query's sub-lists come into shared
//     memory by bulk copies, radix levels find the k-th key, and a bitmap of
//     the taken entries gives the selection in index order.  Ties at the
//     k-th key and rows the sample misjudged go to the block-wide exact
//     selection.
// Blocks are taken longest rows first, dealt to the CTAs in a snake order.
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
constexpr uint32_t T_OFF_END = T_OFF_BAR + 24 * 8;
constexpr uint32_t kTSmem = T_OFF_END + 1024;                     // + alignment slack
// while sampling, the chunk stages hold the sampled rows (padded stride: no
// bank conflicts), the warps' histograms and half of the block's sampled keys
constexpr uint32_t kTSampStride = kTRowB + 16;
constexpr uint32_t T_SMP_ROWS = T_OFF_B;
constexpr uint32_t T_SMP_HIST = T_SMP_ROWS + kBSample * kTSampStride;
constexpr uint32_t T_SMP_KEYS = T_SMP_HIST + 16 * 256 * 4;
// after streaming, the query tiles' and stages' space holds four selection
// groups (a query's candidate slot, copied in, and its scratch) and, behind
// them, the bitmaps of the block-wide selection
constexpr int kSelGroups = 4;                                  // four warps each
constexpr uint32_t kSelHist = kBCap * 8;                       // after the candidate slot
constexpr uint32_t kSelTaken = kSelHist + 3 * 256 * 4;   // three histograms in turn
constexpr uint32_t kSelPre = kSelHist;                    // u16 word prefixes (with scores), after the levels
constexpr uint32_t kSelMisc = kSelTaken + kBWords * 4;    // the warps' counts
constexpr uint32_t kSelBytes = kSelMisc + 256;
constexpr uint32_t T_OFF_SEL = T_OFF_A;
constexpr uint32_t T_OFF_GT = T_OFF_SEL + kSelGroups * kSelBytes;
constexpr uint32_t T_OFF_EQ = T_OFF_GT + kBWords * 4;
constexpr uint32_t T_OFF_PRE = T_OFF_EQ + kBWords * 4;
static_assert(T_OFF_PRE + kBWords * 4 <= T_OFF_QS, "selection groups and bitmaps fit below the head sums");
static_assert(kBWords * 2 <= 3 * 256 * 4 && kSelBytes % 16 == 0, "word prefixes fit the histograms; copies stay aligned");
static_assert(T_SMP_KEYS + (kTQ / 2) * kBSample * 4 <= T_OFF_B + kTStages * kTChunkB, "sampling fits the stages");
static_assert(T_OFF_A + kBMaxN * 4 <= T_OFF_GT, "the exact fallback's keys fit below the selection bitmaps");
static_assert(kTSmem + 9 * 1024 <= 232448, "shared memory per CTA (dynamic + static, about 8.3 KiB)");
constexpr size_t kTSlotBytes = (size_t)kTQ * kBCap * 8;            // candidates of one persistent CTA
constexpr size_t kTHeader = 256;                                   // the block counter, ahead of the slots
// A query's candidate slot (kBCap pairs) holds one sub-list per column part of
// the filter, sized by the part's share of a chunk's columns (96, 96, 64 of
// 256): a row of n <= kBCap entries never overflows it.
__host__ __device__ constexpr uint32_t sub_cap(int part) { return part < 2 ? 3u * kBCap / 8u : 2u * kBCap / 8u; }
__host__ __device__ constexpr uint32_t sub_off(int part) { return part == 0 ? 0u : part == 1 ? 3u * kBCap / 8u : 6u * kBCap / 8u; }
static_assert(sub_off(2) + sub_cap(2) == (uint32_t)kBCap, "the sub-lists fill the slot");
constexpr uint32_t kTTmemCols = 512;                               // two S buffers of 256 columns

// mbarriers
constexpr int TB_KFULL = 0, TB_KFREE = 4, TB_SFULL = 8, TB_SFREE = 10, TB_FIN = 12, TB_SEL = 13;

// One query's top-k by a group of four warps (128 threads, named barrier
// `bid`) from its candidates in shared memory: `cand` holds the three
// sub-lists at their slot offsets with c0, c1, c2 pairs (key << 32 | entry);
// every key lies in [lo, hi].  The exact k-th key by 8-bit radix levels
// (starting at the byte of the highest bit where lo and hi differ; three
// histograms in turn, so one barrier per level), a bitmap of the taken
// entries, and the selection written in index order.  Returns false, writing
// nothing, when keys equal to the k-th key would have to be split.  Every
// thread of the group calls it; the caller separates two calls by a barrier.
__device__ bool group_select_write(const uint64_t *cand, uint32_t c0, uint32_t c1, uint32_t c2, int n, int top_k,
                                   uint32_t lo, uint32_t hi, uint8_t *gbuf, int bid, int32_t *idx_row, float *sc_row)
{
    const int gt = threadIdx.x & 127, lane = threadIdx.x & 31, gw = gt >> 5;
    uint32_t *hist = reinterpret_cast<uint32_t *>(gbuf + kSelHist);   // 3 x 256 bins
    uint32_t *taken = reinterpret_cast<uint32_t *>(gbuf + kSelTaken);
    uint16_t *pre = reinterpret_cast<uint16_t *>(gbuf + kSelPre);
    uint32_t *wsum = reinterpret_cast<uint32_t *>(gbuf + kSelMisc);
    const uint32_t cnt = c0 + c1 + c2;
    auto pair_at = [&](uint32_t u) -> uint64_t {
        const uint32_t j = u < c0 ? u : u < c0 + c1 ? u - c0 + sub_off(1) : u - c0 - c1 + sub_off(2);
        return cand[j];
    };
    const uint32_t k_eff = (uint32_t)(n < top_k ? n : top_k);
    const int words = (n + 31) >> 5;   // at most 1024: eight per thread
    for (int w = gt; w < words; w += 128) taken[w] = 0;
#pragma unroll
    for (int h = 0; h < 2; h++) {
        hist[h * 256 + gt] = 0;
        hist[h * 256 + 128 + gt] = 0;
    }
    // the bits above the highest one where lo and hi differ are common to every key; each
    // level resolves the next (up to) 8 bits below them, so the first level's bins spread
    const uint32_t diff = lo ^ hi;
    const int topbit = diff ? 31 - __clz(diff) : 0;
    const uint32_t low = (2u << topbit) - 1u;   // bits 0 .. topbit (all for topbit = 31)
    uint32_t prefix = lo & ~low, pmask = ~low, remaining = k_eff;
    bool whole = false;
    // this thread's keys (candidates gt, gt + 128, ...) stay in registers for every
    // level; the loops over them stop at the thread's count
    constexpr int KPT = kBCap / 128;
    const int nmine = cnt > (uint32_t)gt ? (int)((cnt - 1 - gt) / 128 + 1) : 0;
    uint32_t kk[KPT];
#pragma unroll
    for (int u = 0; u < KPT; u++) kk[u] = u < nmine ? (uint32_t)(pair_at(gt + 128u * u) >> 32) : 0u;
    tc::named_bar(bid, 128);
    int lvl = 0;
#pragma unroll 1
    for (int hb = topbit; hb >= 0 && !whole; lvl++) {
        const int width = hb >= 7 ? 8 : hb + 1;
        const int sh = hb - width + 1;
        const uint32_t dmask = (1u << width) - 1u;
        hb = sh - 1;
        uint32_t *h = hist + 256 * (lvl % 3);
#pragma unroll
        for (int u = 0; u < KPT; u++) {
            if (u >= nmine) break;
            if ((kk[u] & pmask) == prefix) atomicAdd(&h[(kk[u] >> sh) & dmask], 1u);
        }
        tc::named_bar(bid, 128);
        // the histogram two levels on was last read before this barrier
        uint32_t *hz = hist + 256 * ((lvl + 2) % 3);
        hz[gt] = 0;
        hz[gt + 128] = 0;
        // every warp finds the digit itself
        uint32_t d = 0, above = 0;
        {
            uint32_t c[8], sum = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                c[i] = h[255 - 8 * lane - i];
                sum += c[i];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const uint32_t excl = incl - sum;
            uint32_t dl = 0, al = 0;
            const bool mine = excl < remaining && remaining <= incl;
            if (mine) {
                uint32_t acc = excl;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    if (acc + c[i] >= remaining) {
                        dl = 255 - 8 * lane - i;
                        al = acc;
                        break;
                    }
                    acc += c[i];
                }
            }
            const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
            d = __shfl_sync(0xffffffffu, dl, src);
            above = __shfl_sync(0xffffffffu, al, src);
        }
        remaining -= above;
        prefix |= d << sh;
        pmask |= dmask << sh;
        whole = h[d] == remaining;
    }
    if (!whole) return false;
    const uint32_t kstar = prefix;
#pragma unroll
    for (int u = 0; u < KPT; u++) {
        if (u >= nmine) break;
        if (kk[u] >= kstar) {
            const uint32_t e = (uint32_t)pair_at(gt + 128u * u);
            atomicOr(&taken[e >> 5], 1u << (e & 31));
        }
    }
    tc::named_bar(bid, 128);
    // thread gt takes words 8 gt .. 8 gt + 7; a group scan of their counts
    const int w0 = 8 * gt;
    uint32_t bits[8], mine = 0;
#pragma unroll
    for (int r = 0; r < 8; r++) {
        bits[r] = w0 + r < words ? taken[w0 + r] : 0u;
        mine += (uint32_t)__popc(bits[r]);
    }
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[gw] = incl;
    tc::named_bar(bid, 128);
    uint32_t run = incl - mine;
    for (int x = 0; x < gw; x++) run += wsum[x];
    if (!sc_row) {
        // the selection is staged in shared memory (the candidates are no longer needed)
        // and written out with consecutive threads on consecutive places
        int32_t *stage = reinterpret_cast<int32_t *>(const_cast<uint64_t *>(cand));
#pragma unroll
        for (int r = 0; r < 8; r++) {
            uint32_t b = bits[r];
            while (b) {
                const int j = __ffs(b) - 1;
                b &= b - 1u;
                if (run < (uint32_t)top_k) stage[run] = ((w0 + r) << 5) + j;
                run++;
            }
        }
        tc::named_bar(bid, 128);
        for (int i = gt; i < top_k; i += 128) idx_row[i] = i < (int)k_eff ? stage[i] : -1;
        return true;
    } else {
#pragma unroll
        for (int r = 0; r < 8; r++)
            if (w0 + r < words) {
                pre[w0 + r] = (uint16_t)run;
                run += (uint32_t)__popc(bits[r]);
            }
        tc::named_bar(bid, 128);
        for (uint32_t i = gt; i < cnt; i += 128) {
            const uint64_t c = pair_at(i);
            const uint32_t key = (uint32_t)(c >> 32), e = (uint32_t)c;
            if (key >= kstar) {
                const uint32_t pos = pre[e >> 5] + (uint32_t)__popc(taken[e >> 5] & ((1u << (e & 31)) - 1u));
                if (pos < (uint32_t)top_k) {
                    idx_row[pos] = (int32_t)e;
                    sc_row[pos] = key_score(key);
                }
            }
        }
    }
    for (int i = (int)k_eff + gt; i < top_k; i += 128) {
        idx_row[i] = -1;
        if (sc_row) sc_row[i] = -INFINITY;
    }
    return true;
}

__global__ void __launch_bounds__(kBT, 1)
index_tc_kernel(const __grid_constant__ CUtensorMap map_k, int batch, const int64_t *__restrict__ cu_kv,
                const int64_t *__restrict__ cu_q, const int64_t *__restrict__ cu_csa, int64_t total_q,
                const uint16_t *__restrict__ qI, const uint16_t *__restrict__ kI, int HI, int ratio, int top_k,
                unsigned *__restrict__ next_block, uint64_t *__restrict__ cand_ws, int32_t *__restrict__ idx_out,
                float *__restrict__ score_out, int *err)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ BlockQ s_q[kTQ];
    __shared__ uint32_t s_tau[kTQ], s_cnt[3][kTQ], s_kmax[3][kTQ];   // per column part
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
        for (int g = 0; g < kSelGroups; g++) mbar_init(bar(TB_SEL + g), 1);
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
    uint32_t sel_phase = 0;   // parity of the next candidate copy of this thread's selection group
    bool sel_late = false;    // a candidate copy outlasted its wait (its group's thread 0 only)

    // Blocks in decreasing order of position (a block's rows, and with them its
    // work, grow with its queries' positions), each CTA taking the next one
    // from a counter as it finishes the last: the long rows go first and the
    // short ones fill in behind them.
    __shared__ int64_t s_next;
    for (int r = 0; !stop; r++) {
        if (tid == 0) s_next = (int64_t)atomicAdd(next_block, 1u);
        __syncthreads();
        const int64_t jj = s_next;
        if (jj >= nblocks) break;
        const int64_t blk = nblocks - 1 - jj;
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
        // the three bf16 terms of the head sums, 128-byte swizzled rows (16-byte chunk c of row r at c ^ (r & 7));
        // built again for each further sequence of the block (the selection uses their space)
        auto build_terms = [&]() {
            for (int i = tid; i < kTQ * (kTDI / 2); i += kBT) {
                const int qq = i / (kTDI / 2), d = 2 * (i % (kTDI / 2));
                float x0 = qs[qq * kTDI + d], x1 = qs[qq * kTDI + d + 1];
                const uint32_t off =
                    (uint32_t)qq * kTRowB + (((uint32_t)(d >> 3) ^ (uint32_t)(qq & 7)) << 4) + (d & 7) * 2;
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
        };
        build_terms();

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
            if (tid < kTQ) s_tau[tid] = 0u;
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
                // filter: thread (quarter qr, lane) owns query 32 qr + lane and a third of each
                // chunk's columns, and appends the keys it passes to its own sub-list of the
                // query's candidates (in entry order; no shared counter)
                const int qr = warp & 3, part = (warp - 4) >> 2;
                const int q = 32 * qr + lane;
                const int g0 = 3 * part, g1 = g0 + 3 < 8 ? g0 + 3 : 8;
                const bool q_ok = q >= ga && q < gz && s_q[q].ok;
                const int nq = s_q[q].n;
                const uint32_t tau = s_tau[q];
                // a threshold at or above +0 compares like the raw fp32 bits as signed integers
                const bool tfast = tau >= 0x80000000u;
                const int tb = (int)(tau & 0x7fffffffu);
                const uint32_t cap = sub_cap(part);
                uint64_t *qsub = cand + (int64_t)q * kBCap + sub_off(part);
                uint32_t cntp = 0, kmx = 0;
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
                        // (no early exit here: every lane takes part in the next group's warp-wide load)
                        if (q_ok) {
                            const int ebase = c * kTR + 32 * gi;
                            const int lim = nq - ebase;   // visible entries of the group
                            const uint32_t rm = lim >= 32 ? 0xffffffffu : lim <= 0 ? 0u : (1u << lim) - 1u;
                            uint32_t keys[32], pass = 0, kb = 0;
                            if (tfast) {
                                int mx = (int)0x80000000;
#pragma unroll
                                for (int j = 0; j < 32; j++) {
                                    const int bits = __float_as_int(v[j]);
                                    pass |= (uint32_t)(bits >= tb) << j;
                                    mx = max(mx, bits);
                                    keys[j] = (uint32_t)bits | 0x80000000u;   // the key where it passes
                                }
                                kb = (uint32_t)mx | 0x80000000u;   // bounds every passing key
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; j++) {
                                    keys[j] = score_key(v[j]);
                                    pass |= (uint32_t)(keys[j] >= tau) << j;
                                    kb = max(kb, keys[j]);
                                }
                            }
                            pass &= rm;
                            if (pass) {
                                const uint32_t np = (uint32_t)__popc(pass);
                                if (cntp + np <= cap) {
                                    uint64_t *dst = qsub + cntp;
#pragma unroll
                                    for (int j = 0; j < 32; j++)
                                        if (pass & (1u << j))
                                            *dst++ = ((uint64_t)keys[j] << 32) | (uint32_t)(ebase + j);
                                }
                                cntp += np;   // past the capacity: the row overflowed (exact fallback)
                                kmx = max(kmx, kb);
                            }
                        }
                    }
                }
                s_cnt[part][q] = cntp;
                s_kmax[part][q] = kmx;
            }
            G += (uint32_t)nch;
            if (fail) s_stop = 1;
            __syncthreads();   // candidates complete; the stages and S buffers are idle
            if (s_stop) {
                if (tid == 0) set_error(err, CSA_ERR_TIMEOUT);
                stop = true;
                break;
            }

            // ---- exact selection: four groups of four warps, one query per group at a time;
            // a query's sub-lists come into the group's buffer by bulk copies ----
            {
                const int grp = warp >> 2, gt = tid & 127, bid = 1 + grp;
                uint8_t *gbuf = sm + T_OFF_SEL + grp * kSelBytes;
                const uint32_t gbar = bar(TB_SEL + grp);
                for (int qq = ga + grp; qq < gz; qq += kSelGroups) {
                    const BlockQ Q = s_q[qq];
                    const int64_t qi = q0 + qq;
                    int32_t *idx_row = idx_out + qi * top_k;
                    float *sc_row = score_out ? score_out + qi * top_k : nullptr;
                    int fall = 0;
                    const uint32_t k_eff = (uint32_t)(Q.n < top_k ? Q.n : top_k);
                    const uint32_t c0 = s_cnt[0][qq], c1 = s_cnt[1][qq], c2 = s_cnt[2][qq];
                    const bool over = c0 > sub_cap(0) || c1 > sub_cap(1) || c2 > sub_cap(2);
                    if (!Q.ok || k_eff == 0) {
                        if (!Q.ok && gt == 0) set_error(err, CSA_ERR_DEVICE);
                        for (int i = gt; i < top_k; i += 128) {
                            idx_row[i] = -1;
                            if (sc_row) sc_row[i] = -INFINITY;
                        }
                    } else if (over || c0 + c1 + c2 < k_eff) {
                        fall = 2;   // the sample misjudged the row: every score again
                    } else {
                        const uint64_t *slot = cand + (int64_t)qq * kBCap;
                        if (gt == 0) {
                            const uint32_t cp[3] = {c0, c1, c2};
                            uint32_t bytes = 0;
#pragma unroll
                            for (int p = 0; p < 3; p++) bytes += (8u * cp[p] + 15u) & ~15u;
                            mbar_expect_tx(gbar, bytes);
#pragma unroll
                            for (int p = 0; p < 3; p++)
                                if (cp[p])
                                    bulk_g2s(smem_u32(gbuf) + 8u * sub_off(p), slot + sub_off(p), (8u * cp[p] + 15u) & ~15u,
                                             gbar);
                        }
                        const bool late = tc::named_bar_or(bid, 128, !mbar_wait(gbar, sel_phase));
                        sel_phase ^= 1u;
                        if (late) {
                            // the copy may still land: wait for it once more at the end
                            if (gt == 0) {
                                set_error(err, CSA_ERR_TIMEOUT);
                                sel_late = true;
                            }
                            s_stop = 1;
                            break;
                        }
                        // every candidate key lies in [threshold, largest appended key]
                        const uint32_t kmx = max(max(s_kmax[0][qq], s_kmax[1][qq]), s_kmax[2][qq]);
                        fall = group_select_write(reinterpret_cast<const uint64_t *>(gbuf), c0, c1, c2, Q.n, top_k,
                                                  s_tau[qq], kmx, gbuf, bid, idx_row, sc_row)
                                   ? 0
                                   : 1;   // 1: ties at the k-th key
                        // the next copy rewrites the buffer: these reads come first
                        tc::fence_proxy_async();
                        tc::named_bar(bid, 128);
                    }
                    if (gt == 0) s_fall[qq] = fall;
                }
            }
            __syncthreads();
            if (s_stop) {
                stop = true;
                break;
            }
            // ---- the rare queries the warps left: the whole block, one query at a time ----
            // first the ties at the k-th key (they select among their own candidates),
            // then the rows the sample misjudged (they recompute every key)
            for (int pass = 1; pass <= 2; pass++)
            for (int qq = ga; qq < gz; qq++) {
                const int fall = s_fall[qq];
                if (fall != pass) continue;
                const BlockQ Q = s_q[qq];
                const int64_t qi = q0 + qq;
                int32_t *idx_row = idx_out + qi * top_k;
                float *sc_row = score_out ? score_out + qi * top_k : nullptr;
                if (fall == 1) {
                    // every sub-list is within its capacity here; unused places read as none
                    constexpr int KPT = kBCap / kBT;
                    uint64_t cv[KPT];
#pragma unroll
                    for (int i = 0; i < KPT; i++) {
                        const uint32_t c = tid + i * kBT;   // place in the slot
                        const int part = c < sub_off(1) ? 0 : c < sub_off(2) ? 1 : 2;
                        const uint32_t used = s_cnt[part][qq];
                        cv[i] = c - sub_off(part) < used ? __ldcg(cand + (int64_t)qq * kBCap + c) : ~0ull;
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
                    // exact fallback: every key of this query, computed once (fp32) into shared
                    // memory (the query terms and the stages' first 80 KiB: 128 KiB for
                    // 32768 keys); thread t owns keys t, t + 512, ...
                    uint32_t *fkeys = reinterpret_cast<uint32_t *>(sm + T_OFF_A);
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
                        const int e = i * kBT + tid;
                        ent = e;
                        if (e >= n) return false;
                        key = fkeys[e];
                        return true;
                    };
                    select_write<kBFallKeys>(src, n, top_k, sm + T_OFF_GT, sm + T_OFF_EQ, sm + T_OFF_PRE, s_hist, s_w, s_dig, idx_row, sc_row);
                }
            }
            tc::fence_proxy_async();   // the selection scratch (generic writes) before later bulk loads
            __syncthreads();
            if (gz < nqb) build_terms();   // the selection used the terms' space; another sequence streams next
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
    // no candidate copy or key chunk may still be landing when the CTA ends
    if (sel_late) mbar_wait(bar(TB_SEL + (warp >> 2)), sel_phase ^ 1u);
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
    return kTHeader + (size_t)grid * kTSlotBytes;
}

size_t index_tc_min_ws_bytes() { return kTHeader + kTSlotBytes; }

cudaError_t launch_index_tc(const IndexArgs &a, cudaStream_t st)
{
    if (a.total_q <= 0) return cudaSuccess;
    const int64_t nblocks = (a.total_q + kTQ - 1) / kTQ;
    int64_t grid = nblocks < tc_device_sms() ? nblocks : tc_device_sms();
    const int64_t slots = a.ws_bytes > kTHeader ? (int64_t)((a.ws_bytes - kTHeader) / kTSlotBytes) : 0;   // one per CTA
    if (grid > slots) grid = slots;
    if (grid < 1) return cudaErrorInvalidValue;
    CUtensorMap m_k;
    // with no entries at all the map still needs a valid base: no chunk is loaded then
    const void *kbase = a.total_csa > 0 ? (const void *)a.k_idx : (const void *)a.q_idx;
    const int64_t krows = a.total_csa > 0 ? a.total_csa : 1;
    cudaError_t e = tma_map_bf16(&m_k, kbase, krows, kTDI, kTDI, kTR);
    if (e != cudaSuccess) return e;
    // the block counter starts at zero on every call, whatever an earlier call left
    uint8_t *ws = reinterpret_cast<uint8_t *>(a.ws);
    e = cudaMemsetAsync(ws, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    return launch_kernel("index_tc", index_tc_kernel, dim3((unsigned)grid), dim3(kBT), kTSmem, st, false, m_k,
                         a.batch, a.cu_kv, a.cu_q, a.cu_csa, a.total_q, a.q_idx, a.k_idx, a.n_heads_idx, a.ratio,
                         a.top_k, reinterpret_cast<unsigned *>(ws), reinterpret_cast<uint64_t *>(ws + kTHeader),
                         a.idx_out, a.score_out, a.err);
}

}  // namespace csa
