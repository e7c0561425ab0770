// Shared-KV multi-query attention on the fifth-generation tensor cores
// (tcgen05, accumulators in tensor memory) for prefill-sized batches with
// d = 512 ("DeepSeek-V4 core architecture", §2.2 CSA step 3: each selected
// entry is both key and value, shared by all query heads; §2.3 HCA: dense
// attention over every compressed entry).  The key set of a query is the
// same as in attend.cu: selected (or all visible) entries plus the raw
// tokens of the query's own open block.
//
// One CTA computes 64 heads of one query over one split of its keys (all of
// them when there are at least as many 64-head units as SMs; decode splits a
// query's keys over several CTAs), in tiles of 64 keys.  Keys are the M
// dimension of both products:
//     S^T[key, head] = K[key, :] . Q[head, :]       M = 64 keys,      N = 64, K = 512
//     O^T[d, head]  += K[key, d]^T . P^T[key, head]  M = 4 x 128 d,   N = 64, K = 64
// The shared-memory key tile is the K-major A operand of the first product
// and the MN-major A operand of the second; P is stored key-major (one
// 128-byte row of 64 heads per key) as the MN-major B operand.  With M = 64
// the accumulator row r sits in tensor-memory lane 32 (r / 16) + r % 16.
// Two key stages, two S^T buffers and two P stages let the tensor core run
// S^T of tile t+1 and P V of tile t-1 while the softmax of tile t proceeds,
// and the gather of a stage overlap the other stage's products.  Tensor
// memory: S^T x 2 (64 columns each) and O^T (4 x 64 columns).
//
// Warp roles (384 threads): warps 0-3 softmax (thread (w, l) takes key
// 16 w + l % 16 of the tile, heads 32 (l / 16) .. +31; afterwards row
// d = 128 m + 32 w + l of the output), warp 4 lane 0 issues the MMAs, warp 5
// lane 0 issues the tensor-memory-access (TMA) loads: visible entries, raw
// tail rows and the query tile as 64-row tiles, all in the 128-byte swizzled
// layout the MMAs read.  Selected entries are gathered by warps 6-11 with
// 16-byte cp.async (measured faster than four-row TMA gathers of 128-byte
// rows, whose issue rate bounds a tile at about 4 us).  A tile holds either
// entries or raw tail rows, never both, so each comes from one tensor.  The
// running maximum of a head is raised only when a tile exceeds it by more
// than 2^8 (the accumulated O^T column and sum are then rescaled); the
// result is exact either way because the sum uses the same maximum.
// When queries are split (decode-sized calls), every split writes its
// unnormalised O (fp32, [head][d], staged in the idle key stages and stored
// with one bulk copy) and each head's (max, sum), an empty (-inf, 0) when it
// has no tiles; attend_tc_merge_kernel, launched behind it, combines the
// splits: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// Every wait is bounded: one that runs out reports CSA_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tma.h"

namespace csa {

namespace {

using tc::policy_evict_first;
using tc::policy_evict_last;
using tc::tma_tile2d;

constexpr int kTcThreads = 384;
constexpr int kGatherBase = 192;             // first cp.async gather thread (warp 6)
constexpr int kGatherThreads = 192;          // warps 6-11
constexpr int kTcKeys = 64;                  // keys per tile (M of S^T)
constexpr int kTcHeads = 64;                 // heads per CTA (N)
constexpr int kTcD = 512;
constexpr int kRegions = kTcD / 64;          // 64-column regions of a 128-byte swizzled row
constexpr uint32_t kReg = 64 * 128;          // 8 KiB: 64 rows x 128 bytes
constexpr uint32_t kStage = kRegions * kReg; // 64 KiB key stage
constexpr int kTcIdxCap = 2048;
constexpr float kTcLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;         // raise a head's maximum only beyond 2^8

constexpr uint32_t OFF_Q = 0;                              // 8 regions x (64 heads x 128 B)
constexpr uint32_t OFF_K = OFF_Q + kStage;                 // 2 stages x 8 regions x (64 keys x 128 B)
constexpr uint32_t OFF_P = OFF_K + 2 * kStage;             // 2 stages x (64 keys x 128 B)
constexpr uint32_t OFF_BAR = OFF_P + 2 * kReg;
// barriers: kfull[2], kfree[2] (P V of the stage's tile done), sfull[2], sfree[2], pfull[2], ofull, qfull
constexpr int BAR_KFULL = 0, BAR_KFREE = 2, BAR_SFULL = 4, BAR_SFREE = 6, BAR_PFULL = 8, BAR_OFULL = 10,
              BAR_QFULL = 11;
constexpr uint32_t OFF_MISC = OFF_BAR + 16 * 8;
constexpr uint32_t MISC_TMEM = 0, MISC_FLAG = 4, MISC_M = 32, MISC_L = MISC_M + 256, MISC_MN = MISC_L + 256,
                   MISC_AL = MISC_MN + 256, MISC_RMAX = MISC_AL + 256, MISC_RSUM = MISC_RMAX + 1024,
                   MISC_END = MISC_RSUM + 1024;
constexpr uint32_t OFF_IDX = OFF_MISC + MISC_END;
constexpr uint32_t kTcSmem = OFF_IDX + kTcIdxCap * 4 + 1024;   // + alignment slack
static_assert(kTcSmem <= 232448, "shared memory per CTA");

constexpr uint32_t TM_S = 0;     // S^T buffer s: columns 64 s .. 64 s + 63 (M = 64 lane layout)
constexpr uint32_t TM_O = 128;   // O^T block m: columns 128 + 64 m .. +63
constexpr uint32_t kTmemCols = 512;

// 2^x with subnormal results flushed to zero: a softmax weight below 2^-126
// is negligible beside the running sum, which is at least 1.
__device__ __forceinline__ float fast_exp2_ftz(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
    return r;
}
// Reduce 32 values per lane over the 16 lanes of a half-warp (xor 8, 4, 2, 1):
// on return lane l holds the result for values 2 (l % 16) and 2 (l % 16) + 1.
template <bool MAX>
__device__ __forceinline__ void halfwarp_reduce32(const float *v, float &r0, float &r1)
{
    const int lane = threadIdx.x & 31;
    float a[16];
#pragma unroll
    for (int j = 0; j < 16; j++) {
        const bool up = lane & 8;
        const float keep = up ? v[16 + j] : v[j];
        const float send = up ? v[j] : v[16 + j];
        const float got = __shfl_xor_sync(0xffffffffu, send, 8);
        a[j] = MAX ? fmaxf(keep, got) : keep + got;
    }
#pragma unroll
    for (int o = 4, half = 8; o >= 1; o >>= 1, half >>= 1) {
#pragma unroll
        for (int j = 0; j < half; j++) {
            const bool up = lane & o;
            const float keep = up ? a[half + j] : a[j];
            const float send = up ? a[j] : a[half + j];
            const float got = __shfl_xor_sync(0xffffffffu, send, o);
            a[j] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    r0 = a[0];
    r1 = a[1];
}

// 4-byte cp.async (both addresses 4-byte aligned).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
// The eight 16-byte chunks of one row's chunk column across the eight 64-column
// regions of a key stage: shared addresses dst + 8 KiB r, global src + 128 r
// bytes (r = 0..7), all zero-filled when src_bytes is 0.  Immediate offsets
// keep the issue to one instruction per chunk.
__device__ __forceinline__ void cp_async_16_regions(uint32_t dst, const void *src, int src_bytes, uint64_t pol)
{
    asm volatile(
        "cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n"
        "cp.async.cg.shared.global.L2::cache_hint [%0+8192], [%1+128], 16, %2, %3;\n"
        "cp.async.cg.shared.global.L2::cache_hint [%0+16384], [%1+256], 16, %2, %3;\n"
        "cp.async.cg.shared.global.L2::cache_hint [%0+24576], [%1+384], 16, %2, %3;\n"
        "cp.async.cg.shared.global.L2::cache_hint [%0+32768], [%1+512], 16, %2, %3;\n"
        "cp.async.cg.shared.global.L2::cache_hint [%0+40960], [%1+640], 16, %2, %3;\n"
        "cp.async.cg.shared.global.L2::cache_hint [%0+49152], [%1+768], 16, %2, %3;\n"
        "cp.async.cg.shared.global.L2::cache_hint [%0+57344], [%1+896], 16, %2, %3;\n" ::"r"(dst),
        "l"(src), "r"(src_bytes), "l"(pol)
        : "memory");
}
static_assert(kReg == 8192 && kRegions == 8, "the region offsets of cp_async_16_regions");

// Main keys of a query with n_vis visible entries: the selected entries
// (GATHER: at most top_k), or the visible entries themselves, all of them, or
// with top_k > 0 only the most recent top_k (a sliding window; the first of
// them is entry n_vis - n_main).
__device__ __forceinline__ int tc_main_keys(int64_t n_vis, int top_k)
{
    return (int)(top_k > 0 && n_vis > top_k ? top_k : n_vis);
}

// Key tiles of the query at `p`: the main keys fill ceil(n_main / 64)
// tiles, the raw tail its own ceil(r / 64) tiles.
template <bool GATHER>
__device__ __forceinline__ int tc_tiles(const QueryPos &p, int ratio, int top_k, int *t_main)
{
    const int64_t n_vis = (p.t + 1) / ratio;
    const int n_main = tc_main_keys(n_vis, top_k);
    const int r_tail = (int)((p.t + 1) % ratio);
    const int tm = (n_main + kTcKeys - 1) / kTcKeys;
    if (t_main) *t_main = tm;
    return tm + (r_tail + kTcKeys - 1) / kTcKeys;
}

// A query with T key tiles runs in min(nsplit_max, T) splits; split s takes
// tiles [s T / ns, (s + 1) T / ns).
__device__ __forceinline__ int tc_nsplit(int T, int nsplit_max) { return T < nsplit_max ? T : nsplit_max; }

template <bool GATHER>
__global__ void __launch_bounds__(kTcThreads, 1)
attend_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_ent_rows,
                 const __grid_constant__ CUtensorMap map_kv,
                 int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                 const int64_t *__restrict__ cu_ent, const uint16_t *__restrict__ entries,
                 const int32_t *__restrict__ idx, int H,
                 int ratio, int top_k, float scale_log2, int max_kv_len, int nsplit_max,
                 uint16_t *__restrict__ out, float *__restrict__ lse, float *__restrict__ part_o,
                 float2 *__restrict__ part_ml, int *err)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;          // swizzled tiles need 1024-byte alignment
    uint8_t *sm = smem_raw + (sb - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t qi = blockIdx.x;
    const int HG = H / kTcHeads;
    const int hg = blockIdx.y % HG;
    const int split = blockIdx.y / HG;

    const QueryPos p = query_pos(cu_kv, cu_q, cu_ent, batch, qi);
    const int64_t n_vis = (p.t + 1) / ratio;
    const int r_tail = (int)((p.t + 1) % ratio);
    const bool bad = p.t < 0 || p.t >= p.L || p.L > max_kv_len || p.ne != p.L / ratio;
    // with splits, every slot of (max, sum) is written, empty where a split has
    // no keys, so the merge reads them all without locating the query
    const int64_t ml_slot = ((qi * HG + hg) * nsplit_max + split) * kTcHeads;
    if (bad) {
        if (tid == 0) set_error(err, CSA_ERR_DEVICE);
        if (nsplit_max > 1 && tid < kTcHeads) part_ml[ml_slot + tid] = make_float2(-INFINITY, 0.f);
        return;
    }
    const int n_main = tc_main_keys(n_vis, top_k);
    const int64_t e_first = p.e0 + (GATHER ? 0 : n_vis - n_main);   // dense: the first main entry row
    int T_main = 0;
    const int T_all = tc_tiles<GATHER>(p, ratio, top_k, &T_main);
    const int nsplit = tc_nsplit(T_all, nsplit_max);
    if (split >= nsplit) {   // this query has fewer key tiles than splits
        if (tid < kTcHeads) part_ml[ml_slot + tid] = make_float2(-INFINITY, 0.f);
        return;
    }
    const int t0 = (int)((int64_t)split * T_all / nsplit), t1 = (int)((int64_t)(split + 1) * T_all / nsplit);
    const int T = t1 - t0;
    // main-key slots of this split (selection entries read here)
    const int slot0 = min(t0, T_main) * kTcKeys;
    const int slot1 = min(min(t1, T_main) * kTcKeys, n_main);
    const int64_t tail_row0 = p.kv0 + p.t - r_tail + 1;

    const uint32_t bar0 = sb + OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint8_t *misc = sm + OFF_MISC;
    float *s_m = reinterpret_cast<float *>(misc + MISC_M);
    float *s_l = reinterpret_cast<float *>(misc + MISC_L);
    float *s_al = reinterpret_cast<float *>(misc + MISC_AL);
    float *s_rmax = reinterpret_cast<float *>(misc + MISC_RMAX);   // [4 warps][64 heads]
    float *s_rsum = reinterpret_cast<float *>(misc + MISC_RSUM);
    volatile int *s_flag = reinterpret_cast<volatile int *>(misc + MISC_FLAG);

    if (tid == 0) {
        mbar_init(bar(BAR_QFULL), 1);
        for (int s = 0; s < 2; s++) {
            mbar_init(bar(BAR_KFULL + s), 1 + kGatherThreads);   // TMA issuer + cp.async gatherers
            mbar_init(bar(BAR_KFREE + s), 1);
            mbar_init(bar(BAR_SFULL + s), 1);
            mbar_init(bar(BAR_SFREE + s), 128);
            mbar_init(bar(BAR_PFULL + s), 128);
        }
        mbar_init(bar(BAR_OFULL), 1);
        fence_mbar_init();
    }
    if (tid < kTcHeads) {
        s_m[tid] = -INFINITY;
        s_l[tid] = 0.f;
    }
    if (warp == 4) tc::tmem_alloc(sb + OFF_MISC + MISC_TMEM, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(misc + MISC_TMEM);

    // the query tile is an input of the call: it loads while the kernels
    // before this one finish
    if (warp == 5 && lane == 0) {
        mbar_expect_tx(bar(BAR_QFULL), kStage);
        const int qrow = (int)(qi * H + (int64_t)hg * kTcHeads);
        const uint64_t once = policy_evict_first();
#pragma unroll
        for (int r = 0; r < kRegions; r++)
            tma_tile2d(sb + OFF_Q + r * kReg, &map_q, r * 64, qrow, bar(BAR_QFULL), once);
    }
    // the selection and the entries come from earlier kernels
    griddep_wait();
    // this split's part of the selection (slot1 - slot0 <= top_k <= kTcIdxCap)
    int32_t *s_idx = reinterpret_cast<int32_t *>(sm + OFF_IDX);
    if (GATHER)
        for (int i = slot0 + tid; i < slot1; i += kTcThreads) s_idx[i - slot0] = __ldg(idx + qi * top_k + i);
    __syncthreads();

    if (warp == 5) {
        // ------------------------------------------------------------ producer
        // Tile tt of the split goes to stage tt & 1, once P V of tile tt - 2
        // has released it.  Invalid selections read entry row 0 (the softmax
        // masks them).
        if (lane == 0) {
            const uint64_t keep = policy_evict_last(), once = policy_evict_first();
            int tt = 0;
            for (; tt < T; tt++) {
                const int g = tt & 1;
                if (tt >= 2 && !mbar_wait(bar(BAR_KFREE + g), (uint32_t)(((tt - 2) >> 1) & 1))) {
                    set_error(err, CSA_ERR_TIMEOUT);
                    break;
                }
                const uint32_t stage = sb + OFF_K + g * kStage;
                const uint32_t fb = bar(BAR_KFULL + g);
                const int tile = t0 + tt;
                mbar_expect_tx(fb, (GATHER && tile < T_main) ? 0u : kStage);   // selected entries: cp.async
                if (tile < T_main) {
                    if (!GATHER) {
                        const int row = (int)(e_first + (int64_t)tile * kTcKeys);
#pragma unroll
                        for (int r = 0; r < kRegions; r++)
                            tma_tile2d(stage + r * kReg, &map_ent_rows, r * 64, row, fb, keep);
                    }
                } else {
                    const int row = (int)(tail_row0 + (int64_t)(tile - T_main) * kTcKeys);
#pragma unroll
                    for (int r = 0; r < kRegions; r++) tma_tile2d(stage + r * kReg, &map_kv, r * 64, row, fb, once);
                }
            }
            // no load may still be writing when the CTA ends (normally they
            // have all been consumed): the last phase of each stage
            for (int u = tt - 1; u >= 0 && u >= tt - 2; u--)
                if (!mbar_wait(bar(BAR_KFULL + (u & 1)), (uint32_t)((u >> 1) & 1))) set_error(err, CSA_ERR_TIMEOUT);
            if (!mbar_wait(bar(BAR_QFULL), 0)) set_error(err, CSA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ------------------------------------------------------------ cp.async gatherers
        // Thread pt copies 16-byte chunk pt % 8 of rows pt / 8, + 24, ... in
        // every region of selected-entry tiles; every thread arrives on each
        // tile's KFULL (after its own copies landed), whatever the tile.
        const int pt = tid - kGatherBase;
        const int pc = pt & 7, pk0 = pt >> 3;
        constexpr int RSTEP = kGatherThreads / 8;                 // 24 rows per pass
        constexpr int KPP = (kTcKeys + RSTEP - 1) / RSTEP;        // 3 rows per thread
        const uint64_t keep = policy_evict_last();
        for (int tt = 0; tt < T; tt++) {
            const int g = tt & 1;
            if (tt >= 2 && !mbar_wait(bar(BAR_KFREE + g), (uint32_t)(((tt - 2) >> 1) & 1))) {
                set_error(err, CSA_ERR_TIMEOUT);
                break;
            }
            const int tile = t0 + tt;
            if (GATHER && tile < T_main) {
                const uint32_t stage = sb + OFF_K + g * kStage;
#pragma unroll
                for (int i = 0; i < KPP; i++) {
                    const int k = pk0 + RSTEP * i;
                    if (k < kTcKeys) {
                        const int slot = tile * kTcKeys + k;
                        const int e = slot < slot1 ? s_idx[slot - slot0] : -1;
                        const bool v = e >= 0 && (int64_t)e < n_vis;
                        const uint16_t *src = entries + (p.e0 + (v ? e : 0)) * kTcD;
                        cp_async_16_regions(stage + k * 128 + ((pc ^ (k & 7)) << 4), src + pc * 8, v ? 16 : 0, keep);
                    }
                }
                cp_async_commit();
                cp_async_wait<0>();
                tc::fence_proxy_async();
            }
            mbar_arrive(bar(BAR_KFULL + g));
        }
        cp_async_wait<0>();
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        // S(t) and PV(t) are each issued in tile order; the issuer polls both
        // and issues whichever is ready first (S(t) needs tile t and a free S
        // buffer, PV(t) needs P(t)), so neither the gather of the next tile nor
        // the softmax of the current one stalls the other product.
        if (lane == 0) {
            constexpr uint32_t id_qk = tc::idesc_bf16_f32(64, kTcHeads, false, false);
            constexpr uint32_t id_pv = tc::idesc_bf16_f32(128, kTcHeads, true, true);
            const uint64_t qa0 = tc::sdesc_sw128(sb + OFF_K, 16, 1024);
            const uint64_t qb0 = tc::sdesc_sw128(sb + OFF_Q, 16, 1024);
            const uint64_t pa0 = tc::sdesc_sw128(sb + OFF_K, kReg, 1024);
            const uint64_t pb0 = tc::sdesc_sw128(sb + OFF_P, kReg, 1024);
            bool ok = mbar_wait(bar(BAR_QFULL), 0);   // the query tile
            int nq = 0, np = 0;                       // next S tile, next PV tile
            uint64_t idle0 = global_ns();
            while (ok && np < T) {
                bool did = false;
                if (nq < T && nq <= np + 1) {
                    const int sidx = nq & 1;
                    if ((nq < 2 || mbar_test(bar(BAR_SFREE + sidx), (uint32_t)(((nq - 2) >> 1) & 1))) &&
                        mbar_test(bar(BAR_KFULL + sidx), (uint32_t)((nq >> 1) & 1))) {
                        tc::fence_after_sync();
                        // descriptors advance by adding (byte offset >> 4) to the address field
                        const uint64_t a0 = qa0 + (uint64_t)((sidx * kStage) >> 4);
                        const uint32_t dS = tmem + TM_S + 64 * sidx;
#pragma unroll
                        for (int j = 0; j < kTcD / 16; j++) {
                            const uint64_t off = (uint64_t)(((j >> 2) * kReg + (j & 3) * 32) >> 4);
                            tc::mma_ss(dS, a0 + off, qb0 + off, id_qk, j != 0);
                        }
                        tc::mma_commit(bar(BAR_SFULL + sidx));
                        nq++;
                        did = true;
                    }
                }
                if (np < nq) {
                    const int sidx = np & 1;
                    if (mbar_test(bar(BAR_PFULL + sidx), (uint32_t)((np >> 1) & 1))) {
                        tc::fence_after_sync();
                        const uint64_t a0 = pa0 + (uint64_t)((sidx * kStage) >> 4);
                        const uint64_t b0 = pb0 + (uint64_t)((sidx * kReg) >> 4);
#pragma unroll
                        for (int m = 0; m < 4; m++)
#pragma unroll
                            for (int k4 = 0; k4 < kTcKeys / 16; k4++)
                                tc::mma_ss(tmem + TM_O + 64 * m, a0 + (uint64_t)((2 * m * kReg + k4 * 2048) >> 4),
                                           b0 + (uint64_t)((k4 * 2048) >> 4), id_pv, np > 0 || k4 > 0);
                        tc::mma_commit(bar(BAR_KFREE + sidx));
                        np++;
                        did = true;
                    }
                }
                if (did) {
                    idle0 = global_ns();
                } else {
                    // back off briefly: this warp shares its scheduler with a softmax warp
                    __nanosleep(20);
                    if (global_ns() - idle0 > kWaitLimitNs) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) set_error(err, CSA_ERR_TIMEOUT);
            // every issued product completes before the CTA ends
            tc::mma_commit(bar(BAR_OFULL));
            if (!mbar_wait(bar(BAR_OFULL), 0)) set_error(err, CSA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax (128 threads)
        // Thread (w, l) takes key 16 w + l % 16 of each tile for heads
        // 32 hh .. 32 hh + 31 (hh = l / 16).  It keeps the running maximum of
        // those heads in registers (the same in every thread of the half) and
        // its own partial sums of their weights over its keys; the sums are
        // reduced over keys once, after the last tile.  A tile reduces its
        // maximum over keys only when one of its scores exceeds the running
        // maximum by more than 2^8 (one OR-reducing barrier per tile decides),
        // which after the first tiles is rare.
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int hh = lane >> 4;                 // head half: heads 32 hh .. 32 hh + 31
        const int key = 16 * warp + (lane & 15);  // key of the tile this thread takes
        bool ok = true;
        bool fail = false;   // a wait of this thread gave up (acted on at the next barrier reduction)
        float m_run[32], l_part[32];
#pragma unroll
        for (int j = 0; j < 32; j++) {
            m_run[j] = -INFINITY;
            l_part[j] = 0.f;
        }
        for (int t = 0; t < T; t++) {
            const int sidx = t & 1;
            if (!mbar_wait(bar(BAR_SFULL + sidx), (uint32_t)((t >> 1) & 1))) fail = true;
            tc::fence_after_sync();
            float v[64];
            tc::tmem_ld32(tmem + lane_base + TM_S + 64 * sidx, v);
            tc::tmem_ld32(tmem + lane_base + TM_S + 64 * sidx + 32, v + 32);
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            mbar_arrive(bar(BAR_SFREE + sidx));
            // lanes 0-15 hold the tile's rows: hand heads 32-63 to lanes 16-31
            float s[32];
#pragma unroll
            for (int j = 0; j < 32; j++) {
                const float other = __shfl_xor_sync(0xffffffffu, v[32 + j], 16);
                s[j] = hh ? other : v[j];
            }
            const int tile = t0 + t;
            bool valid;
            if (tile < T_main) {
                const int slot = tile * kTcKeys + key;
                valid = slot < n_main;
                if (GATHER && valid) {
                    const int e = s_idx[slot - slot0];
                    valid = e >= 0 && (int64_t)e < n_vis;
                    if (e >= 0 && !valid) set_error(err, CSA_ERR_DEVICE);   // an index that is not visible
                }
            } else {
                valid = (tile - T_main) * kTcKeys + key < r_tail;
            }
            bool exceed = false;
#pragma unroll
            for (int j = 0; j < 32; j++) {
                s[j] = valid ? s[j] * scale_log2 : -INFINITY;
                exceed |= s[j] > m_run[j] + kRescaleLog2;   // a finite score always exceeds -inf
            }
            bool rescale = false;
            if (tc::named_bar_or(1, 128, exceed || fail)) {
                if (tc::named_bar_or(1, 128, fail)) {   // a wait gave up: every thread leaves together
                    ok = false;
                    break;
                }
                float r0, r1;
                halfwarp_reduce32<true>(s, r0, r1);
                const int h2 = 32 * hh + 2 * (lane & 15);
                s_rmax[warp * 64 + h2] = r0;
                s_rmax[warp * 64 + h2 + 1] = r1;
                if (tid == 0) s_flag[1] = 0;
                tc::named_bar(1, 128);
                if (tid < kTcHeads) {
                    const float M = fmaxf(fmaxf(s_rmax[tid], s_rmax[64 + tid]), fmaxf(s_rmax[128 + tid], s_rmax[192 + tid]));
                    const float m_old = s_m[tid];
                    float m_new = m_old, alpha = 1.f;
                    if (M > m_old + kRescaleLog2 || (m_old == -INFINITY && M != -INFINITY)) {
                        m_new = M;
                        alpha = fast_exp2(m_old - m_new);   // 0 when nothing was accumulated yet
                        if (t > 0) s_flag[1] = 1;
                    }
                    s_m[tid] = m_new;
                    s_al[tid] = alpha;
                }
                tc::named_bar(1, 128);
                rescale = s_flag[1] != 0;
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    m_run[j] = s_m[32 * hh + j];
                    l_part[j] *= s_al[32 * hh + j];
                }
            }
#pragma unroll
            for (int j = 0; j < 32; j++) {
                s[j] = (m_run[j] == -INFINITY) ? 0.f : fast_exp2_ftz(s[j] - m_run[j]);
                l_part[j] += s[j];
            }
            // This P stage was last read by P V of tile t - 2, which must be done.
            // A rescale of the O^T columns also needs P V of tile t - 1 done; the
            // lazy maximum makes that rare, so P V of the previous tile usually
            // still runs while this tile's probabilities are written.
            if (rescale ? (t >= 1 && !mbar_wait(bar(BAR_KFREE + ((t - 1) & 1)), (uint32_t)(((t - 1) >> 1) & 1)))
                        : (t >= 2 && !mbar_wait(bar(BAR_KFREE + (t & 1)), (uint32_t)(((t - 2) >> 1) & 1))))
                fail = true;
            {
                uint8_t *prow = sm + OFF_P + sidx * kReg + key * 128;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const int ch = 4 * hh + c;
                    uint4 w;
                    w.x = pack_bf16x2(s[8 * c + 0], s[8 * c + 1]);
                    w.y = pack_bf16x2(s[8 * c + 2], s[8 * c + 3]);
                    w.z = pack_bf16x2(s[8 * c + 4], s[8 * c + 5]);
                    w.w = pack_bf16x2(s[8 * c + 6], s[8 * c + 7]);
                    *reinterpret_cast<uint4 *>(prow + ((ch ^ (key & 7)) << 4)) = w;
                }
            }
            if (rescale) {
                tc::fence_after_sync();
#pragma unroll 1
                for (int c = 0; c < 8; c++) {
                    float o[32];
                    const uint32_t ta = tmem + lane_base + TM_O + 32 * c;
                    tc::tmem_ld32(ta, o);
                    tc::tmem_wait_ld();
                    const float *al = s_al + 32 * (c & 1);
#pragma unroll
                    for (int j = 0; j < 32; j++) o[j] *= al[j];
                    tc::tmem_st32(ta, o);
                }
                tc::tmem_wait_st();
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            mbar_arrive(bar(BAR_PFULL + sidx));
        }
        // the weights' sums over keys, once: lanes (keys) within each warp, then the warps
        if (tc::named_bar_or(1, 128, fail)) ok = false;
        {
            float r0, r1;
            halfwarp_reduce32<false>(l_part, r0, r1);
            const int h2 = 32 * hh + 2 * (lane & 15);
            s_rsum[warp * 64 + h2] = r0;
            s_rsum[warp * 64 + h2 + 1] = r1;
        }
        tc::named_bar(1, 128);
        if (tid < kTcHeads) s_l[tid] = s_rsum[tid] + s_rsum[64 + tid] + s_rsum[128 + tid] + s_rsum[192 + tid];
        // epilogue: O^T / l -> out[head][d] (bf16), lse
        bool done = ok && mbar_wait(bar(BAR_OFULL), 0);
        done = !tc::named_bar_or(1, 128, !done);   // also: s_l is complete
        if (done && nsplit_max > 1) {   // the merge normalises, also a query's only split
            // partial result: unnormalised O^T -> [head][d] fp32 in the key
            // stages (every product is done with them), one bulk store
            tc::fence_after_sync();
            float *stg = reinterpret_cast<float *>(sm + OFF_K);
#pragma unroll 1
            for (int c = 0; c < 8; c++) {
                float o[32];
                tc::tmem_ld32(tmem + lane_base + TM_O + 32 * c, o);
                tc::tmem_wait_ld();
                const int d = 128 * (c >> 1) + tid;
                const int h0 = 32 * (c & 1);
#pragma unroll
                for (int j = 0; j < 32; j++) stg[(h0 + j) * kTcD + d] = o[j];
            }
            tc::fence_proxy_async();
            tc::named_bar(1, 128);
            const int64_t slot = ((qi * HG + hg) * nsplit_max + split) * kTcHeads;
            if (tid == 0) {
                bulk_s2g(part_o + slot * kTcD, sb + OFF_K, kTcHeads * kTcD * 4);
                bulk_commit();
                bulk_wait_read();
            }
            if (tid < kTcHeads) part_ml[slot + tid] = make_float2(s_m[tid], s_l[tid]);
        } else if (done) {
            // 1/l once per head; the bf16 result [64 heads][512] is staged in
            // the key stages (every product is done with them) and leaves with
            // one bulk copy: the query's 64 head rows are contiguous in `out`
            if (tid < kTcHeads) {
                const float l = s_l[tid];
                s_al[tid] = l > 0.f ? 1.f / l : 0.f;
            }
            tc::named_bar(1, 128);
            tc::fence_after_sync();
            uint16_t *stg = reinterpret_cast<uint16_t *>(sm + OFF_K);
#pragma unroll 1
            for (int c = 0; c < 8; c++) {
                float o[32];
                tc::tmem_ld32(tmem + lane_base + TM_O + 32 * c, o);
                tc::tmem_wait_ld();
                const int d = 128 * (c >> 1) + tid;
                const int h0 = 32 * (c & 1);
#pragma unroll
                for (int j = 0; j < 32; j++)
                    stg[(h0 + j) * kTcD + d] = (uint16_t)(pack_bf16x2(o[j] * s_al[h0 + j], 0.f) & 0xffffu);
            }
            tc::fence_proxy_async();
            tc::named_bar(1, 128);
            if (tid == 0) {
                bulk_s2g(out + (qi * H + (int64_t)hg * kTcHeads) * kTcD, sb + OFF_K, kTcHeads * kTcD * 2);
                bulk_commit();
                bulk_wait_read();
            }
            if (lse && tid < kTcHeads)
                lse[qi * H + (int64_t)hg * kTcHeads + tid] = (s_m[tid] + log2f(s_l[tid])) * kTcLn2;
        } else if (tid == 0) {
            set_error(err, CSA_ERR_TIMEOUT);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    // The merge kernel may launch once every CTA is here (or has exited); the
    // first thread of a CTA to execute the trigger fires it, so it follows the
    // barrier.  Launched earlier, the merge CTAs would wait on SMs that
    // attention CTAs need.
    griddep_launch();
    tc::fence_after_sync();
    if (warp == 4) tc::tmem_dealloc(tmem, kTmemCols);
}

// Combines the splits of the queries that have more than one.  CTA (i, h)
// takes head h of query i; thread c holds columns 4 c .. 4 c + 3 and keeps
// the loads of up to kMergeBatch splits in flight at once (the partial
// results are read from L2, so the merge is bound by how many loads are in
// flight).  One 4-warp CTA fits beside a resident attention CTA, so the
// grid, launched early, waits on every SM.
constexpr int kMergeThreads = kTcD / 4;
constexpr int kMergeBatch = 8;

template <bool GATHER>
__global__ void __launch_bounds__(kMergeThreads, 8)
attend_tc_merge_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                       const int64_t *__restrict__ cu_ent, int H, int ratio, int top_k, int nsplit_max,
                       const float *__restrict__ part_o, const float2 *__restrict__ part_ml,
                       uint16_t *__restrict__ out, float *__restrict__ lse)
{
    const int c = threadIdx.x;
    const int64_t qi = blockIdx.x;
    const int head = blockIdx.y;
    // every split slot holds a (max, sum): empty (-inf, 0) where the query has
    // fewer tiles than splits, or a layout error (its row then reads zeros)
    const int nsplit = nsplit_max;
    griddep_wait();            // the partial results are complete
    const int64_t base = (qi * (H / kTcHeads) + head / kTcHeads) * nsplit_max * kTcHeads + head % kTcHeads;
    // up to kMergeBatch splits' (max, sum) and columns are loaded at once, one
    // round trip; the maximum over the batches so far is carried, and what was
    // accumulated is rescaled when it rises (never within a single batch)
    float M = -INFINITY, Ls = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 *po = reinterpret_cast<const float4 *>(part_o + base * kTcD) + c;
    for (int s0 = 0; s0 < nsplit; s0 += kMergeBatch) {
        float4 v[kMergeBatch];
        float2 ml[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; u++) {
            if (s0 + u < nsplit) {
                v[u] = __ldcg(po + (int64_t)(s0 + u) * kTcHeads * (kTcD / 4));
                ml[u] = __ldcg(part_ml + base + (int64_t)(s0 + u) * kTcHeads);
            }
        }
        float Mb = M;
#pragma unroll
        for (int u = 0; u < kMergeBatch; u++)
            if (s0 + u < nsplit) Mb = fmaxf(Mb, ml[u].x);
        if (Mb > M) {
            const float r = M == -INFINITY ? 0.f : fast_exp2(M - Mb);   // nothing accumulated under -inf
            Ls *= r;
            acc.x *= r;
            acc.y *= r;
            acc.z *= r;
            acc.w *= r;
            M = Mb;
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; u++) {
            if (s0 + u < nsplit && ml[u].x != -INFINITY) {   // an empty split's columns are not read
                const float w = fast_exp2(ml[u].x - M);
                Ls = fmaf(w, ml[u].y, Ls);
                acc.x = fmaf(w, v[u].x, acc.x);
                acc.y = fmaf(w, v[u].y, acc.y);
                acc.z = fmaf(w, v[u].z, acc.z);
                acc.w = fmaf(w, v[u].w, acc.w);
            }
        }
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(out + (qi * H + head) * (int64_t)kTcD + 4 * c) = pk;
    if (lse && c == 0) lse[qi * H + head] = (M + log2f(Ls)) * kTcLn2;
}

// ---------------------------------------------------------------------------
// Persistent form, for calls with one split per query (prefill-sized): one
// CTA per SM walks work items (64 heads of one query), taken longest first
// from a counter in the workspace, so that an item's query tile, selection
// and first key tiles load while the previous item's last tiles and
// epilogue run.  The roles and products are those of attend_tc_kernel; key
// tiles are numbered across items, so the stage, S and P barriers keep their
// phases.  The TMA warp takes each item and publishes its record in a ring of
// four slots, one item ahead of the item whose loads it issues; the gather
// warps, the MMA issuer, the softmax warps and the epilogue warps each release
// a slot once they have read it.  Per item: the query tile is reloaded once
// every S^T of the previous item has completed (QFREE), the item's first P V
// overwrites O^T once the previous epilogue has read it (OFREE), and the
// selection indices rotate through three buffers (IDXFULL / IDXFREE), the
// gather warps copying the next item's while the current one runs.  The softmax warps hand each item's per-head maximum,
// sum and 1 / sum to four epilogue warps through a two-slot buffer (LFULL /
// LFREE) and go straight on to the next item; the epilogue warps (one per
// tensor-memory lane quarter) store O / l from registers (two neighbouring d
// of one head per thread) and the LSE, and the last CTA to finish returns the
// counters to zero.
constexpr int kTcpIdxCap = 1024;   // selection indices per buffer
constexpr int kTcpIdxBufs = 3;
constexpr int kTcpRing = 4;
constexpr uint32_t OFF_BARP = OFF_P + 2 * kReg;
constexpr int PB_KFULL = 0, PB_KFREE = 2, PB_SFULL = 4, PB_SFREE = 6, PB_PFULL = 8, PB_OFULL = 10, PB_QFULL = 11,
              PB_QFREE = 12, PB_OFREE = 13, PB_IDXFULL = 14, PB_IDXFREE = 17, PB_IFULL = 20, PB_IFREE = 24,
              PB_FIN = 28, PB_LFULL = 29, PB_LFREE = 31, PB_COUNT = 33;
// warps 6-7 gather selected entries, warps 8-11 (one per tensor-memory lane quarter) write the epilogue
constexpr int kTcpGatherThreads = 64;
constexpr int kTcpEpiBase = 256;
constexpr uint32_t OFF_MISCP = OFF_BARP + 40 * 8;
static_assert(PB_COUNT <= 40, "persistent barriers fit their area");

struct alignas(16) TcItem {
    int64_t qi;          // query
    int64_t n_vis;       // visible entries
    int64_t e0;          // first entry row of the query's sequence
    int64_t tail_row0;   // first raw row of the query's open block
    int hg;              // 64-head group
    int T;               // key tiles; 0: skip the item (layout error), -1: no more items
    int T_main;          // tiles of selected (or visible) entries
    int n_main;          // selected (or visible) entries
    int r_tail;          // raw tail rows
};
constexpr uint32_t OFF_RING = OFF_MISCP + MISC_END;
constexpr uint32_t OFF_IDXP = (OFF_RING + kTcpRing * (uint32_t)sizeof(TcItem) + 15u) & ~15u;
constexpr uint32_t OFF_LBUF = OFF_IDXP + kTcpIdxBufs * kTcpIdxCap * 4;   // [2][3][64]: per item buffer, max, sum, 1 / sum of each head
constexpr uint32_t kTcpSmem = OFF_LBUF + 2 * 3 * kTcHeads * 4 + 1024;   // + alignment slack
static_assert(kTcpSmem <= 232448, "shared memory per CTA");
constexpr size_t kTcpHeader = 256;   // workspace: next item, CTAs done

template <bool GATHER>
__global__ void __launch_bounds__(kTcThreads, 1)
attend_tcp_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_ent_rows,
                  const __grid_constant__ CUtensorMap map_kv, int batch, const int64_t *__restrict__ cu_kv,
                  const int64_t *__restrict__ cu_q, const int64_t *__restrict__ cu_ent,
                  const uint16_t *__restrict__ entries, const int32_t *__restrict__ idx, int H, int ratio, int top_k,
                  float scale_log2, int max_kv_len, int64_t n_items, unsigned *__restrict__ counters,
                  uint16_t *__restrict__ out, float *__restrict__ lse, int *err)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;          // swizzled tiles need 1024-byte alignment
    uint8_t *sm = smem_raw + (sb - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HG = H / kTcHeads;
    auto bar = [&](int i) { return sb + OFF_BARP + 8u * (uint32_t)i; };
    uint8_t *misc = sm + OFF_MISCP;
    float *s_m = reinterpret_cast<float *>(misc + MISC_M);
    float *s_al = reinterpret_cast<float *>(misc + MISC_AL);
    float *s_rmax = reinterpret_cast<float *>(misc + MISC_RMAX);   // [4 warps][64 heads]
    float *s_rsum = reinterpret_cast<float *>(misc + MISC_RSUM);
    volatile int *s_flag = reinterpret_cast<volatile int *>(misc + MISC_FLAG);
    TcItem *ring = reinterpret_cast<TcItem *>(sm + OFF_RING);
    int32_t *s_idx0 = reinterpret_cast<int32_t *>(sm + OFF_IDXP);

    if (tid == 0) {
        mbar_init(bar(PB_QFULL), 1);
        mbar_init(bar(PB_QFREE), 1);
        for (int s = 0; s < 2; s++) {
            mbar_init(bar(PB_KFULL + s), 1 + kTcpGatherThreads);   // TMA issuer + cp.async gatherers
            mbar_init(bar(PB_KFREE + s), 1);
            mbar_init(bar(PB_SFULL + s), 1);
            mbar_init(bar(PB_SFREE + s), 128);
            mbar_init(bar(PB_PFULL + s), 128);
            mbar_init(bar(PB_LFULL + s), 128);   // the softmax warps: the item's (max, sum) are written
            mbar_init(bar(PB_LFREE + s), 128);   // the epilogue warps: read
        }
        for (int b = 0; b < kTcpIdxBufs; b++) {
            mbar_init(bar(PB_IDXFULL + b), kTcpGatherThreads);
            mbar_init(bar(PB_IDXFREE + b), 128);
        }
        mbar_init(bar(PB_OFULL), 1);
        mbar_init(bar(PB_OFREE), 128);
        for (int k = 0; k < kTcpRing; k++) {
            mbar_init(bar(PB_IFULL + k), 1);
            mbar_init(bar(PB_IFREE + k), 4);   // gather warps, MMA issuer, softmax warps, epilogue warps
        }
        mbar_init(bar(PB_FIN), 1);
        fence_mbar_init();
    }
    if (warp == 4) tc::tmem_alloc(sb + OFF_MISCP + MISC_TMEM, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(misc + MISC_TMEM);
    // the selection and the entries come from earlier kernels
    griddep_wait();
    // record k of the ring, once published (every calling thread waits)
    auto item_at = [&](uint32_t k, TcItem &it) -> bool {
        if (!mbar_wait(bar(PB_IFULL + (int)(k % kTcpRing)), (k / kTcpRing) & 1u)) return false;
        it = ring[k % kTcpRing];
        return true;
    };

    if (warp == 5) {
        // ------------------------------------------------------------ items, query tiles, TMA loads
        bool ok = true;
        uint32_t g = 0, ri = 0;   // key tiles and items with tiles so far
        const uint64_t keep = policy_evict_last(), once = policy_evict_first();
        // take item k, longest rows first, and publish its record
        auto publish = [&](uint32_t k, TcItem &it) -> bool {
            const int slot = (int)(k % kTcpRing);
            int okw = 1;
            if (lane == 0 && k >= kTcpRing && !mbar_wait(bar(PB_IFREE + slot), ((k - kTcpRing) / kTcpRing) & 1u)) okw = 0;
            if (!__shfl_sync(0xffffffffu, okw, 0)) return false;
            unsigned j = 0;
            if (lane == 0) j = atomicAdd(counters, 1u);
            j = __shfl_sync(0xffffffffu, j, 0);
            it.T = -1;
            if ((int64_t)j < n_items) {
                const int64_t jj = n_items - 1 - (int64_t)j;
                it.qi = jj / HG;
                it.hg = (int)(jj % HG);
                const QueryPos p = query_pos(cu_kv, cu_q, cu_ent, batch, it.qi);
                const bool bad = p.t < 0 || p.t >= p.L || p.L > max_kv_len || p.ne != p.L / ratio;
                it.n_vis = (p.t + 1) / ratio;
                it.r_tail = (int)((p.t + 1) % ratio);
                it.n_main = tc_main_keys(it.n_vis, top_k);
                // gathered rows are indexed from the sequence's first entry,
                // dense tiles start at the first main entry
                it.e0 = p.e0 + (GATHER ? 0 : it.n_vis - it.n_main);
                it.tail_row0 = p.kv0 + p.t - it.r_tail + 1;
                it.T = bad ? 0 : tc_tiles<GATHER>(p, ratio, top_k, &it.T_main);
                if (bad && lane == 0) set_error(err, CSA_ERR_DEVICE);
            }
            if (lane == 0) {
                ring[slot] = it;
                mbar_arrive(bar(PB_IFULL + slot));
            }
            __syncwarp();
            return true;
        };
        // With many items per CTA the next record goes out before this item's
        // loads, so that the other roles can prepare the next item while this
        // one runs; with few, a CTA holding an item it has not started would
        // leave another CTA without work, so the next item is taken after them.
        const bool ahead = n_items >= 8 * (int64_t)gridDim.x;
        TcItem nxt;
        if (!publish(0, nxt)) ok = false;
        for (uint32_t k = 0; ok && nxt.T >= 0; k++) {
            const TcItem it = nxt;
            if (ahead && !publish(k + 1, nxt)) {
                ok = false;
                break;
            }
            if (it.T == 0) {
                if (!ahead && !publish(k + 1, nxt)) ok = false;
                continue;
            }
            int okw = 1;
            if (lane == 0) {
                // the query tile: every S^T of the previous item is done with it
                if (ri > 0 && !mbar_wait(bar(PB_QFREE), (ri - 1) & 1u)) okw = 0;
                if (okw) {
                    mbar_expect_tx(bar(PB_QFULL), kStage);
                    const int qrow = (int)(it.qi * H + (int64_t)it.hg * kTcHeads);
#pragma unroll
                    for (int r = 0; r < kRegions; r++)
                        tma_tile2d(sb + OFF_Q + r * kReg, &map_q, r * 64, qrow, bar(PB_QFULL), once);
                }
                // tile g of the CTA goes to stage g & 1 once P V of tile g - 2 has released it;
                // selected entries are gathered by warps 6-7, this thread only arrives for them
                for (int tt = 0; okw && tt < it.T; tt++) {
                    const int s = (int)(g & 1u);
                    if (g >= 2 && !mbar_wait(bar(PB_KFREE + s), ((g - 2) >> 1) & 1u)) {
                        okw = 0;
                        break;
                    }
                    const uint32_t stage = sb + OFF_K + s * kStage;
                    const uint32_t fb = bar(PB_KFULL + s);
                    mbar_expect_tx(fb, (GATHER && tt < it.T_main) ? 0u : kStage);
                    if (tt < it.T_main) {
                        if (!GATHER) {
                            const int row = (int)(it.e0 + (int64_t)tt * kTcKeys);
#pragma unroll
                            for (int r = 0; r < kRegions; r++)
                                tma_tile2d(stage + r * kReg, &map_ent_rows, r * 64, row, fb, keep);
                        }
                    } else {
                        const int row = (int)(it.tail_row0 + (int64_t)(tt - it.T_main) * kTcKeys);
#pragma unroll
                        for (int r = 0; r < kRegions; r++) tma_tile2d(stage + r * kReg, &map_kv, r * 64, row, fb, once);
                    }
                    g++;
                }
            }
            g = __shfl_sync(0xffffffffu, g, 0);
            ri++;
            if (!__shfl_sync(0xffffffffu, okw, 0)) {
                ok = false;
                break;
            }
            if (!ahead && !publish(k + 1, nxt)) ok = false;
        }
        if (lane == 0) {
            if (!ok) set_error(err, CSA_ERR_TIMEOUT);
            // no load may still be landing when the CTA ends: the last phase of
            // each stage and of the query tile
            for (int64_t u = (int64_t)g - 1; u >= 0 && u >= (int64_t)g - 2; u--)
                if (!mbar_wait(bar(PB_KFULL + (int)(u & 1)), (uint32_t)((u >> 1) & 1))) set_error(err, CSA_ERR_TIMEOUT);
            if (ri > 0 && !mbar_wait(bar(PB_QFULL), (ri - 1) & 1u)) set_error(err, CSA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == 6 || warp == 7) {
        // ------------------------------------------------------------ selection indices, cp.async gathers
        // Thread pt copies 16-byte chunk pt % 8 of rows pt / 8, + 8, ... in
        // every region of selected-entry tiles; every thread arrives on each
        // tile's KFULL (after its own copies landed), whatever the tile.
        const int pt = tid - kGatherBase;
        const int pc = pt & 7, pk0 = pt >> 3;
        constexpr int RSTEP = kTcpGatherThreads / 8;              // 8 rows per pass
        constexpr int KPP = (kTcKeys + RSTEP - 1) / RSTEP;        // 8 rows per thread
        const uint64_t keep = policy_evict_last();
        bool fail = false;
        bool pre = false;   // the indices of item ri were copied during item ri - 1
        uint32_t g = 0, ri = 0;
        for (uint32_t k = 0;; k++) {
            TcItem it;
            if (!item_at(k, it)) fail = true;
            if (tc::named_bar_or(2, kTcpGatherThreads, fail)) break;   // every gatherer leaves together
            if (pt == 0) mbar_arrive(bar(PB_IFREE + (int)(k % kTcpRing)));   // all have read the record
            if (it.T < 0) break;
            if (it.T == 0) continue;
            const int buf = (int)(ri % kTcpIdxBufs);
            int32_t *s_idx = s_idx0 + buf * kTcpIdxCap;
            if (GATHER) {
                if (pre) {
                    cp_async_wait<0>();   // this thread's copies of the indices
                } else {
                    // this buffer was last read by the softmax of item ri - 3
                    if (ri >= kTcpIdxBufs &&
                        !mbar_wait(bar(PB_IDXFREE + buf), ((ri - kTcpIdxBufs) / kTcpIdxBufs) & 1u))
                        fail = true;
                    if (tc::named_bar_or(2, kTcpGatherThreads, fail)) break;
                    for (int i = pt; i < it.n_main; i += kTcpGatherThreads) s_idx[i] = __ldg(idx + it.qi * top_k + i);
                }
                tc::named_bar(2, kTcpGatherThreads);
                mbar_arrive(bar(PB_IDXFULL + buf));
                // The next record, if it is out and has tiles, is item ri + 1: copy its
                // indices into their buffer (last read by the softmax of item ri - 2)
                // while this item's tiles are gathered.
                pre = false;
                const bool out = tc::named_bar_or(2, kTcpGatherThreads,
                                                  mbar_test(bar(PB_IFULL + (int)((k + 1) % kTcpRing)), ((k + 1) / kTcpRing) & 1u));
                if (out) {
                    TcItem nx;
                    if (!item_at(k + 1, nx)) fail = true;   // complete: returns at once
                    const uint32_t rn = ri + 1;
                    const int bn = (int)(rn % kTcpIdxBufs);
                    if (!fail && nx.T > 0 && rn >= kTcpIdxBufs &&
                        !mbar_wait(bar(PB_IDXFREE + bn), ((rn - kTcpIdxBufs) / kTcpIdxBufs) & 1u))
                        fail = true;
                    pre = !tc::named_bar_or(2, kTcpGatherThreads, fail) && nx.T > 0;
                    if (pre) {
                        int32_t *s_nx = s_idx0 + bn * kTcpIdxCap;
                        for (int i = pt; i < nx.n_main; i += kTcpGatherThreads)
                            cp_async_4(smem_u32(s_nx + i), idx + nx.qi * top_k + i);
                        cp_async_commit();
                    }
                }
            }
            for (int tt = 0; tt < it.T && !fail; tt++, g++) {
                const int s = (int)(g & 1u);
                if (g >= 2 && !mbar_wait(bar(PB_KFREE + s), ((g - 2) >> 1) & 1u)) {
                    fail = true;
                    break;
                }
                if (GATHER && tt < it.T_main) {
                    const uint32_t stage = sb + OFF_K + s * kStage;
#pragma unroll
                    for (int i = 0; i < KPP; i++) {
                        const int kr = pk0 + RSTEP * i;
                        if (kr < kTcKeys) {
                            const int slot = tt * kTcKeys + kr;
                            const int e = slot < it.n_main ? s_idx[slot] : -1;
                            const bool v = e >= 0 && (int64_t)e < it.n_vis;
                            const uint16_t *src = entries + (it.e0 + (v ? e : 0)) * kTcD;
                            cp_async_16_regions(stage + kr * 128 + ((pc ^ (kr & 7)) << 4), src + pc * 8, v ? 16 : 0, keep);
                        }
                    }
                    cp_async_commit();
                    cp_async_wait<0>();
                    tc::fence_proxy_async();
                }
                mbar_arrive(bar(PB_KFULL + s));
            }
            ri++;
        }
        cp_async_wait<0>();
        if (fail && pt == 0) set_error(err, CSA_ERR_TIMEOUT);
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        // S(t) and PV(t) are each issued in tile order (numbered across items);
        // the issuer polls both and issues whichever is ready first.  The first
        // S of an item waits for its query tile, the first PV for the previous
        // epilogue; the last S of an item frees the query tile, the last PV
        // completes the item's O^T.
        if (lane == 0) {
            constexpr uint32_t id_qk = tc::idesc_bf16_f32(64, kTcHeads, false, false);
            constexpr uint32_t id_pv = tc::idesc_bf16_f32(128, kTcHeads, true, true);
            const uint64_t qa0 = tc::sdesc_sw128(sb + OFF_K, 16, 1024);
            const uint64_t qb0 = tc::sdesc_sw128(sb + OFF_Q, 16, 1024);
            const uint64_t pa0 = tc::sdesc_sw128(sb + OFF_K, kReg, 1024);
            const uint64_t pb0 = tc::sdesc_sw128(sb + OFF_P, kReg, 1024);
            bool ok = true;
            uint32_t kS = 0, kP = 0;        // next ring record of each side
            uint32_t riS = 0, riP = 0;      // items with tiles begun by each side
            uint32_t nq = 0, np = 0;        // next S tile, next PV tile
            uint32_t startS = 0, endS = 0, startP = 0, endP = 0;   // tiles of the current item of each side
            bool hS = false, hP = false, doneS = false, doneP = false;
            uint64_t idle0 = global_ns();
            while (ok) {
                bool did = false;
                while (!hS && !doneS && mbar_test(bar(PB_IFULL + (int)(kS % kTcpRing)), (kS / kTcpRing) & 1u)) {
                    const int T = ring[kS % kTcpRing].T;
                    kS++;
                    if (T < 0) doneS = true;
                    else if (T > 0) {
                        hS = true;
                        startS = nq;
                        endS = nq + (uint32_t)T;
                    }
                }
                while (!hP && !doneP && mbar_test(bar(PB_IFULL + (int)(kP % kTcpRing)), (kP / kTcpRing) & 1u)) {
                    const int T = ring[kP % kTcpRing].T;
                    mbar_arrive(bar(PB_IFREE + (int)(kP % kTcpRing)));   // this side reads the record last
                    kP++;
                    if (T < 0) doneP = true;
                    else if (T > 0) {
                        hP = true;
                        startP = np;
                        endP = np + (uint32_t)T;
                    }
                }
                if (doneS && doneP) break;   // every product issued
                if (hS && nq <= np + 1) {
                    const int sidx = (int)(nq & 1u);
                    bool ready = (nq < 2 || mbar_test(bar(PB_SFREE + sidx), ((nq - 2) >> 1) & 1u)) &&
                                 mbar_test(bar(PB_KFULL + sidx), (nq >> 1) & 1u);
                    if (ready && nq == startS) ready = mbar_test(bar(PB_QFULL), riS & 1u);   // the item's query tile
                    if (ready) {
                        tc::fence_after_sync();
                        // descriptors advance by adding (byte offset >> 4) to the address field
                        const uint64_t a0 = qa0 + (uint64_t)((sidx * kStage) >> 4);
                        const uint32_t dS = tmem + TM_S + 64 * sidx;
#pragma unroll
                        for (int j = 0; j < kTcD / 16; j++) {
                            const uint64_t off = (uint64_t)(((j >> 2) * kReg + (j & 3) * 32) >> 4);
                            tc::mma_ss(dS, a0 + off, qb0 + off, id_qk, j != 0);
                        }
                        tc::mma_commit(bar(PB_SFULL + sidx));
                        nq++;
                        if (nq == endS) {   // the item's last S^T: the query tile is free once it completes
                            tc::mma_commit(bar(PB_QFREE));
                            riS++;
                            hS = false;
                        }
                        did = true;
                    }
                }
                if (hP && np < nq) {
                    const int sidx = (int)(np & 1u);
                    const bool first = np == startP;
                    bool ready = mbar_test(bar(PB_PFULL + sidx), (np >> 1) & 1u);
                    if (ready && first && riP > 0) ready = mbar_test(bar(PB_OFREE), (riP - 1) & 1u);
                    if (ready) {
                        tc::fence_after_sync();
                        const uint64_t a0 = pa0 + (uint64_t)((sidx * kStage) >> 4);
                        const uint64_t b0 = pb0 + (uint64_t)((sidx * kReg) >> 4);
#pragma unroll
                        for (int m = 0; m < 4; m++)
#pragma unroll
                            for (int k4 = 0; k4 < kTcKeys / 16; k4++)
                                tc::mma_ss(tmem + TM_O + 64 * m, a0 + (uint64_t)((2 * m * kReg + k4 * 2048) >> 4),
                                           b0 + (uint64_t)((k4 * 2048) >> 4), id_pv, !first || k4 > 0);
                        tc::mma_commit(bar(PB_KFREE + sidx));
                        np++;
                        if (np == endP) {   // the item's last P V: its O^T is complete once it completes
                            tc::mma_commit(bar(PB_OFULL));
                            riP++;
                            hP = false;
                        }
                        did = true;
                    }
                }
                if (did) {
                    idle0 = global_ns();
                } else {
                    // back off briefly: this warp shares its scheduler with a softmax warp
                    __nanosleep(20);
                    if (global_ns() - idle0 > kWaitLimitNs) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) set_error(err, CSA_ERR_TIMEOUT);
            // every issued product completes before the CTA ends
            tc::mma_commit(bar(PB_FIN));
            if (!mbar_wait(bar(PB_FIN), 0)) set_error(err, CSA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp >= 8) {
        // ------------------------------------------------------------ epilogue (warps 8-11)
        // Warp w reads lanes 32 (w % 4) .. + 31 of O^T (rows d = 128 m + 32 (w % 4) + lane)
        // once the item's last P V is done and the softmax has handed over each
        // head's (max, sum); O / l -> out[head][d] (bf16), two neighbouring d of
        // one head per store, and the log-sum-exp.
        const int et = tid - kTcpEpiBase;
        const int quarter = warp & 3;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        bool fail = false;
        uint32_t ri = 0;
        for (uint32_t k = 0;; k++) {
            TcItem it;
            if (!item_at(k, it)) fail = true;
            if (tc::named_bar_or(3, 128, fail)) break;   // every epilogue thread leaves together
            if (et == 0) mbar_arrive(bar(PB_IFREE + (int)(k % kTcpRing)));   // all have read the record
            if (it.T < 0) break;
            if (it.T == 0) continue;
            const int buf = (int)(ri & 1u);
            const float *lb = reinterpret_cast<const float *>(sm + OFF_LBUF) + buf * 3 * kTcHeads;
            if (!mbar_wait(bar(PB_OFULL), ri & 1u)) fail = true;
            if (!mbar_wait(bar(PB_LFULL + buf), (ri >> 1) & 1u)) fail = true;
            if (tc::named_bar_or(3, 128, fail)) break;
            tc::fence_after_sync();
            const int64_t row0 = it.qi * H + (int64_t)it.hg * kTcHeads;
#pragma unroll 1
            for (int c = 0; c < 8; c++) {
                float o[32];
                tc::tmem_ld32(tmem + lane_base + TM_O + 32 * c, o);
                tc::tmem_wait_ld();
                if (c == 7) {   // O^T is read: the next item's first P V may overwrite it
                    tc::fence_before_sync();
                    mbar_arrive(bar(PB_OFREE));
                }
                const int d = 128 * (c >> 1) + 32 * quarter + lane;   // this thread's row of O^T
                const int h0 = 32 * (c & 1);
                // lanes 2i and 2i+1 hold d and d+1: the even lane stores (d, d+1) of
                // head h0 + j, the odd lane those of head h0 + j + 1
                const bool odd = lane & 1;
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float a = o[j] * lb[2 * kTcHeads + h0 + j], b = o[j + 1] * lb[2 * kTcHeads + h0 + j + 1];
                    const float got = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
                    const uint32_t pk = odd ? pack_bf16x2(got, b) : pack_bf16x2(a, got);
                    const int h = h0 + j + (odd ? 1 : 0);
                    *reinterpret_cast<uint32_t *>(out + (row0 + h) * kTcD + (d & ~1)) = pk;
                }
            }
            if (lse && et < kTcHeads) lse[row0 + et] = (lb[et] + log2f(lb[kTcHeads + et])) * kTcLn2;
            mbar_arrive(bar(PB_LFREE + buf));   // this thread reads the buffer no more
            ri++;
        }
        if (fail && et == 0) set_error(err, CSA_ERR_TIMEOUT);
    } else {
        // ------------------------------------------------------------ softmax (128 threads)
        // As in attend_tc_kernel, per item: thread (w, l) takes key 16 w + l % 16
        // of each tile for heads 32 hh .. 32 hh + 31, keeps the running maxima in
        // registers and its partial sums, reduced once after the item's last tile.
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int hh = lane >> 4;                 // head half: heads 32 hh .. 32 hh + 31
        const int key = 16 * warp + (lane & 15);  // key of the tile this thread takes
        bool fail = false;   // a wait of this thread gave up (acted on at the next barrier reduction)
        uint32_t g = 0, ri = 0;
        for (uint32_t k = 0;; k++) {
            TcItem it;
            if (!item_at(k, it)) fail = true;
            if (tc::named_bar_or(1, 128, fail)) break;   // every softmax thread leaves together
            if (tid == 0) mbar_arrive(bar(PB_IFREE + (int)(k % kTcpRing)));   // all have read the record
            if (it.T < 0) break;
            if (it.T == 0) continue;
            const int ibuf = (int)(ri % kTcpIdxBufs);
            const int32_t *s_idx = s_idx0 + ibuf * kTcpIdxCap;
            if (GATHER && !mbar_wait(bar(PB_IDXFULL + ibuf), (ri / kTcpIdxBufs) & 1u)) fail = true;
            float m_run[32], l_part[32];
#pragma unroll
            for (int j = 0; j < 32; j++) {
                m_run[j] = -INFINITY;
                l_part[j] = 0.f;
            }
            if (tid < kTcHeads) s_m[tid] = -INFINITY;   // read by the others after a barrier
            for (int t = 0; t < it.T; t++, g++) {
                const int sidx = (int)(g & 1u);
                if (!mbar_wait(bar(PB_SFULL + sidx), (g >> 1) & 1u)) fail = true;
                tc::fence_after_sync();
                float v[64];
                tc::tmem_ld32(tmem + lane_base + TM_S + 64 * sidx, v);
                tc::tmem_ld32(tmem + lane_base + TM_S + 64 * sidx + 32, v + 32);
                tc::tmem_wait_ld();
                tc::fence_before_sync();
                mbar_arrive(bar(PB_SFREE + sidx));
                // lanes 0-15 hold the tile's rows: hand heads 32-63 to lanes 16-31
                float sc[32];
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    const float other = __shfl_xor_sync(0xffffffffu, v[32 + j], 16);
                    sc[j] = hh ? other : v[j];
                }
                bool valid;
                if (t < it.T_main) {
                    const int slot = t * kTcKeys + key;
                    valid = slot < it.n_main;
                    if (GATHER && valid) {
                        const int e = s_idx[slot];
                        valid = e >= 0 && (int64_t)e < it.n_vis;
                        if (e >= 0 && !valid) set_error(err, CSA_ERR_DEVICE);   // an index that is not visible
                    }
                } else {
                    valid = (t - it.T_main) * kTcKeys + key < it.r_tail;
                }
                bool exceed = false;
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    sc[j] = valid ? sc[j] * scale_log2 : -INFINITY;
                    exceed |= sc[j] > m_run[j] + kRescaleLog2;   // a finite score always exceeds -inf
                }
                bool rescale = false;
                if (tc::named_bar_or(1, 128, exceed || fail)) {
                    if (tc::named_bar_or(1, 128, fail)) break;   // a wait gave up: every thread leaves together
                    float r0, r1;
                    halfwarp_reduce32<true>(sc, r0, r1);
                    const int h2 = 32 * hh + 2 * (lane & 15);
                    s_rmax[warp * 64 + h2] = r0;
                    s_rmax[warp * 64 + h2 + 1] = r1;
                    if (tid == 0) s_flag[1] = 0;
                    tc::named_bar(1, 128);
                    if (tid < kTcHeads) {
                        const float M = fmaxf(fmaxf(s_rmax[tid], s_rmax[64 + tid]), fmaxf(s_rmax[128 + tid], s_rmax[192 + tid]));
                        const float m_old = s_m[tid];
                        float m_new = m_old, alpha = 1.f;
                        if (M > m_old + kRescaleLog2 || (m_old == -INFINITY && M != -INFINITY)) {
                            m_new = M;
                            alpha = fast_exp2(m_old - m_new);   // 0 when nothing was accumulated yet
                            if (t > 0) s_flag[1] = 1;
                        }
                        s_m[tid] = m_new;
                        s_al[tid] = alpha;
                    }
                    tc::named_bar(1, 128);
                    rescale = s_flag[1] != 0;
#pragma unroll
                    for (int j = 0; j < 32; j++) {
                        m_run[j] = s_m[32 * hh + j];
                        l_part[j] *= s_al[32 * hh + j];
                    }
                }
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    sc[j] = (m_run[j] == -INFINITY) ? 0.f : fast_exp2_ftz(sc[j] - m_run[j]);
                    l_part[j] += sc[j];
                }
                // This P stage was last read by P V of tile g - 2, which must be done.
                // A rescale of the O^T columns also needs P V of tile g - 1 (of this item) done.
                if (rescale ? (t >= 1 && !mbar_wait(bar(PB_KFREE + (int)((g - 1) & 1u)), ((g - 1) >> 1) & 1u))
                            : (g >= 2 && !mbar_wait(bar(PB_KFREE + sidx), ((g - 2) >> 1) & 1u)))
                    fail = true;
                {
                    uint8_t *prow = sm + OFF_P + sidx * kReg + key * 128;
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const int ch = 4 * hh + c;
                        uint4 w;
                        w.x = pack_bf16x2(sc[8 * c + 0], sc[8 * c + 1]);
                        w.y = pack_bf16x2(sc[8 * c + 2], sc[8 * c + 3]);
                        w.z = pack_bf16x2(sc[8 * c + 4], sc[8 * c + 5]);
                        w.w = pack_bf16x2(sc[8 * c + 6], sc[8 * c + 7]);
                        *reinterpret_cast<uint4 *>(prow + ((ch ^ (key & 7)) << 4)) = w;
                    }
                }
                if (rescale) {
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < 8; c++) {
                        float o[32];
                        const uint32_t ta = tmem + lane_base + TM_O + 32 * c;
                        tc::tmem_ld32(ta, o);
                        tc::tmem_wait_ld();
                        const float *al = s_al + 32 * (c & 1);
#pragma unroll
                        for (int j = 0; j < 32; j++) o[j] *= al[j];
                        tc::tmem_st32(ta, o);
                    }
                    tc::tmem_wait_st();
                }
                tc::fence_proxy_async();
                tc::fence_before_sync();
                mbar_arrive(bar(PB_PFULL + sidx));
            }
            if (GATHER) mbar_arrive(bar(PB_IDXFREE + ibuf));   // this thread reads the indices no more
            // the weights' sums over keys, once: lanes (keys) within each warp, then the warps
            if (tc::named_bar_or(1, 128, fail)) break;
            {
                float r0, r1;
                halfwarp_reduce32<false>(l_part, r0, r1);
                const int h2 = 32 * hh + 2 * (lane & 15);
                s_rsum[warp * 64 + h2] = r0;
                s_rsum[warp * 64 + h2 + 1] = r1;
            }
            tc::named_bar(1, 128);
            // hand the item's (max, sum) of each head to the epilogue warps; this
            // buffer was last read by the epilogue of item ri - 2
            const int buf = (int)(ri & 1u);
            float *lb = reinterpret_cast<float *>(sm + OFF_LBUF) + buf * 3 * kTcHeads;
            if (ri >= 2 && !mbar_wait(bar(PB_LFREE + buf), ((ri - 2) >> 1) & 1u)) fail = true;
            if (tid < kTcHeads) {
                const float l = s_rsum[tid] + s_rsum[64 + tid] + s_rsum[128 + tid] + s_rsum[192 + tid];
                lb[tid] = s_m[tid];
                lb[kTcHeads + tid] = l;
                lb[2 * kTcHeads + tid] = l > 0.f ? 1.f / l : 0.f;
            }
            mbar_arrive(bar(PB_LFULL + buf));
            ri++;
        }
        if (fail && tid == 0) set_error(err, CSA_ERR_TIMEOUT);
    }
    tc::fence_before_sync();
    __syncthreads();
    griddep_launch();
    tc::fence_after_sync();
    if (warp == 4) tc::tmem_dealloc(tmem, kTmemCols);
    // the last CTA to finish returns the counters to zero for the next call
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(counters + 1, 1u) == gridDim.x - 1) {
            counters[0] = 0u;
            counters[1] = 0u;
        }
    }
}

// Key splits.  With fewer 64-head units than `share` SMs, a unit's tiles are
// spread over as many CTAs as keep the grid within one wave of `share` CTAs.
struct TcPlan {
    int nsplit_max;   // splits of a query with at least that many key tiles
    bool persist;     // one split per query: the persistent kernel, one CTA per SM
};

TcPlan tc_plan(const AttendArgs &a)
{
    const int share = a.sm_share > 0 ? a.sm_share : (a.num_sms > 0 ? a.num_sms : 148);
    const int64_t units = a.total_q * (a.n_heads / kTcHeads);
    const int64_t max_vis = a.max_kv_len / a.ratio;
    int64_t mk = (a.top_k > 0 && max_vis > a.top_k ? a.top_k : max_vis) + (a.ratio - 1);
    if (mk > a.max_kv_len) mk = a.max_kv_len;   // the tail never exceeds the sequence
    if (mk < 1) mk = 1;
    const int64_t tiles = (mk + kTcKeys - 1) / kTcKeys;
    int64_t want = units >= share ? 1 : share / units;
    if (want > tiles) want = tiles;
    if (want > 64) want = 64;   // the merge reads at most 64 splits
    if (want < 1) want = 1;
    TcPlan pl;
    pl.nsplit_max = (int)want;
    pl.persist = want == 1 && units >= share && (a.idx == nullptr || a.top_k <= kTcpIdxCap);
    return pl;
}

size_t tc_ws_bytes(const AttendArgs &a, const TcPlan &pl, float **part_o, float2 **part_ml)
{
    if (pl.persist) {   // the item counters
        if (part_o) *part_o = nullptr;
        if (part_ml) *part_ml = nullptr;
        return kTcpHeader;
    }
    if (pl.nsplit_max <= 1) {
        if (part_o) *part_o = nullptr;
        if (part_ml) *part_ml = nullptr;
        return 0;
    }
    const size_t slots = (size_t)a.total_q * (a.n_heads / kTcHeads) * pl.nsplit_max * kTcHeads;
    const size_t ml = (slots * sizeof(float2) + 255) / 256 * 256;
    if (part_ml) *part_ml = reinterpret_cast<float2 *>(a.ws);
    if (part_o) *part_o = reinterpret_cast<float *>(static_cast<char *>(a.ws) + ml);
    return ml + slots * kTcD * sizeof(float);
}

// A [rows, 512] bf16 row-major matrix as a TMA source: boxes of 64 columns
// (128 bytes, swizzled) by box_rows rows.
cudaError_t rows_map(CUtensorMap *m, const void *base, int64_t rows, uint32_t box_rows)
{
    return tma_map_bf16(m, base, rows, kTcD, 64, box_rows);
}

template <bool GATHER>
cudaError_t launch_tc(const AttendArgs &a, cudaStream_t st)
{
    const TcPlan pl = tc_plan(a);
    float *part_o = nullptr;
    float2 *part_ml = nullptr;
    tc_ws_bytes(a, pl, &part_o, &part_ml);
    const int HG = a.n_heads / kTcHeads;
    if ((int64_t)HG * pl.nsplit_max > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)a.total_q, (unsigned)(HG * pl.nsplit_max));
    const float scale_log2 = a.scale * 1.4426950408889634f;
    // Tensor maps: the query rows [total_q * H, 512], the entries and the raw
    // KV rows, each in 64-row tiles.  With no entries at all the entry map
    // points at the KV rows; no tile reads it then.
    CUtensorMap m_q, m_ent_rows, m_kv;
    const bool have_ent = a.entries != nullptr && a.n_ent_rows > 0;
    const void *ent = have_ent ? (const void *)a.entries : (const void *)a.kv;
    const int64_t ent_rows = have_ent ? a.n_ent_rows : a.n_kv_rows;
    cudaError_t e = rows_map(&m_q, a.q, a.total_q * a.n_heads, 64);
    if (e == cudaSuccess) e = rows_map(&m_ent_rows, ent, ent_rows, 64);
    if (e == cudaSuccess) e = rows_map(&m_kv, a.kv, a.n_kv_rows, 64);
    if (e != cudaSuccess) return e;
    if (pl.persist) {
        // the counters start at zero whatever an earlier call left; the last CTA zeroes them again
        if (!a.ws || a.ws_bytes < kTcpHeader) return cudaErrorInvalidValue;
        unsigned *counters = static_cast<unsigned *>(a.ws);
        e = cudaMemsetAsync(counters, 0, 2 * sizeof(unsigned), st);
        if (e != cudaSuccess) return e;
        const int64_t n_items = a.total_q * HG;
        const int sms = a.num_sms > 0 ? a.num_sms : 148;
        const unsigned pgrid = (unsigned)(n_items < sms ? n_items : sms);
        return launch_kernel(GATHER ? "sparse_attend" : "dense_attend", attend_tcp_kernel<GATHER>, dim3(pgrid),
                             dim3(kTcThreads), kTcpSmem, st, a.pdl, m_q, m_ent_rows, m_kv, a.batch, a.cu_kv, a.cu_q,
                             a.cu_ent, static_cast<const uint16_t *>(ent), a.idx, a.n_heads, a.ratio, a.top_k,
                             scale_log2, a.max_kv_len, n_items, counters, a.out, a.lse, a.err);
    }
    e = launch_kernel(GATHER ? "sparse_attend" : "dense_attend", attend_tc_kernel<GATHER>, grid, dim3(kTcThreads),
                      kTcSmem, st, a.pdl, m_q, m_ent_rows, m_kv, a.batch, a.cu_kv, a.cu_q, a.cu_ent,
                      static_cast<const uint16_t *>(ent), a.idx, a.n_heads, a.ratio, a.top_k, scale_log2, a.max_kv_len, pl.nsplit_max, a.out, a.lse,
                      part_o, part_ml, a.err);
    if (e != cudaSuccess || pl.nsplit_max <= 1) return e;
    // The merge overlaps the attention's tail only on a dependent-launch chain
    // (a.pdl); otherwise its many small CTAs, launched early, would wait on
    // SMs that other work on the GPU needs.
    const dim3 mgrid((unsigned)a.total_q, (unsigned)a.n_heads);
    return launch_kernel(GATHER ? "sparse_merge" : "dense_merge", attend_tc_merge_kernel<GATHER>, mgrid,
                         dim3(kMergeThreads), 0, st, a.pdl, a.batch, a.cu_kv, a.cu_q, a.cu_ent, a.n_heads,
                         a.ratio, a.top_k, pl.nsplit_max, (const float *)part_o, (const float2 *)part_ml,
                         a.out, a.lse);
}

}  // namespace

bool attend_tc_applicable(const AttendArgs &a)
{
    // row coordinates of the TMA loads are 32-bit
    return a.d == kTcD && a.n_heads % kTcHeads == 0 && (a.idx == nullptr || a.top_k <= kTcIdxCap) &&
           a.total_q * a.n_heads < 0x7fffffffLL && a.n_kv_rows < 0x7fffffffLL && a.n_ent_rows < 0x7fffffffLL &&
           tma_available();
}

size_t attend_tc_workspace_bytes(const AttendArgs &a) { return tc_ws_bytes(a, tc_plan(a), nullptr, nullptr); }

cudaError_t launch_attend_tc(const AttendArgs &a, cudaStream_t st)
{
    if (a.total_q <= 0) return cudaSuccess;
    return a.idx ? launch_tc<true>(a, st) : launch_tc<false>(a, st);
}

// ---- TMA descriptors (declared in tma.h) ----
namespace {
// cuTensorMapEncodeTiled from the driver (looked up once).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}
}  // namespace

bool tma_available() { return encode_fn() != nullptr; }

cudaError_t tma_map_bf16(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, uint32_t box_cols,
                         uint32_t box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 f = encode_fn();
    if (!f) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace csa
