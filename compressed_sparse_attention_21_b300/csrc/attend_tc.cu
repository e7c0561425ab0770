// Shared-KV multi-query attention on the fifth-generation tensor cores
// (tcgen05, accumulators in tensor memory) for prefill-sized batches with
// d = 512 ("DeepSeek-V4 core architecture", §2.2 CSA step 3: each selected
// entry is both key and value, shared by all query heads; §2.3 HCA: dense
// attention over every compressed entry).  The key set of a query is the
// same as in attend.cu: selected (or all visible) entries plus the raw
// tokens of the query's own open block.
//
// One CTA computes 64 heads of one query over all of its keys, 128 keys per
// tile.  Keys are the M dimension of both products, so that every tensor-
// memory accumulator keeps the 128-lane layout (lane = row):
//     S^T[key, head] = K[key, :] . Q[head, :]       M = 128 keys, N = 64, K = 512
//     O^T[d, head]  += K[key, d]^T . P^T[key, head]  M = 4 x 128 d,   N = 64, K = 128
// The same shared-memory key tile is the K-major A operand of the first
// product and the MN-major A operand of the second; P is stored key-major
// (one 128-byte row of 64 heads per key) as the MN-major B operand.  S^T takes 64 tensor-
// memory columns and O^T 256.
//
// Warp roles (256 threads): warps 0-3 run the softmax (thread i owns key i
// of the tile, then row d = 128 m + i of the output), warp 4 lane 0 issues
// the MMAs, warps 5-7 gather key rows into the swizzled tile with cp.async.
// The tile is split in eight 64-column regions with their own barriers, so
// the next tile's regions reload as soon as the products reading them are
// done.  The running maximum of a head is raised only when a tile exceeds it
// by more than 2^8 (then the accumulated O^T column and sum are rescaled);
// the result is exact either way because the sum uses the same maximum.
// Every wait is bounded: one that runs out reports CSA_ERR_TIMEOUT.
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace csa {

namespace {

constexpr int kTcThreads = 256;
constexpr int kTcKeys = 128;                 // keys per tile (M)
constexpr int kTcHeads = 64;                 // heads per CTA (N)
constexpr int kTcD = 512;
constexpr int kRegions = kTcD / 64;          // 64-column regions of a 128-byte swizzled row
constexpr int kProd = 96;                    // producer threads (warps 5-7)
constexpr int kProdBase = 160;
constexpr uint32_t kRegK = kTcKeys * 128;    // 16 KiB per key region
constexpr uint32_t kRegQ = kTcHeads * 128;   // 8 KiB per query region
constexpr int kTcIdxCap = 2048;
constexpr float kTcLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;         // raise a head's maximum only beyond 2^8

constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + kRegions * kRegQ;      // 64 KiB
constexpr uint32_t OFF_P = OFF_K + kRegions * kRegK;      // + 128 KiB
constexpr uint32_t OFF_BAR = OFF_P + 2 * kRegQ;           // + 16 KiB
constexpr int BAR_KFULL = 0, BAR_KFREE = 8, BAR_SFULL = 12, BAR_SFREE = 13, BAR_PFULL = 14, BAR_OFULL = 15;
constexpr uint32_t OFF_MISC = OFF_BAR + 16 * 8;
// misc: tmem slot, flags, per-head m / l / new max / alpha, per-warp tile max and sum
constexpr uint32_t MISC_TMEM = 0, MISC_FLAG = 4, MISC_M = 16, MISC_L = MISC_M + 256, MISC_MN = MISC_L + 256,
                   MISC_AL = MISC_MN + 256, MISC_RMAX = MISC_AL + 256, MISC_RSUM = MISC_RMAX + 1024,
                   MISC_END = MISC_RSUM + 1024;
constexpr uint32_t OFF_IDX = OFF_MISC + MISC_END;
constexpr uint32_t kTcSmem = OFF_IDX + kTcIdxCap * 4 + 1024;   // + alignment slack
static_assert(kTcSmem <= 232448, "shared memory per CTA");

constexpr uint32_t TM_S = 0;     // S^T: columns 0..63
constexpr uint32_t TM_O = 64;    // O^T block m: columns 64 + 64 m .. +63
constexpr uint32_t kTmemCols = 512;

// Butterfly reduction of 64 values per lane over the 32 lanes of a warp: on
// return lane L holds the result for heads 2L and 2L+1 in r0, r1.
template <bool MAX>
__device__ __forceinline__ void warp_reduce64(const float *v, float &r0, float &r1)
{
    const int lane = threadIdx.x & 31;
    float a[32];
#pragma unroll
    for (int j = 0; j < 32; j++) {
        const bool up = lane & 16;
        const float keep = up ? v[32 + j] : v[j];
        const float send = up ? v[j] : v[32 + j];
        const float got = __shfl_xor_sync(0xffffffffu, send, 16);
        a[j] = MAX ? fmaxf(keep, got) : keep + got;
    }
#pragma unroll
    for (int o = 8, half = 16; o >= 1; o >>= 1, half >>= 1) {
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

struct TcKeys {
    const uint16_t *entries;   // the sequence's first entry row
    const uint16_t *tail;      // first raw tail row
    const int32_t *idx;        // sparse: the query's selection (shared or global memory)
    int64_t n_vis;
    int n_main, n_keys;
};

template <bool GATHER>
__device__ __forceinline__ const uint16_t *tc_key_row(const TcKeys &ks, int slot)
{
    if (slot < ks.n_main) {
        if (GATHER) {
            const int e = ks.idx[slot];
            if (e < 0 || (int64_t)e >= ks.n_vis) return nullptr;
            return ks.entries + (int64_t)e * kTcD;
        }
        return ks.entries + (int64_t)slot * kTcD;
    }
    if (slot < ks.n_keys) return ks.tail + (int64_t)(slot - ks.n_main) * kTcD;
    return nullptr;
}

template <bool GATHER>
__global__ void __launch_bounds__(kTcThreads, 1)
attend_tc_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                 const int64_t *__restrict__ cu_ent, const uint16_t *__restrict__ q,
                 const uint16_t *__restrict__ entries, const uint16_t *__restrict__ kv,
                 const int32_t *__restrict__ idx, int H, int ratio, int top_k, float scale_log2, int max_kv_len,
                 uint16_t *__restrict__ out, float *__restrict__ lse, int *err)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;          // swizzled tiles need 1024-byte alignment
    uint8_t *sm = smem_raw + (sb - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t qi = blockIdx.x;
    const int hg = blockIdx.y;

    const QueryPos p = query_pos(cu_kv, cu_q, cu_ent, batch, qi);
    const int64_t n_vis = (p.t + 1) / ratio;
    const int r_tail = (int)((p.t + 1) % ratio);
    const bool bad = p.t < 0 || p.t >= p.L || p.L > max_kv_len ||
                     p.ne != p.L / ratio;
    if (bad) {
        if (tid == 0) set_error(err, CSA_ERR_DEVICE);
        return;
    }
    TcKeys ks;
    ks.entries = entries + p.e0 * kTcD;
    ks.tail = kv + (p.kv0 + p.t - r_tail + 1) * kTcD;
    ks.idx = GATHER ? idx + qi * top_k : nullptr;
    ks.n_vis = n_vis;
    ks.n_main = GATHER ? (int)(n_vis < top_k ? n_vis : top_k) : (int)n_vis;
    ks.n_keys = ks.n_main + r_tail;
    const int T = (ks.n_keys + kTcKeys - 1) / kTcKeys;

    const uint32_t bar0 = sb + OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint8_t *misc = sm + OFF_MISC;
    float *s_m = reinterpret_cast<float *>(misc + MISC_M);
    float *s_l = reinterpret_cast<float *>(misc + MISC_L);
    float *s_mn = reinterpret_cast<float *>(misc + MISC_MN);
    float *s_al = reinterpret_cast<float *>(misc + MISC_AL);
    float *s_rmax = reinterpret_cast<float *>(misc + MISC_RMAX);   // [4 warps][64 heads]
    float *s_rsum = reinterpret_cast<float *>(misc + MISC_RSUM);
    volatile int *s_flag = reinterpret_cast<volatile int *>(misc + MISC_FLAG);

    if (tid == 0) {
        for (int r = 0; r < kRegions; r++) mbar_init(bar(BAR_KFULL + r), kProd);
        for (int m = 0; m < 4; m++) mbar_init(bar(BAR_KFREE + m), 1);
        mbar_init(bar(BAR_SFULL), 1);
        mbar_init(bar(BAR_SFREE), 128);
        mbar_init(bar(BAR_PFULL), 128);
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

    // the selection and the entries come from earlier kernels
    griddep_wait();
    if (GATHER && ks.n_main <= kTcIdxCap) {
        int32_t *s_idx = reinterpret_cast<int32_t *>(sm + OFF_IDX);
        for (int i = tid; i < ks.n_main; i += kTcThreads) s_idx[i] = __ldg(ks.idx + i);
        ks.idx = s_idx;
    }
    __syncthreads();

    if (warp >= 5) {
        // ------------------------------------------------------------ producers
        // Thread pt copies chunk pc (16 bytes) of key rows pk0, pk0 + 12, ...:
        // a warp covers four whole 128-byte row segments per instruction.  The
        // row sources of a tile are looked up once; the eight regions are then
        // issued back to back and published in order as they land.
        const int pt = tid - kProdBase;
        const int pc = pt & 7, pk0 = pt >> 3;
        constexpr int RSTEP = kProd / 8;                          // 12 rows per pass
        constexpr int KPP = (kTcKeys + RSTEP - 1) / RSTEP;        // 11 rows per thread
        const uint16_t *qrow = q + (qi * H + (int64_t)hg * kTcHeads) * kTcD;
        bool ok = true;
        for (int t = 0; t < T && ok; t++) {
            const uint16_t *src[KPP];
#pragma unroll
            for (int i = 0; i < KPP; i++) {
                const int k = pk0 + RSTEP * i;
                src[i] = k < kTcKeys ? tc_key_row<GATHER>(ks, t * kTcKeys + k) : nullptr;
            }
#pragma unroll 1
            for (int r = 0; r < kRegions; r++) {
                if (t > 0 && (r & 1) == 0 && !mbar_wait(bar(BAR_KFREE + r / 2), (uint32_t)((t - 1) & 1))) {
                    set_error(err, CSA_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                if (t == 0)   // the Q region travels with the first tile's region
#pragma unroll
                    for (int i = 0; i < (kTcHeads + RSTEP - 1) / RSTEP; i++) {
                        const int h = pk0 + RSTEP * i;
                        if (h < kTcHeads)
                            cp_async_16(sb + OFF_Q + r * kRegQ + h * 128 + ((pc ^ (h & 7)) << 4),
                                        qrow + (int64_t)h * kTcD + r * 64 + pc * 8, 16);
                    }
#pragma unroll
                for (int i = 0; i < KPP; i++) {
                    const int k = pk0 + RSTEP * i;
                    if (k < kTcKeys)
                        cp_async_16(sb + OFF_K + r * kRegK + k * 128 + ((pc ^ (k & 7)) << 4),
                                    src[i] ? (const void *)(src[i] + r * 64 + pc * 8) : (const void *)kv,
                                    src[i] ? 16 : 0);
                }
                cp_async_commit();
            }
            if (!ok) break;
            // publish the regions in order as their copies complete
            cp_async_wait<7>(); tc::fence_proxy_async(); mbar_arrive(bar(BAR_KFULL + 0));
            cp_async_wait<6>(); tc::fence_proxy_async(); mbar_arrive(bar(BAR_KFULL + 1));
            cp_async_wait<5>(); tc::fence_proxy_async(); mbar_arrive(bar(BAR_KFULL + 2));
            cp_async_wait<4>(); tc::fence_proxy_async(); mbar_arrive(bar(BAR_KFULL + 3));
            cp_async_wait<3>(); tc::fence_proxy_async(); mbar_arrive(bar(BAR_KFULL + 4));
            cp_async_wait<2>(); tc::fence_proxy_async(); mbar_arrive(bar(BAR_KFULL + 5));
            cp_async_wait<1>(); tc::fence_proxy_async(); mbar_arrive(bar(BAR_KFULL + 6));
            cp_async_wait<0>(); tc::fence_proxy_async(); mbar_arrive(bar(BAR_KFULL + 7));
        }
        cp_async_wait<0>();
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = tc::idesc_bf16_f32(128, kTcHeads, false, false);
            constexpr uint32_t id_pv = tc::idesc_bf16_f32(128, kTcHeads, true, true);
            bool ok = true;
            for (int t = 0; t < T && ok; t++) {
                if (t > 0 && !mbar_wait(bar(BAR_SFREE), (uint32_t)((t - 1) & 1))) {
                    ok = false;
                    break;
                }
                for (int r = 0; r < kRegions && ok; r++) {
                    if (!mbar_wait(bar(BAR_KFULL + r), (uint32_t)(t & 1))) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
#pragma unroll
                    for (int ks4 = 0; ks4 < 4; ks4++) {
                        const uint64_t a = tc::sdesc_sw128(sb + OFF_K + r * kRegK + ks4 * 32, 16, 1024);
                        const uint64_t b = tc::sdesc_sw128(sb + OFF_Q + r * kRegQ + ks4 * 32, 16, 1024);
                        tc::mma_ss(tmem + TM_S, a, b, id_qk, (r | ks4) != 0);
                    }
                }
                if (!ok) break;
                tc::mma_commit(bar(BAR_SFULL));
                if (!mbar_wait(bar(BAR_PFULL), (uint32_t)(t & 1))) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
#pragma unroll 1
                for (int m = 0; m < 4; m++) {
#pragma unroll
                    for (int k8 = 0; k8 < 8; k8++) {
                        const uint64_t a = tc::sdesc_sw128(sb + OFF_K + 2 * m * kRegK + k8 * 2048, kRegK, 1024);
                        const uint64_t b = tc::sdesc_sw128(sb + OFF_P + k8 * 2048, kRegK, 1024);
                        tc::mma_ss(tmem + TM_O + 64 * m, a, b, id_pv, t > 0 || k8 > 0);
                    }
                    tc::mma_commit(bar(BAR_KFREE + m));
                }
            }
            if (!ok) set_error(err, CSA_ERR_TIMEOUT);
            // every issued product completes before the CTA ends
            tc::mma_commit(bar(BAR_OFULL));
            if (!mbar_wait(bar(BAR_OFULL), 0)) set_error(err, CSA_ERR_TIMEOUT);
            s_flag[2] = ok ? 1 : 0;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax (128 threads)
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        uint8_t *sP = sm + OFF_P;
        bool ok = true;
        for (int t = 0; t < T; t++) {
            if (tid == 0) s_flag[0] = mbar_wait(bar(BAR_SFULL), (uint32_t)(t & 1)) ? 1 : 0;
            tc::named_bar(1, 128);
            if (!s_flag[0]) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            float s[64];
            tc::tmem_ld32(tmem + lane_base + TM_S, s);
            tc::tmem_ld32(tmem + lane_base + TM_S + 32, s + 32);
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            mbar_arrive(bar(BAR_SFREE));

            const int slot = t * kTcKeys + tid;
            bool valid = slot < ks.n_keys;
            if (GATHER && valid && slot < ks.n_main) {
                const int e = ks.idx[slot];
                valid = e >= 0 && (int64_t)e < ks.n_vis;
            }
#pragma unroll
            for (int h = 0; h < 64; h++) s[h] = valid ? s[h] * scale_log2 : -INFINITY;
            float r0, r1;
            warp_reduce64<true>(s, r0, r1);
            s_rmax[warp * 64 + 2 * lane] = r0;
            s_rmax[warp * 64 + 2 * lane + 1] = r1;
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
                s_mn[tid] = m_new;
                s_al[tid] = alpha;
            }
            tc::named_bar(1, 128);
            if (s_flag[1]) {
                // O^T columns of the raised heads scale by alpha (the previous
                // tile's products are complete: S^T of this tile was committed after them)
#pragma unroll 1
                for (int c = 0; c < 8; c++) {
                    float v[32];
                    const uint32_t ta = tmem + lane_base + TM_O + 32 * c;
                    tc::tmem_ld32(ta, v);
                    tc::tmem_wait_ld();
                    const float *al = s_al + 32 * (c & 1);
#pragma unroll
                    for (int j = 0; j < 32; j++) v[j] *= al[j];
                    tc::tmem_st32(ta, v);
                }
                tc::tmem_wait_st();
            }
            // P^T[head][key] in bf16 into the swizzled B tile; row sums
#pragma unroll
            for (int h = 0; h < 64; h++) {
                const float mn = s_mn[h];
                s[h] = (mn == -INFINITY) ? 0.f : fast_exp2(s[h] - mn);
            }
            {
                // this key's 64 heads form one 128-byte swizzled row of the P tile
                uint8_t *prow = sP + tid * 128;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    uint4 v;
                    v.x = pack_bf16x2(s[8 * c + 0], s[8 * c + 1]);
                    v.y = pack_bf16x2(s[8 * c + 2], s[8 * c + 3]);
                    v.z = pack_bf16x2(s[8 * c + 4], s[8 * c + 5]);
                    v.w = pack_bf16x2(s[8 * c + 6], s[8 * c + 7]);
                    *reinterpret_cast<uint4 *>(prow + ((c ^ (tid & 7)) << 4)) = v;
                }
            }
            warp_reduce64<false>(s, r0, r1);
            s_rsum[warp * 64 + 2 * lane] = r0;
            s_rsum[warp * 64 + 2 * lane + 1] = r1;
            tc::fence_proxy_async();
            tc::fence_before_sync();
            tc::named_bar(1, 128);
            if (tid < kTcHeads) {
                const float ls = s_rsum[tid] + s_rsum[64 + tid] + s_rsum[128 + tid] + s_rsum[192 + tid];
                s_l[tid] = s_l[tid] * s_al[tid] + ls;
                s_m[tid] = s_mn[tid];
            }
            mbar_arrive(bar(BAR_PFULL));
        }
        // epilogue: O^T / l -> out[head][d] (bf16), lse
        if (tid == 0) s_flag[0] = ok ? (mbar_wait(bar(BAR_OFULL), 0) ? 1 : 0) : 0;
        tc::named_bar(1, 128);
        if (s_flag[0]) {
            tc::fence_after_sync();
            uint16_t *orow = out + (qi * H + (int64_t)hg * kTcHeads) * kTcD;
#pragma unroll 1
            for (int c = 0; c < 8; c++) {
                float v[32];
                tc::tmem_ld32(tmem + lane_base + TM_O + 32 * c, v);
                tc::tmem_wait_ld();
                const int d = 128 * (c >> 1) + tid;
                const int h0 = 32 * (c & 1);
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    const float l = s_l[h0 + j];
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    orow[(int64_t)(h0 + j) * kTcD + d] = (uint16_t)f32_to_bf16_bits(v[j] * inv);
                }
            }
            if (lse && tid < kTcHeads)
                lse[qi * H + (int64_t)hg * kTcHeads + tid] = (s_m[tid] + log2f(s_l[tid])) * kTcLn2;
        } else if (tid == 0) {
            set_error(err, CSA_ERR_TIMEOUT);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 4) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool attend_tc_applicable(const AttendArgs &a)
{
    const int share = a.num_sms > 0 ? a.num_sms : 148;
    return a.d == kTcD && a.n_heads % kTcHeads == 0 && a.total_q * (a.n_heads / kTcHeads) >= share &&
           (a.idx == nullptr || a.top_k <= kTcIdxCap) && a.total_q <= 0x7fffffffLL;
}

cudaError_t launch_attend_tc(const AttendArgs &a, cudaStream_t st)
{
    if (a.total_q <= 0) return cudaSuccess;
    const dim3 grid((unsigned)a.total_q, (unsigned)(a.n_heads / kTcHeads));
    const float scale_log2 = a.scale * 1.4426950408889634f;
    if (a.idx)
        return launch_kernel("sparse_attend", attend_tc_kernel<true>, grid, dim3(kTcThreads), kTcSmem, st, a.pdl,
                             a.batch, a.cu_kv, a.cu_q, a.cu_ent, a.q, a.entries, a.kv, a.idx, a.n_heads, a.ratio,
                             a.top_k, scale_log2, a.max_kv_len, a.out, a.lse, a.err);
    return launch_kernel("dense_attend", attend_tc_kernel<false>, grid, dim3(kTcThreads), kTcSmem, st, a.pdl,
                         a.batch, a.cu_kv, a.cu_q, a.cu_ent, a.q, a.entries, a.kv, a.idx, a.n_heads, a.ratio,
                         a.top_k, scale_log2, a.max_kv_len, a.out, a.lse, a.err);
}

}  // namespace csa
