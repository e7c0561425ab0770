// Shared-KV multi-query attention over compressed entries plus the query's
// own raw tail ("DeepSeek-V4 core architecture", §2.2 CSA step 3: each
// selected entry is both key and value and all query heads share it; §2.3
// HCA: dense attention over every compressed entry).
//
// For the query at position t of sequence b the key set is
//   sparse (CSA): { entries[idx[i, s]] : idx >= 0 }  U  raw tokens t-r+1 .. t
//   dense  (HCA): { entries[j] : j < floor((t+1)/m) } U  raw tokens t-r+1 .. t
// with r = (t+1) mod m, and every key is its own value.
//
// One CTA computes HT query heads of one query over one split of its keys:
// the H heads of an MQA query form the M dimension of the tile (they share
// every key), keys stream through a double-buffered shared-memory ring in
// tiles of 64 rows gathered with cp.async, S = Q K^T and O += P K run on the
// bf16 tensor cores (mma.m16n8k16, fp32 accumulate), and the softmax is
// online in the log2 domain.  P is rounded to bf16 for the PV product.
// When a query's keys are split over several CTAs (decode), each split
// writes (O, max, sum) to the workspace and the last split to finish
// (atomic ticket, no waiting) merges them.
#include "common.cuh"
#include "launch.h"

namespace csa {

namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;               // keys per tile
constexpr int kSStride = 72;            // fp32 row stride of the score tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxSplits = 64;
constexpr int kIdxCap = 1792;           // selected indices of one split held in shared memory

__host__ __device__ constexpr int64_t align_up64(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

template <int D, int HT>
struct Cfg {
    static constexpr int MT = HT / 16;          // m16 tiles
    static constexpr int DS = 8 / MT;           // warps per m16 tile (PV: column slices)
    static constexpr int DSW = D / DS;          // PV columns per warp
    static constexpr int NT8 = DSW / 8;         // PV n8 tiles per warp
    static constexpr int QKN = MT;              // QK n8 tiles per warp (8 per tile / DS)
    static constexpr int CPR = D / 8;           // 16-byte chunks per row
    static constexpr int RB = 2 * D;            // bytes per bf16 row
    static constexpr int TPR = kThreads / HT;   // softmax threads per row
    static constexpr int CPT = kTile / TPR;     // softmax columns per thread
    static constexpr size_t q_bytes = size_t(HT) * RB;
    static constexpr size_t k_bytes = size_t(kTile) * RB;
    static constexpr size_t s_bytes = size_t(HT) * kSStride * 4;
    static constexpr size_t p_bytes = size_t(HT) * kTile * 2;
    static constexpr int NST = (HT == 16 && D == 512) ? 3 : 2;   // key tiles in the ring
    static constexpr size_t off_q = 0;
    static constexpr size_t off_k0 = off_q + q_bytes;
    static constexpr size_t off_s = off_k0 + NST * k_bytes;
    static constexpr size_t off_p = off_s + s_bytes;
    static constexpr size_t off_stats = off_p + p_bytes;             // m, l, alpha: 3*HT floats
    static constexpr size_t off_valid = off_stats + 3 * HT * 4;      // NST x 64 flags
    static constexpr size_t off_idx = off_valid + NST * kTile * 4;   // this split's selection
    static constexpr size_t smem = off_idx + kIdxCap * 4 + 16;
    static_assert(smem <= 232448, "shared memory per CTA");
    static_assert(HT == 16 || HT == 64, "head tile");
    static_assert(NT8 % 2 == 0, "PV n-tiles come in pairs");
    static_assert(CPR >= 8, "swizzle needs 8 chunks per row");
};

// byte offset of 16-byte chunk `chunk` of row `row` in a swizzled tile
template <int RB>
__device__ __forceinline__ uint32_t swz(int row, int chunk)
{
    return (uint32_t)(row * RB + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t &r0, uint32_t &r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}

struct KeySet {
    const uint16_t *safe;      // any valid global address (source of zero-size copies)
    const uint16_t *entries;   // sequence's first entry row
    const uint16_t *tail;      // first raw tail token row
    const int32_t *idx;        // sparse: this query's idx row (indexed by slot); dense: nullptr
    int64_t n_vis;             // visible entries
    int n_main;                // main key slots (entries)
    int n_keys;                // main + tail
};

template <int D, bool GATHER>
__device__ __forceinline__ const uint16_t *key_row(const KeySet &ks, int slot, int *err)
{
    if (slot < ks.n_main) {
        if (GATHER) {
            const int e = ks.idx[slot];   // shared memory (prefetched) or global
            if (e < 0) return nullptr;
            if ((int64_t)e >= ks.n_vis) {
                set_error(err, CSA_ERR_DEVICE);
                return nullptr;
            }
            return ks.entries + (int64_t)e * D;
        }
        return ks.entries + (int64_t)slot * D;
    }
    if (slot < ks.n_keys) return ks.tail + (int64_t)(slot - ks.n_main) * D;
    return nullptr;
}

template <int D, int HT, bool GATHER>
__device__ __forceinline__ void load_tile(uint8_t *smem, uint32_t sbase_k, int *s_valid, const KeySet &ks,
                                          int slot0, int *err)
{
    using C = Cfg<D, HT>;
    const int tid = threadIdx.x;
    const int chunk = tid % C::CPR;
#pragma unroll 4
    for (int row = tid / C::CPR; row < kTile; row += kThreads / C::CPR) {
        const uint16_t *src = key_row<D, GATHER>(ks, slot0 + row, err);
        const uint32_t dst = sbase_k + swz<C::RB>(row, chunk);
        cp_async_16(dst, src ? (const void *)(src + chunk * 8) : (const void *)ks.safe, src ? 16 : 0);
        if (chunk == 0) s_valid[row] = src != nullptr;
    }
}

template <int D, int HT, bool GATHER>
__global__ void __launch_bounds__(kThreads, 1)
attend_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
              const int64_t *__restrict__ cu_ent, const uint16_t *__restrict__ q,
              const uint16_t *__restrict__ entries, const uint16_t *__restrict__ kv,
              const int32_t *__restrict__ idx, int H, int ratio, int top_k, float scale_log2, int kps,
              int nsplit_max, int max_kv_len, uint16_t *__restrict__ out, float *__restrict__ lse,
              float *__restrict__ part_o, float *__restrict__ part_ml, uint32_t *__restrict__ tickets, int *err)
{
    using C = Cfg<D, HT>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int HG = (H + HT - 1) / HT;
    const int hg = blockIdx.y % HG;
    const int split = blockIdx.y / HG;
    const int64_t qi = blockIdx.x;

    const QueryPos p = query_pos(cu_kv, cu_q, cu_ent, batch, qi);
    const int64_t n_vis = (p.t + 1) / ratio;
    const int r_tail = (int)((p.t + 1) % ratio);
    const bool bad = p.t < 0 || p.t >= p.L || p.L > max_kv_len ||
                     p.ne != p.L / ratio;
    if (bad) {
        if (tid == 0) set_error(err, CSA_ERR_DEVICE);
        return;
    }
    KeySet ks;
    ks.safe = kv;
    // main keys: the selected entries (at most top_k), or all visible entries,
    // or with top_k > 0 only the most recent top_k of them (a sliding window)
    ks.n_main = (int)(top_k > 0 && n_vis > top_k ? top_k : n_vis);
    ks.entries = entries + (p.e0 + (GATHER ? 0 : n_vis - ks.n_main)) * D;
    ks.tail = kv + (p.kv0 + p.t - r_tail + 1) * D;
    ks.idx = GATHER ? idx + qi * top_k : nullptr;
    ks.n_vis = n_vis;
    ks.n_keys = ks.n_main + r_tail;
    const int nsplit = (ks.n_keys + kps - 1) / kps;
    if (split >= nsplit) return;
    const int key0 = split * kps;
    const int key1 = min(ks.n_keys, key0 + kps);
    const int ntiles = (key1 - key0 + kTile - 1) / kTile;

    const uint32_t sb = smem_u32(smem);
    const uint32_t sQ = sb + C::off_q;
    float *sS = reinterpret_cast<float *>(smem + C::off_s);
    const uint32_t sP = sb + C::off_p;
    float *s_m = reinterpret_cast<float *>(smem + C::off_stats);
    float *s_l = s_m + HT;
    float *s_alpha = s_l + HT;
    int *s_valid = reinterpret_cast<int *>(smem + C::off_valid);

    // Q tile (rows beyond H are zero) and the first key tile
    {
        const int chunk = tid % C::CPR;
        for (int row = tid / C::CPR; row < HT; row += kThreads / C::CPR) {
            const int h = hg * HT + row;
            const uint16_t *src = q + (qi * H + (h < H ? h : 0)) * (int64_t)D + chunk * 8;
            cp_async_16(sQ + swz<C::RB>(row, chunk), src, h < H ? 16 : 0);
        }
    }
    // everything below reads what earlier kernels produced (selection, entries)
    // or writes what they may still read: wait for them
    griddep_wait();
    if (GATHER) {
        // this split's selected indices, read once: the gathers then need no
        // global round trip of their own
        const int i1 = min(key1, ks.n_main);
        if (i1 - key0 <= kIdxCap) {
            int32_t *s_idx = reinterpret_cast<int32_t *>(smem + C::off_idx);
            for (int i = key0 + tid; i < i1; i += kThreads) s_idx[i - key0] = __ldg(ks.idx + i);
            __syncthreads();
            ks.idx = s_idx - key0;
        }
    }
    // the first NST-1 key tiles (the Q tile travels with the first group)
#pragma unroll
    for (int st = 0; st < C::NST - 1; st++) {
        if (st < ntiles)
            load_tile<D, HT, GATHER>(smem, sb + C::off_k0 + st * C::k_bytes, s_valid + st * kTile, ks,
                                     key0 + st * kTile, err);
        cp_async_commit();
    }
    for (int i = tid; i < HT; i += kThreads) {
        s_m[i] = -INFINITY;
        s_l[i] = 0.f;
    }

    const int mt = warp / C::DS;     // m16 tile of this warp
    const int ds = warp % C::DS;     // column slice (PV) / key slice (QK)
    const int g = lane >> 2, c4 = lane & 3;

    float o[C::NT8][4];
#pragma unroll
    for (int i = 0; i < C::NT8; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    for (int it = 0; it < ntiles; it++) {
        const int buf = it % C::NST;
        const uint32_t sK = sb + C::off_k0 + buf * C::k_bytes;
        const int nxt = it + C::NST - 1;   // refills the stage computed in the previous iteration
        if (nxt < ntiles)
            load_tile<D, HT, GATHER>(smem, sb + C::off_k0 + (nxt % C::NST) * C::k_bytes,
                                     s_valid + (nxt % C::NST) * kTile, ks, key0 + nxt * kTile, err);
        cp_async_commit();
        cp_async_wait<C::NST - 1>();
        __syncthreads();

        // ---- S = Q K^T for rows of tile mt, keys [ds*QKN*8, +QKN*8) ----
        float sacc[C::QKN][4];
#pragma unroll
        for (int j = 0; j < C::QKN; j++) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
        const int n0 = ds * C::QKN * 8;
#pragma unroll 4
        for (int kk = 0; kk < D / 16; kk++) {
            uint32_t a[4];
            {
                const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int ch = kk * 2 + (lane >> 4);
                ldmatrix_x4(sQ + swz<C::RB>(row, ch), a[0], a[1], a[2], a[3]);
            }
            if constexpr (C::QKN == 1) {
                uint32_t b0, b1;
                const int row = n0 + (lane & 7);
                const int ch = kk * 2 + ((lane >> 3) & 1);
                ldmatrix_x2(sK + swz<C::RB>(row, ch), b0, b1);
                mma_bf16_16816(sacc[0], a, b0, b1);
            } else {
#pragma unroll
                for (int j = 0; j < C::QKN; j += 2) {
                    uint32_t b0, b1, b2, b3;
                    const int row = n0 + j * 8 + (lane & 7) + (lane >> 4) * 8;
                    const int ch = kk * 2 + ((lane >> 3) & 1);
                    ldmatrix_x4(sK + swz<C::RB>(row, ch), b0, b1, b2, b3);
                    mma_bf16_16816(sacc[j], a, b0, b1);
                    mma_bf16_16816(sacc[j + 1], a, b2, b3);
                }
            }
        }
        {
            const int *valid = s_valid + buf * kTile;
#pragma unroll
            for (int j = 0; j < C::QKN; j++) {
                const int col = n0 + j * 8 + 2 * c4;
                const bool v0 = valid[col] != 0, v1 = valid[col + 1] != 0;
                float2 lo, hi;
                lo.x = v0 ? sacc[j][0] * scale_log2 : -INFINITY;
                lo.y = v1 ? sacc[j][1] * scale_log2 : -INFINITY;
                hi.x = v0 ? sacc[j][2] * scale_log2 : -INFINITY;
                hi.y = v1 ? sacc[j][3] * scale_log2 : -INFINITY;
                *reinterpret_cast<float2 *>(sS + (mt * 16 + g) * kSStride + col) = lo;
                *reinterpret_cast<float2 *>(sS + (mt * 16 + g + 8) * kSStride + col) = hi;
            }
        }
        __syncthreads();

        // ---- online softmax: TPR threads per row, CPT columns each ----
        {
            const int row = tid / C::TPR;
            const int c0 = (tid % C::TPR) * C::CPT;
            float s[C::CPT];
#pragma unroll
            for (int i = 0; i < C::CPT; i += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(sS + row * kSStride + c0 + i);
                s[i] = v.x;
                s[i + 1] = v.y;
                s[i + 2] = v.z;
                s[i + 3] = v.w;
            }
            float mx = s[0];
#pragma unroll
            for (int i = 1; i < C::CPT; i++) mx = fmaxf(mx, s[i]);
#pragma unroll
            for (int off = 1; off < C::TPR; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_old = s_m[row];
            const float m_new = fmaxf(m_old, mx);
            const bool none = m_new == -INFINITY;
            const float alpha = none ? 1.f : fast_exp2(m_old - m_new);
            float sum = 0.f;
            uint32_t pk[C::CPT / 2];
#pragma unroll
            for (int i = 0; i < C::CPT; i += 2) {
                const float p0 = none ? 0.f : fast_exp2(s[i] - m_new);
                const float p1 = none ? 0.f : fast_exp2(s[i + 1] - m_new);
                sum += p0 + p1;
                pk[i / 2] = pack_bf16x2(p0, p1);
            }
#pragma unroll
            for (int off = 1; off < C::TPR; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            uint8_t *pbase = smem + C::off_p;
            if constexpr (C::CPT >= 8) {
#pragma unroll
                for (int i = 0; i < C::CPT; i += 8) {
                    const int ch = (c0 + i) >> 3;
                    *reinterpret_cast<uint4 *>(pbase + swz<kTile * 2>(row, ch)) =
                        make_uint4(pk[i / 2], pk[i / 2 + 1], pk[i / 2 + 2], pk[i / 2 + 3]);
                }
            } else {
                const int ch = c0 >> 3;
                *reinterpret_cast<uint2 *>(pbase + swz<kTile * 2>(row, ch) + (c0 & 7) * 2) =
                    make_uint2(pk[0], pk[1]);
            }
            __syncwarp();
            if (tid % C::TPR == 0) {
                s_m[row] = m_new;
                s_l[row] = s_l[row] * alpha + sum;
                s_alpha[row] = alpha;
            }
        }
        __syncthreads();

        // ---- O = alpha * O + P K  for rows of tile mt, columns of slice ds ----
        {
            const float a_lo = s_alpha[mt * 16 + g], a_hi = s_alpha[mt * 16 + g + 8];
#pragma unroll
            for (int i = 0; i < C::NT8; i++) {
                o[i][0] *= a_lo;
                o[i][1] *= a_lo;
                o[i][2] *= a_hi;
                o[i][3] *= a_hi;
            }
#pragma unroll
            for (int kk = 0; kk < kTile / 16; kk++) {
                uint32_t a[4];
                {
                    const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int ch = kk * 2 + (lane >> 4);
                    ldmatrix_x4(sP + swz<kTile * 2>(row, ch), a[0], a[1], a[2], a[3]);
                }
#pragma unroll
                for (int np = 0; np < C::NT8 / 2; np++) {
                    uint32_t b0, b1, b2, b3;
                    const int row = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int ch = (ds * C::DSW + np * 16) / 8 + (lane >> 4);
                    ldmatrix_x4_trans(sK + swz<C::RB>(row, ch), b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * np], a, b0, b1);
                    mma_bf16_16816(o[2 * np + 1], a, b2, b3);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // ---- epilogue ----
    const int r_lo = mt * 16 + g, r_hi = r_lo + 8;
    const int h_lo = hg * HT + r_lo, h_hi = hg * HT + r_hi;
    if (nsplit == 1) {
        const float l_lo = s_l[r_lo], l_hi = s_l[r_hi];
        const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f, inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
#pragma unroll
        for (int i = 0; i < C::NT8; i++) {
            const int col = ds * C::DSW + i * 8 + 2 * c4;
            if (h_lo < H)
                *reinterpret_cast<uint32_t *>(out + (qi * H + h_lo) * (int64_t)D + col) =
                    pack_bf16x2(o[i][0] * inv_lo, o[i][1] * inv_lo);
            if (h_hi < H)
                *reinterpret_cast<uint32_t *>(out + (qi * H + h_hi) * (int64_t)D + col) =
                    pack_bf16x2(o[i][2] * inv_hi, o[i][3] * inv_hi);
        }
        if (lse && ds == 0 && c4 == 0) {
            if (h_lo < H) lse[qi * H + h_lo] = (s_m[r_lo] + log2f(l_lo)) * kLn2;
            if (h_hi < H) lse[qi * H + h_hi] = (s_m[r_hi] + log2f(l_hi)) * kLn2;
        }
        return;
    }

    // split: publish the partial state, the last split merges
    const int64_t unit = qi * HG + hg;
    float *po = part_o + (unit * nsplit_max + split) * (int64_t)HT * D;
    float *pml = part_ml + (unit * nsplit_max + split) * (int64_t)HT * 2;
#pragma unroll
    for (int i = 0; i < C::NT8; i++) {
        const int col = ds * C::DSW + i * 8 + 2 * c4;
        *reinterpret_cast<float2 *>(po + r_lo * D + col) = make_float2(o[i][0], o[i][1]);
        *reinterpret_cast<float2 *>(po + r_hi * D + col) = make_float2(o[i][2], o[i][3]);
    }
    for (int i = tid; i < HT; i += kThreads) {
        pml[2 * i] = s_m[i];
        pml[2 * i + 1] = s_l[i];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(tickets + unit, 1u) == (uint32_t)(nsplit - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // merge weights per row: w_s = 2^(m_s - M), L = sum_s w_s l_s  (reuse the key ring)
    float *s_wt = reinterpret_cast<float *>(smem + C::off_k0);   // [HT][nsplit]
    float *s_inv = s_wt + HT * kMaxSplits;                       // [HT]
    float *s_lse = s_inv + HT;                                   // [HT]
    for (int row = tid; row < HT; row += kThreads) {
        const float *ml = part_ml + unit * nsplit_max * (int64_t)HT * 2;
        float M = -INFINITY;
        for (int s = 0; s < nsplit; s++) M = fmaxf(M, __ldcg(ml + (s * HT + row) * 2));
        float Lsum = 0.f;
        for (int s = 0; s < nsplit; s++) {
            const float ms = __ldcg(ml + (s * HT + row) * 2);
            const float w = (ms == -INFINITY) ? 0.f : fast_exp2(ms - M);
            s_wt[row * kMaxSplits + s] = w;
            Lsum += w * __ldcg(ml + (s * HT + row) * 2 + 1);
        }
        s_inv[row] = Lsum > 0.f ? 1.f / Lsum : 0.f;
        s_lse[row] = (M + log2f(Lsum)) * kLn2;
    }
    __syncthreads();
    // weighted sum of the partial outputs: U float4 columns per thread at a
    // time, so that U loads per split are in flight instead of one
    const float *pbase = part_o + unit * nsplit_max * (int64_t)HT * D;
    constexpr int NE = HT * D / 4;
    constexpr int EPT = NE / kThreads;
    constexpr int U = EPT < 4 ? EPT : 4;
    static_assert(NE % kThreads == 0 && EPT % U == 0, "merge tiling");
    for (int e0 = 0; e0 < EPT; e0 += U) {
        int rows[U], cols[U];
        float4 acc[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int e = tid + (e0 + u) * kThreads;
            rows[u] = e / (D / 4);
            cols[u] = (e % (D / 4)) * 4;
            acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll 2
        for (int s = 0; s < nsplit; s++) {
            float4 v[U];
#pragma unroll
            for (int u = 0; u < U; u++)
                v[u] = __ldcg(reinterpret_cast<const float4 *>(pbase + ((int64_t)s * HT + rows[u]) * D + cols[u]));
#pragma unroll
            for (int u = 0; u < U; u++) {
                const float w = s_wt[rows[u] * kMaxSplits + s];
                acc[u].x = fmaf(w, v[u].x, acc[u].x);
                acc[u].y = fmaf(w, v[u].y, acc[u].y);
                acc[u].z = fmaf(w, v[u].z, acc[u].z);
                acc[u].w = fmaf(w, v[u].w, acc[u].w);
            }
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int h = hg * HT + rows[u];
            if (h >= H) continue;
            const float inv = s_inv[rows[u]];
            uint2 pk;
            pk.x = pack_bf16x2(acc[u].x * inv, acc[u].y * inv);
            pk.y = pack_bf16x2(acc[u].z * inv, acc[u].w * inv);
            *reinterpret_cast<uint2 *>(out + (qi * H + h) * (int64_t)D + cols[u]) = pk;
        }
    }
    if (lse)
        for (int row = tid; row < HT; row += kThreads)
            if (hg * HT + row < H) lse[qi * H + hg * HT + row] = s_lse[row];
    if (tid == 0) tickets[unit] = 0;   // leave the ticket zeroed for the next call
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct Plan {
    int HT, HG;
    int max_keys;
    int kps;          // keys per split (multiple of kTile)
    int nsplit_max;
};

constexpr int kMinSplitKeys = 128;   // fewest keys worth a split of their own

Plan make_plan(const AttendArgs &a)
{
    Plan pl;
    const int share = a.sm_share > 0 ? a.sm_share : (a.num_sms > 0 ? a.num_sms : 148);
    // Head tile.  When there are at least as many 64-head units as SMs (prefill),
    // 64 heads of a query share every key tile a CTA loads.  Otherwise (decode)
    // 16-head tiles spread a query over more SMs without splitting its keys:
    // every key split costs an fp32 partial output of HT x d, which at d = 512
    // and 64 heads is as many bytes as 128 keys.
    const int64_t units64 = a.total_q * ((a.n_heads + 63) / 64);
    pl.HT = (a.n_heads <= 16 || units64 < share) ? 16 : 64;
    pl.HG = (a.n_heads + pl.HT - 1) / pl.HT;
    const int64_t max_vis = a.max_kv_len / a.ratio;
    int64_t mk = (a.top_k > 0 && max_vis > a.top_k ? a.top_k : max_vis) + (a.ratio - 1);
    if (mk > a.max_kv_len) mk = a.max_kv_len;   // tail never exceeds the sequence
    if (mk < 1) mk = 1;
    pl.max_keys = (int)mk;
    // Key splits: as many as keep every unit's CTAs within one wave of `share`
    // CTAs, and no fewer than kMinSplitKeys keys per split.
    const int64_t units = a.total_q * pl.HG;
    int64_t want = units >= share ? 1 : share / units;
    const int64_t by_keys = (mk + kMinSplitKeys - 1) / kMinSplitKeys;
    if (want > by_keys) want = by_keys;
    if (want > kMaxSplits) want = kMaxSplits;
    if (want < 1) want = 1;
    int64_t kps = align_up64((mk + want - 1) / want, kTile);
    if (kps < kTile) kps = kTile;
    int64_t ns = (mk + kps - 1) / kps;
    while (ns > kMaxSplits) {
        kps += kTile;
        ns = (mk + kps - 1) / kps;
    }
    pl.kps = (int)kps;
    pl.nsplit_max = (int)ns;
    return pl;
}

struct WsA {
    float *part_o;
    float *part_ml;
    uint32_t *tickets;
};

size_t ws_bytes_for(const AttendArgs &a, const Plan &pl, WsA *w)
{
    if (pl.nsplit_max <= 1) {
        if (w) *w = WsA{nullptr, nullptr, nullptr};
        return 0;
    }
    const int64_t units = a.total_q * pl.HG;
    const int64_t tick = align_up64(units * 4, 256);
    const int64_t ml = align_up64(units * pl.nsplit_max * (int64_t)pl.HT * 2 * 4, 256);
    const int64_t po = align_up64(units * pl.nsplit_max * (int64_t)pl.HT * a.d * 4, 256);
    if (w) {
        char *p = static_cast<char *>(a.ws);
        w->tickets = reinterpret_cast<uint32_t *>(p);
        w->part_ml = reinterpret_cast<float *>(p + tick);
        w->part_o = reinterpret_cast<float *>(p + tick + ml);
    }
    return (size_t)(tick + ml + po);
}

template <int D, int HT, bool GATHER>
cudaError_t launch_t(const AttendArgs &a, const Plan &pl, const WsA &w, cudaStream_t st)
{
    using C = Cfg<D, HT>;
    if (pl.HG * pl.nsplit_max > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)a.total_q, (unsigned)(pl.HG * pl.nsplit_max));
    const float scale_log2 = a.scale * kLog2e;
    return launch_kernel(GATHER ? "sparse_attend" : "dense_attend", attend_kernel<D, HT, GATHER>, grid,
                         dim3(kThreads), C::smem, st, a.pdl, a.batch, a.cu_kv, a.cu_q, a.cu_ent, a.q, a.entries, a.kv,
                         a.idx, a.n_heads, a.ratio, a.top_k, scale_log2, pl.kps, pl.nsplit_max, a.max_kv_len,
                         a.out, a.lse, w.part_o, w.part_ml, w.tickets, a.err);
}

template <int D, bool GATHER>
cudaError_t launch_d(const AttendArgs &a, const Plan &pl, const WsA &w, cudaStream_t st)
{
    if (pl.HT == 16) return launch_t<D, 16, GATHER>(a, pl, w, st);
    return launch_t<D, 64, GATHER>(a, pl, w, st);
}

}  // namespace

bool attend_supported(int n_heads, int d)
{
    if (d != 128 && d != 512) return false;
    return (n_heads >= 1 && n_heads <= 16) || (n_heads % 64 == 0 && n_heads <= 256);
}

size_t attend_workspace_bytes(const AttendArgs &a)
{
    if (a.total_q <= 0) return 0;
    if (attend_tc_applicable(a)) return attend_tc_workspace_bytes(a);
    return ws_bytes_for(a, make_plan(a), nullptr);
}

cudaError_t launch_attend(const AttendArgs &a, cudaStream_t st)
{
    if (a.total_q <= 0) return cudaSuccess;
    if (attend_tc_applicable(a)) return launch_attend_tc(a, st);
    const Plan pl = make_plan(a);
    WsA w;
    ws_bytes_for(a, pl, &w);
    const bool gather = a.idx != nullptr;
    if (a.d == 128) return gather ? launch_d<128, true>(a, pl, w, st) : launch_d<128, false>(a, pl, w, st);
    if (a.d == 512) return gather ? launch_d<512, true>(a, pl, w, st) : launch_d<512, false>(a, pl, w, st);
    return cudaErrorInvalidValue;
}

}  // namespace csa
