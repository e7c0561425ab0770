// Token-level compression: softmax-gated pooling of m adjacent tokens' KV into
// one entry ("DeepSeek-V4 core architecture", §2.2 CSA step 1 with m = 4;
// §2.3 HCA with m = 128).  Block j of a sequence holds tokens j*m .. j*m+m-1;
// its entry is sum_t softmax_block(z)_t * c_t, in fp32, rounded to bf16 once.
//
// One CTA owns one 128-token span of one sequence and reads each token row
// once with 16-byte loads.  The small ratio (CSA, m <= 32) is reduced inside
// a thread: a thread owns whole m-token units for 8 channels.  The large
// ratio (HCA, m = 64 or 128) accumulates the same loaded rows into a second
// register set and is reduced across the CTA's row lanes in shared memory,
// so the fused CSA+HCA pass reads the raw KV exactly once.
//
// Only blocks whose last token is a query position are written (all complete
// blocks for a prefill, the block closed by the newest token for a decode).
#include "common.cuh"
#include "launch.h"

namespace csa {

namespace {

constexpr int kCompressThreads = 256;
constexpr int kSpan = 128;
constexpr int kSliceCols = 128;   // columns per CTA (a d = 512 row is split over 4 CTAs)

template <int D, int MS, int MB>
__device__ __forceinline__ void compress_body(const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                                              const int64_t *__restrict__ cu_s, const int64_t *__restrict__ cu_b,
                                              int batch, const uint16_t *__restrict__ kv,
                                              const float *__restrict__ gate, uint16_t *__restrict__ out_s,
                                              uint16_t *__restrict__ out_b, int *err)
{
    constexpr int CS = D < kSliceCols ? D : kSliceCols;   // columns of this CTA's slice
    constexpr int G = CS / 8;                      // 16-byte column groups per slice row
    constexpr int R = kCompressThreads / G;        // row lanes
    constexpr int U = MS > 0 ? MS : 4;             // tokens per unit
    constexpr int NU = kSpan / U;                  // units per span
    constexpr int UPT = (NU + R - 1) / R;          // units per thread
    constexpr int NB = MB > 0 ? kSpan / MB : 0;    // large blocks per span
    static_assert(kCompressThreads % G == 0, "slice groups must divide the CTA");
    static_assert(MS == 0 || (kSpan % MS == 0 && MS <= 32), "small ratio");
    static_assert(MB == 0 || MB == 64 || MB == 128, "large ratio");
    static_assert(UPT * U <= 32, "row registers per thread");

    __shared__ float s_wred[kCompressThreads / 32];
    __shared__ float s_zmax[2], s_zsum[2];
    __shared__ float s_red[NB > 0 ? R * NB * CS : 1];

    griddep_launch();
    const int b = blockIdx.x;
    const int64_t kv0 = cu_kv[b];
    const int64_t L = cu_kv[b + 1] - kv0;
    const int64_t nq = cu_q[b + 1] - cu_q[b];
    const bool bad = nq < 0 || nq > L || (MS > 0 && cu_s[b + 1] - cu_s[b] != L / MS) ||
                     (MB > 0 && cu_b[b + 1] - cu_b[b] != L / MB);
    if (bad) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_error(err, CSA_ERR_DEVICE);
        return;
    }
    if (nq == 0) return;
    const int64_t lo = L - nq;                      // first query position
    const int64_t t0 = (lo / kSpan + blockIdx.y) * kSpan;
    if (t0 >= L) return;

    const int tid = threadIdx.x;
    const int g = tid % G, r = tid / G;
    const int col0 = blockIdx.z * CS;               // first column of the slice

    // Which large blocks of this span are complete and end at a query position.
    bool do_big[NB > 0 ? NB : 1];
    bool any_big = false;
#pragma unroll
    for (int bb = 0; bb < NB; bb++) {
        const int64_t first = t0 + bb * MB;
        do_big[bb] = (first + MB <= L) && (first + MB - 1 >= lo);
        any_big |= do_big[bb];
    }

    // This thread's units: u = r + i*R.  Load every row it needs first (one
    // round trip to memory), then reduce.
    uint4 row[UPT][U];
    float z[UPT][U];
    bool small_needed[UPT], big_read[UPT];
#pragma unroll
    for (int i = 0; i < UPT; i++) {
        const int u = r + i * R;
        const int64_t tu = t0 + (int64_t)u * U;     // first token of the unit
        const bool in_span = u < NU;
        const bool complete = in_span && tu + U <= L;
        small_needed[i] = MS > 0 && complete && (tu + U - 1 >= lo);
        big_read[i] = false;
        if constexpr (MB > 0) big_read[i] = in_span && do_big[(u * U) / MB];
        const bool need = small_needed[i] || big_read[i];
#pragma unroll
        for (int k = 0; k < U; k++) {
            row[i][k] = need ? __ldg(reinterpret_cast<const uint4 *>(kv + (kv0 + tu + k) * D + col0) + g)
                             : make_uint4(0, 0, 0, 0);
            z[i][k] = need ? __ldg(gate + kv0 + tu + k) : 0.f;
        }
    }

    if constexpr (NB > 0) {
        // softmax statistics of the large blocks: warp w < 4 holds tokens 32w..32w+31
        const int w = tid / 32, lane = tid % 32;
        const int bb_w = (w * 32) / MB;
        float zz = -INFINITY;
        if (any_big && w < 4 && do_big[bb_w]) zz = gate[kv0 + t0 + w * 32 + lane];
        float m = warp_max(zz);
        if (lane == 0) s_wred[w] = m;
        __syncthreads();
        if (tid < NB) {
            float mm = -INFINITY;
            for (int ww = tid * MB / 32; ww < (tid + 1) * MB / 32; ww++) mm = fmaxf(mm, s_wred[ww]);
            s_zmax[tid] = mm;
        }
        __syncthreads();
        float e = 0.f;
        if (any_big && w < 4 && do_big[bb_w]) e = expf(zz - s_zmax[bb_w]);
        e = warp_sum(e);
        if (lane == 0) s_wred[w] = e;
        __syncthreads();
        if (tid < NB) {
            float ss = 0.f;
            for (int ww = tid * MB / 32; ww < (tid + 1) * MB / 32; ww++) ss += s_wred[ww];
            s_zsum[tid] = ss;
        }
        __syncthreads();
    }

    float acc_b[NB > 0 ? NB : 1][8];
#pragma unroll
    for (int bb = 0; bb < (NB > 0 ? NB : 1); bb++)
#pragma unroll
        for (int x = 0; x < 8; x++) acc_b[bb][x] = 0.f;

#pragma unroll
    for (int i = 0; i < UPT; i++) {
        const int u = r + i * R;
        const int64_t tu = t0 + (int64_t)u * U;
        if (small_needed[i]) {
            float zm = z[i][0];
#pragma unroll
            for (int k = 1; k < U; k++) zm = fmaxf(zm, z[i][k]);
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            float den = 0.f;
#pragma unroll
            for (int k = 0; k < U; k++) {
                const float wgt = expf(z[i][k] - zm);
                den += wgt;
                const uint32_t wd[4] = {row[i][k].x, row[i][k].y, row[i][k].z, row[i][k].w};
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    acc[2 * c] = fmaf(wgt, bf16_lo(wd[c]), acc[2 * c]);
                    acc[2 * c + 1] = fmaf(wgt, bf16_hi(wd[c]), acc[2 * c + 1]);
                }
            }
            const float inv = 1.f / den;
            uint4 o;
            o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            o.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
            o.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
            const int64_t e = cu_s[b] + tu / (MS > 0 ? MS : 1);
            reinterpret_cast<uint4 *>(out_s + e * D + col0)[g] = o;
        }
        if constexpr (NB > 0) {
            if (big_read[i]) {
                const int bb = (u * U) / MB;
#pragma unroll
                for (int k = 0; k < U; k++) {
                    const float wgt = expf(z[i][k] - s_zmax[bb]);
                    const uint32_t wd[4] = {row[i][k].x, row[i][k].y, row[i][k].z, row[i][k].w};
#pragma unroll
                    for (int c = 0; c < 4; c++) {
#pragma unroll
                        for (int q = 0; q < NB; q++) {
                            if (q == bb) {
                                acc_b[q][2 * c] = fmaf(wgt, bf16_lo(wd[c]), acc_b[q][2 * c]);
                                acc_b[q][2 * c + 1] = fmaf(wgt, bf16_hi(wd[c]), acc_b[q][2 * c + 1]);
                            }
                        }
                    }
                }
            }
        }
    }

    if constexpr (NB > 0) {
        if (!any_big) return;                        // uniform across the CTA
#pragma unroll
        for (int bb = 0; bb < NB; bb++)
#pragma unroll
            for (int x = 0; x < 8; x++) s_red[(r * NB + bb) * CS + g * 8 + x] = acc_b[bb][x];
        __syncthreads();
        for (int p = tid; p < NB * (CS / 2); p += kCompressThreads) {
            const int bb = p / (CS / 2), x = 2 * (p % (CS / 2));
            if (!do_big[bb]) continue;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int rr = 0; rr < R; rr++) {
                s0 += s_red[(rr * NB + bb) * CS + x];
                s1 += s_red[(rr * NB + bb) * CS + x + 1];
            }
            const float inv = 1.f / s_zsum[bb];
            const int64_t e = cu_b[b] + (t0 + bb * MB) / MB;
            reinterpret_cast<uint32_t *>(out_b + e * D + col0)[x / 2] = pack_bf16x2(s0 * inv, s1 * inv);
        }
    }
}

// Launched behind another kernel of the same call (CompressArgs::pdl), this
// grid reads nothing that kernel writes, but every CTA waits for it before
// exiting, whatever path it took: whatever waits for this grid may rely on the
// earlier one too.
template <int D, int MS, int MB>
__global__ void __launch_bounds__(kCompressThreads)
compress_kernel(const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q,
                const int64_t *__restrict__ cu_s, const int64_t *__restrict__ cu_b, int batch,
                const uint16_t *__restrict__ kv, const float *__restrict__ gate,
                uint16_t *__restrict__ out_s, uint16_t *__restrict__ out_b, int *err)
{
    compress_body<D, MS, MB>(cu_kv, cu_q, cu_s, cu_b, batch, kv, gate, out_s, out_b, err);
    griddep_wait();
}

template <int D, int MS, int MB>
cudaError_t launch_compress_t(const CompressArgs &a, cudaStream_t st)
{
    const int64_t spans_kv = (a.max_kv_len + kSpan - 1) / kSpan;
    const int64_t spans_q = (a.max_q_len + kSpan - 1) / kSpan + 1;
    const int64_t spans = spans_kv < spans_q ? spans_kv : spans_q;
    if (spans <= 0 || a.batch <= 0) return cudaSuccess;
    if (spans > 65535) return cudaErrorInvalidConfiguration;   // > 8M tokens per sequence
    constexpr int slices = D / (D < kSliceCols ? D : kSliceCols);
    dim3 grid((unsigned)a.batch, (unsigned)spans, (unsigned)slices);
    return launch_kernel("compress", compress_kernel<D, MS, MB>, grid, dim3(kCompressThreads), 0,
                         st, a.pdl, a.cu_kv, a.cu_q, a.cu_small, a.cu_big, a.batch, a.kv, a.gate,
                         a.out_small, a.out_big, a.err);
}

template <int D>
cudaError_t dispatch_ratio(const CompressArgs &a, cudaStream_t st)
{
    const int ms = a.ratio_small, mb = a.ratio_big;
    if (ms == 4 && mb == 128) return launch_compress_t<D, 4, 128>(a, st);
    if (mb == 0) {
        switch (ms) {
        case 1: return launch_compress_t<D, 1, 0>(a, st);
        case 2: return launch_compress_t<D, 2, 0>(a, st);
        case 4: return launch_compress_t<D, 4, 0>(a, st);
        case 8: return launch_compress_t<D, 8, 0>(a, st);
        case 16: return launch_compress_t<D, 16, 0>(a, st);
        case 32: return launch_compress_t<D, 32, 0>(a, st);
        default: break;
        }
    }
    if (ms == 0) {
        if (mb == 64) return launch_compress_t<D, 0, 64>(a, st);
        if (mb == 128) return launch_compress_t<D, 0, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

bool compress_supported(int d, int ratio_small, int ratio_big)
{
    if (d != 128 && d != 512) return false;
    if (ratio_small == 4 && ratio_big == 128) return true;
    if (ratio_big == 0)
        return ratio_small == 1 || ratio_small == 2 || ratio_small == 4 || ratio_small == 8 ||
               ratio_small == 16 || ratio_small == 32;
    if (ratio_small == 0) return ratio_big == 64 || ratio_big == 128;
    return false;
}

cudaError_t launch_compress(const CompressArgs &a, cudaStream_t st)
{
    if (a.d == 128) return dispatch_ratio<128>(a, st);
    if (a.d == 512) return dispatch_ratio<512>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace csa
