// Inverse rotary correction of attention outputs ("DeepSeek V4's architecture
// debt chain", Constraint 1 -> Innovation 1: the compressed entries carry no
// per-token position, so the attention output receives an inverse RoPE
// correction).  The pages give no convention; the readings: the last d_rope
// dims of each head are rotated, paired as (2i, 2i + 1) within that slice,
// pair i at frequency theta_i = base^(-2i / d_rope), and the output of the
// query at position t is turned by the angle -t * theta_i:
//     (x, y) -> (x cos phi + y sin phi, -x sin phi + y cos phi),  phi = t theta_i.
//
// In place on [total_q, H, d] bf16, HBM-bound: one warp per query, many
// queries in flight per SM, no block-wide barrier.  A lane owns the 16-byte
// vectors (four pairs) of one column group of the rope slice across heads,
// so it turns its four angles once per query: t theta_i in double precision,
// reduced modulo 2 pi there (t theta_i reaches 2^20 radians at a 1M
// context), sine and cosine in fp32; each pair is rotated in fp32 and
// rounded to bf16 once.
#include "common.cuh"
#include "launch.h"

namespace csa {

namespace {

constexpr int kRopeThreads = 256;
constexpr int kRopeMaxPairs = 256;   // d_rope <= 512

// The four (cos, sin) of column group c8 (pairs 4 c8 .. 4 c8 + 3) at position t.
__device__ __forceinline__ void rope_angles(const double *theta, int c8, int64_t t, float (&c)[4], float (&s)[4])
{
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    constexpr double kInvTwoPi = 0.15915494309189533576888376337251;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        double phi = (double)t * theta[4 * c8 + k];
        phi = fma(-floor(phi * kInvTwoPi), kTwoPi, phi);   // into [0, 2 pi)
        sincosf((float)phi, &s[k], &c[k]);
    }
}

__device__ __forceinline__ uint4 rope_turn(uint4 w, const float (&c)[4], const float (&s)[4])
{
    uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const float x = bf16_lo(wd[k]), y = bf16_hi(wd[k]);
        const float xr = fmaf(x, c[k], y * s[k]), yr = fmaf(y, c[k], -(x * s[k]));
        wd[k] = f32_to_bf16_bits(xr) | (f32_to_bf16_bits(yr) << 16);
    }
    return make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

__global__ void __launch_bounds__(kRopeThreads)
inverse_rope_kernel(int batch, const int64_t *__restrict__ cu_kv, const int64_t *__restrict__ cu_q, int64_t total_q,
                    int H, int d, int d_rope, double base, uint16_t *__restrict__ out, int *err)
{
    __shared__ double s_theta[kRopeMaxPairs];
    const int lane = threadIdx.x & 31;
    const int npairs = d_rope / 2;
    for (int i = threadIdx.x; i < npairs; i += kRopeThreads) s_theta[i] = pow(base, -2.0 * i / d_rope);
    __syncthreads();
    const int vph = d_rope / 8;                   // 16-byte vectors per head's slice
    const int nvec = H * vph;
    const bool fixed = 32 % vph == 0;             // this lane's column group is the same for every head
    const int64_t warps = (int64_t)gridDim.x * (kRopeThreads / 32);
    for (int64_t qi = (int64_t)blockIdx.x * (kRopeThreads / 32) + (threadIdx.x >> 5); qi < total_q; qi += warps) {
        const QueryPos p = query_pos(cu_kv, cu_q, nullptr, batch, qi);
        if (p.t < 0 || p.t >= p.L) {   // the same for the whole warp
            if (lane == 0) set_error(err, CSA_ERR_DEVICE);
            continue;
        }
        uint16_t *row0 = out + (qi * H) * (int64_t)d + (d - d_rope);
        float c[4], s[4];
        if (fixed) {
            const int c8 = lane % vph;
            rope_angles(s_theta, c8, p.t, c, s);
            const int step = 32 / vph;
            // four heads' vectors loaded before any is written back
            for (int h0 = lane / vph; h0 < H; h0 += 4 * step) {
                uint4 w[4];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int h = h0 + k * step;
                    if (h < H) w[k] = *reinterpret_cast<const uint4 *>(row0 + (int64_t)h * d + c8 * 8);
                }
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int h = h0 + k * step;
                    if (h < H) *reinterpret_cast<uint4 *>(row0 + (int64_t)h * d + c8 * 8) = rope_turn(w[k], c, s);
                }
            }
        } else {
            for (int v = lane; v < nvec; v += 32) {
                const int h = v / vph, c8 = v - h * vph;
                rope_angles(s_theta, c8, p.t, c, s);
                uint4 *ptr = reinterpret_cast<uint4 *>(row0 + (int64_t)h * d + c8 * 8);
                *ptr = rope_turn(*ptr, c, s);
            }
        }
    }
}

}  // namespace

bool inverse_rope_supported(int d, int d_rope)
{
    return d >= 8 && d % 8 == 0 && d_rope >= 8 && d_rope % 8 == 0 && d_rope <= d && d_rope / 2 <= kRopeMaxPairs;
}

cudaError_t launch_inverse_rope(const RopeArgs &a, cudaStream_t st)
{
    if (a.total_q <= 0) return cudaSuccess;
    // one query per warp; up to eight CTAs (64 warps) per SM
    const int64_t want = (a.total_q + kRopeThreads / 32 - 1) / (kRopeThreads / 32);
    const int64_t cap = 8 * (int64_t)(a.num_sms > 0 ? a.num_sms : 148);
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    return launch_kernel("inverse_rope", inverse_rope_kernel, dim3(grid), dim3(kRopeThreads), 0, st, false, a.batch,
                         a.cu_kv, a.cu_q, a.total_q, a.n_heads, a.d, a.d_rope, a.base, a.out, a.err);
}

}  // namespace csa
