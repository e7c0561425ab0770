// Device helpers shared by the CSA/HCA kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "csa.h"

namespace csa {

// --------------------------------------------------------------------------
// Error word: kernels record the first problem they see (atomic, first wins)
// and skip the offending work; they never trap.
// --------------------------------------------------------------------------
__device__ __forceinline__ void set_error(int *err, int code)
{
    if (err) atomicCAS(err, 0, code);
}

// --------------------------------------------------------------------------
// Packed layout lookups.
// --------------------------------------------------------------------------
// Sequence that owns packed row `i` of a cu array (the last b with cu[b] <= i).
__device__ __forceinline__ int find_seq(const int64_t *cu, int batch, int64_t i)
{
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

struct QueryPos {
    int b;          // sequence
    int64_t t;      // 0-based position of the query within its sequence
    int64_t L;      // sequence length
};

// Queries of sequence b are its last n_q positions.
__device__ __forceinline__ QueryPos query_pos(const int64_t *cu_kv, const int64_t *cu_q,
                                              int batch, int64_t qi)
{
    QueryPos p;
    p.b = find_seq(cu_q, batch, qi);
    p.L = __ldg(cu_kv + p.b + 1) - __ldg(cu_kv + p.b);
    const int64_t nq = __ldg(cu_q + p.b + 1) - __ldg(cu_q + p.b);
    p.t = p.L - nq + (qi - __ldg(cu_q + p.b));
    return p;
}

// --------------------------------------------------------------------------
// bf16 <-> fp32 (bit-level; round-to-nearest-even on the way down).
// --------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7f800000u) == 0x7f800000u)            // inf / nan: keep, quiet nans
        return (u >> 16) | ((u & 0x007fffffu) ? 0x40u : 0u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return u >> 16;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    return f32_to_bf16_bits(lo) | (f32_to_bf16_bits(hi) << 16);
}

// Order-preserving map of an fp32 score onto uint32 (larger key = larger score);
// -0 is folded onto +0 so equal scores get equal keys.
__device__ __forceinline__ uint32_t score_key(float s)
{
    uint32_t u = __float_as_uint(s == 0.0f ? 0.0f : s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k)
{
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

// --------------------------------------------------------------------------
// PTX wrappers.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes = 0 zero-fills the destination.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D(16x8 fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace csa
