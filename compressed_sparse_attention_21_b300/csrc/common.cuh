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
struct QueryPos {
    int b;          // sequence
    int64_t t;      // 0-based position of the query within its sequence
    int64_t L;      // sequence length
    int64_t kv0;    // first token row of the sequence
    int64_t e0;     // first entry row of the sequence (entry array passed in)
    int64_t ne;     // entries of the sequence
};

// Queries of sequence b are its last n_q positions.  Warp-cooperative: every
// lane of the calling warp must call it with the same arguments.  The 32
// lanes probe cu_q together (one round trip to memory per factor of 32 in
// the batch), then the sequence's offsets arrive in one more round trip;
// cu_e (an entry prefix array) may be null.
__device__ __forceinline__ QueryPos query_pos(const int64_t *cu_kv, const int64_t *cu_q, const int64_t *cu_e,
                                              int batch, int64_t qi)
{
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = batch - 1;          // invariant: cu_q[lo] <= qi
    while (hi > lo) {
        const int stride = (hi - lo + 32) / 32;
        const int at = min(lo + lane * stride, hi);
        const unsigned m = __ballot_sync(0xffffffffu, __ldg(cu_q + at) <= qi);
        const int L = m ? 31 - __clz(m) : 0;   // last probe at or below qi (lane 0, unless cu_q is malformed)
        const int nlo = min(lo + L * stride, hi);
        const int nhi = (L < 31 && lo + (L + 1) * stride <= hi) ? lo + (L + 1) * stride - 1 : hi;
        lo = nlo;
        hi = nhi;
    }
    const int b = lo;
    int64_t v = 0;
    if (lane < 6) {
        const int64_t *arr = lane < 2 ? cu_kv : (lane < 4 ? cu_q : cu_e);
        if (arr) v = __ldg(arr + b + (lane & 1));
    }
    const int64_t kv0 = __shfl_sync(0xffffffffu, v, 0), kv1 = __shfl_sync(0xffffffffu, v, 1);
    const int64_t q0 = __shfl_sync(0xffffffffu, v, 2), q1 = __shfl_sync(0xffffffffu, v, 3);
    const int64_t e0 = __shfl_sync(0xffffffffu, v, 4), e1 = __shfl_sync(0xffffffffu, v, 5);
    QueryPos p;
    p.b = b;
    p.L = kv1 - kv0;
    p.t = p.L - (q1 - q0) + (qi - q0);
    p.kv0 = kv0;
    p.e0 = e0;
    p.ne = e1 - e0;
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

// Two floats -> packed bf16 pair (lo in the low half), round to nearest even,
// in one conversion instruction.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^x by the hardware approximation (ex2.approx: relative error about 2^-22;
// 2^-inf = 0).  Used for softmax weights, which are rounded to bf16 afterwards.
__device__ __forceinline__ float fast_exp2(float x)
{
    float r;
    asm("ex2.approx.f32 %0, %1;\n" : "=f"(r) : "f"(x));
    return r;
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

// --------------------------------------------------------------------------
// mbarrier + bulk (TMA) copies.  Waits are bounded: a wait that runs out
// returns false and the caller reports CSA_ERR_TIMEOUT instead of hanging.
// --------------------------------------------------------------------------
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;   // 0.2 s of wall time

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Non-blocking test of the phase with `parity`.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Wait for the phase with `parity` to complete; gives up (returns false)
// after kWaitLimitNs of wall time.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}
// Contiguous global -> shared copy by the bulk-copy (TMA) engine; completes
// `bytes` of transaction count on `bar`.  Both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Bulk copy shared -> global (16-byte aligned addresses, size a multiple of
// 16), tracked by the issuing thread's bulk group.  Shared-memory writes of
// other threads must be ordered before it with fence.proxy.async and a barrier.
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// every bulk group of this thread complete (its global writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
// every bulk group of this thread has read its shared-memory source (the
// source may be reused or the CTA may exit; the global writes complete on
// their own and are visible once the grid has completed)
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }

// Warp 0: in a 256-bin histogram walked from the top bin down, find the bin
// that holds the `remaining`-th largest element; report it and the count of
// elements in higher bins.
__device__ __forceinline__ void find_digit_256(const uint32_t *hist, uint32_t remaining, uint32_t *out_digit,
                                               uint32_t *out_above)
{
    const int lane = threadIdx.x & 31;
    uint32_t c[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        c[i] = hist[255 - 8 * lane - i];
        sum += c[i];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - sum;
    if (excl < remaining && remaining <= incl) {
        uint32_t acc = excl;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            if (acc + c[i] >= remaining) {
                *out_digit = 255 - 8 * lane - i;
                *out_above = acc;
                break;
            }
            acc += c[i];
        }
    }
}

// Shared-memory histogram increment.  A plain atomic: measured on B300 with
// 512 threads, shared atomics retire 16-30 lanes per cycle per SM (lanes of a
// warp on one address are merged), while aggregating the lanes first with
// __match_any_sync managed 0.6.
__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t bin, bool valid)
{
    if (valid) atomicAdd(hist + bin, 1u);
}

// CTA-wide exclusive scan of one value per thread; returns the prefix and
// the total.  s_w holds 2 * NT/32 + 1 words.
template <int NT>
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t *s_w, uint32_t &total)
{
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t t = lane < NW ? s_w[lane] : 0u;
        uint32_t ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += u;
        }
        if (lane < NW) s_w[NW + lane] = ti - t;
        if (lane == 31) s_w[2 * NW] = ti;
    }
    __syncthreads();
    total = s_w[2 * NW];
    const uint32_t r = s_w[NW + warp] + incl - v;
    __syncthreads();   // s_w may be reused right away
    return r;
}

// Thread-block clusters: rank within the cluster, the cluster-wide barrier
// (release/acquire: shared-memory writes before it are visible to the peers
// after it), and loads from a peer CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// the two halves of cluster_sync: arrive early, wait later
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory"); }
// address of the same shared-memory location in the CTA of cluster rank `rank`
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Programmatic dependent launch.  griddep_wait() blocks until every grid this
// one depends on has completed and its memory is visible (a no-op for a
// launch without a programmatic dependency); griddep_launch() lets the grids
// that depend on this one begin launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

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
