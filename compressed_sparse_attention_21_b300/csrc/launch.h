// Internal launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "csa.h"

namespace csa {

// ---- per-kernel timing (diagnostics; off unless csa_timing_enable(1)) ----
bool timing_enabled();
void timing_record(const char *name, cudaEvent_t start, cudaEvent_t stop);

// Raise a kernel's dynamic shared memory limit (remembered per kernel and device).
cudaError_t ensure_smem_fn(const void *kern, size_t smem);

// Launch `kern` on `st`.  With `pdl` the launch carries programmatic stream
// serialisation: it may begin while the kernel before it on the stream is
// still running, and must execute griddep_wait() before it touches anything
// that kernel (or any earlier work) writes or reads.
// Like launch_kernel, with thread-block clusters of `cluster_x` CTAs along x
// (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(const char *name, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t st, bool pdl, unsigned cluster_x, Args &&...args);

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(const char *name, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool pdl, Args &&...args)
{
    return launch_kernel_cluster(name, kern, grid, block, smem, st, pdl, 1u, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(const char *name, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t st, bool pdl, unsigned cluster_x, Args &&...args)
{
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024) {
        e = ensure_smem_fn(reinterpret_cast<const void *>(kern), smem);
        if (e != cudaSuccess) return e;
    }
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    const bool timed = timing_enabled();
    if (timed) {
        cudaEventCreate(&e0);
        cudaEventCreate(&e1);
        cudaEventRecord(e0, st);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (pdl && !timed) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        na++;
    }
    if (cluster_x > 8) {   // beyond the portable cluster size
        e = cudaFuncSetAttribute(reinterpret_cast<const void *>(kern), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    if (cluster_x > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster_x;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        na++;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (timed) {
        cudaEventRecord(e1, st);
        timing_record(name, e0, e1);
    }
    return e;
}

// ---- compression ----
struct CompressArgs {
    int batch;
    int max_kv_len, max_q_len;
    const int64_t *cu_kv, *cu_q;
    const int64_t *cu_small, *cu_big;   // entry prefix arrays for the two ratios
    int d;
    int ratio_small;                    // 0 = none, else power of two <= 32
    int ratio_big;                      // 0 = none, else 64 or 128
    const uint16_t *kv;
    const float *gate;
    uint16_t *out_small, *out_big;
    int *err;
    bool pdl;   // may overlap the stream's previous kernel (and completes only after it)
};
bool compress_supported(int d, int ratio_small, int ratio_big);
cudaError_t launch_compress(const CompressArgs &a, cudaStream_t st);

// ---- inverse rotary correction of attention outputs ----
struct RopeArgs {
    int batch;
    int64_t total_q;
    const int64_t *cu_kv, *cu_q;
    int n_heads, d, d_rope;
    double base;
    uint16_t *out;   // [total_q, n_heads, d], corrected in place
    int *err;
    int num_sms;
};
bool inverse_rope_supported(int d, int d_rope);
cudaError_t launch_inverse_rope(const RopeArgs &a, cudaStream_t st);

// ---- indexer + top-k ----
struct IndexArgs {
    int batch;
    int max_kv_len, max_q_len;
    int64_t total_q;
    int64_t total_csa;    // rows of k_idx (all sequences)
    bool pdl;             // the key scan of the multi-kernel paths may overlap the stream's previous kernel
    cudaEvent_t scan_done;  // if set: recorded on the stream once every key has been scored
    const int64_t *cu_kv, *cu_q, *cu_csa;
    const uint16_t *q_idx, *k_idx;
    bool fp8;               // the keys are E4M3 codes k_fp8 with row scales k_scale (k_idx unused);
    const uint8_t *k_fp8;   // null only when there are no entries
    const float *k_scale;
    int n_heads_idx, d_idx, ratio, top_k;
    int32_t *idx_out;
    float *score_out;
    void *ws;
    size_t ws_bytes;
    int *err;
    // if set, the call also runs this compression (hybrid step): ahead of the
    // indexer on the single-kernel paths; on the key-scan paths after the
    // first key scan, overlapping it, and before the select (the scan reads no
    // compressed entry; everything after the select needs them).  scan_done
    // is then recorded after it too.
    const CompressArgs *compress;
};
bool index_supported(int n_heads_idx, int d_idx, int top_k);
// prefill-sized batches (index_block.cu): tensor-core score tiles, sampled
// threshold, exact selection among the candidates
bool index_block_applicable(const IndexArgs &a);
size_t index_block_ws_bytes(const IndexArgs &a);      // for a full grid of persistent CTAs
size_t index_block_min_ws_bytes();                      // one CTA (the kernel fits its grid to ws_bytes)
cudaError_t launch_index_block(const IndexArgs &a, cudaStream_t st);
// prefill-sized batches with d_idx = 64 (index_tc.cu): tensor-memory score
// tiles of 128 queries x 256 keys, the same selection
bool index_tc_applicable(const IndexArgs &a);
size_t index_tc_ws_bytes(const IndexArgs &a);         // for a full grid of persistent CTAs
size_t index_tc_min_ws_bytes();                         // one CTA (the kernel fits its grid to ws_bytes)
cudaError_t launch_index_tc(const IndexArgs &a, cudaStream_t st);
size_t index_workspace_bytes(const IndexArgs &a);
// FP8 keys (fp8 set): the chunk scan and the clustered select, rows of up
// to index_fp8_max_n() entries
int64_t index_fp8_max_n();
size_t index_fp8_workspace_bytes(const IndexArgs &a);
// E4M3 codes and per-row fp32 scales of rows indexer keys (d_idx values each)
cudaError_t launch_quantize_index_keys(const uint16_t *k_idx, int64_t rows, int d_idx, uint8_t *k_fp8,
                                       float *k_scale, cudaStream_t st);
// the same, only for the rows of the entries the layout's query positions close
cudaError_t launch_quantize_closed_keys(int batch, const int64_t *cu_kv, const int64_t *cu_q, const int64_t *cu_csa,
                                        int64_t total_q, int ratio, const uint16_t *k_idx, int d_idx, uint8_t *k_fp8,
                                        float *k_scale, int *err, cudaStream_t st);
cudaError_t launch_index_topk(const IndexArgs &a, cudaStream_t st);
// Library-owned scratch of lightning_index_topk_static (see indexer.cu):
// its device address on the current device (looked up on first use), and the
// leading bytes of a workspace that must be zero before a call.
constexpr size_t kIndexStaticScratchBytes = CSA_INDEX_STATIC_SCRATCH_BYTES;
cudaError_t index_static_scratch(void **ptr);
size_t index_static_zero_bytes(const IndexArgs &a);
size_t index_static_need_bytes(const IndexArgs &a);   // smallest scratch the call can run in

// ---- attention ----
struct AttendArgs {
    int batch;
    int max_kv_len, max_q_len;
    int64_t total_q;
    const int64_t *cu_kv, *cu_q, *cu_ent;
    const uint16_t *q, *entries, *kv;
    const int32_t *idx;   // sparse: [total_q, top_k]; dense: nullptr
    int64_t n_ent_rows;   // rows of `entries` (all sequences)
    int64_t n_kv_rows;    // rows of `kv` (all sequences)
    int n_heads, d, ratio, top_k;
    float scale;
    uint16_t *out;
    float *lse;
    void *ws;
    size_t ws_bytes;
    int *err;
    bool pdl;             // may overlap the stream's previous kernel
    int num_sms;          // SMs of the current device (sizes the split-KV grid)
    int sm_share;         // SMs this launch may count on (concurrent branches)
};
bool attend_supported(int n_heads, int d);
// tcgen05 path (attend_tc.cu): d = 512, heads a multiple of 64; decode-sized
// batches split each query's keys over several CTAs and merge the partial
// results (workspace: the partial outputs).
bool attend_tc_applicable(const AttendArgs &a);
size_t attend_tc_workspace_bytes(const AttendArgs &a);
cudaError_t launch_attend_tc(const AttendArgs &a, cudaStream_t st);
size_t attend_workspace_bytes(const AttendArgs &a);
cudaError_t launch_attend(const AttendArgs &a, cudaStream_t st);

}  // namespace csa
