// C-ABI entry points of the CSA + HCA library: host-side argument checks,
// per-device state, workspace carving and the two-branch hybrid step.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "csa.h"
#include "launch.h"

namespace csa {

// Device error word (one per device that loads the library).
static __device__ int g_error_word;

namespace {

struct DeviceState {
    bool ready = false;
    int *err = nullptr;
    int num_sms = 0;
};

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

csa_status_t device_state(DeviceState **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return CSA_ERR_CUDA;
        s.err = static_cast<int *>(p);
        if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return CSA_ERR_CUDA;
        s.ready = true;
    }
    *out = &s;
    return CSA_OK;
}

// The helper stream and events of hybrid_attend, one set per (device, caller
// stream), so that calls on different streams (or captured into different
// graphs) never record or wait on each other's events.  `mu` is held while a
// call issues its work, so two host threads issuing on the same stream do not
// interleave their event records either.  Created on first use and kept until
// the process exits.
struct Helper {
    cudaStream_t aux = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, sdone = nullptr;
    std::mutex mu;
};
constexpr size_t kMaxHelpers = 256;
std::map<std::pair<int, cudaStream_t>, std::unique_ptr<Helper>> g_helpers;
std::mutex g_helpers_mu;

// The helper of (current device, st); null once kMaxHelpers pairs have one
// (the call then runs both branches on `st`, one after the other).
csa_status_t helper_for(cudaStream_t st, Helper **out)
{
    *out = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_helpers_mu);
    const auto key = std::make_pair(dev, st);
    auto it = g_helpers.find(key);
    if (it != g_helpers.end()) {
        *out = it->second.get();
        return CSA_OK;
    }
    if (g_helpers.size() >= kMaxHelpers) return CSA_OK;
    std::unique_ptr<Helper> h(new Helper);
    if (cudaStreamCreateWithFlags(&h->aux, cudaStreamNonBlocking) != cudaSuccess) return CSA_ERR_CUDA;
    if (cudaEventCreateWithFlags(&h->fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->join, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->sdone, cudaEventDisableTiming) != cudaSuccess)
        return CSA_ERR_CUDA;
    *out = h.get();
    g_helpers.emplace(key, std::move(h));
    return CSA_OK;
}

// Address of the device error word on the current device, without creating
// the helper stream and events of device_state (for the scratch-free entry).
std::mutex g_err_mu;
int *g_err_ptr[kMaxDevices];

csa_status_t error_word(int **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_err_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return CSA_ERR_CUDA;
        g_err_ptr[dev] = static_cast<int *>(p);
    }
    *out = g_err_ptr[dev];
    return CSA_OK;
}

// ---- timing registry ----
std::atomic<bool> g_timing{false};
std::mutex g_timing_mu;
struct Pending {
    std::string name;
    cudaEvent_t a, b;
};
std::vector<Pending> g_pending;
std::map<std::string, std::pair<int64_t, double>> g_timing_acc;

// ---- dynamic shared memory grants ----
std::mutex g_smem_mu;
std::map<std::pair<int, const void *>, size_t> g_smem;

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

csa_status_t from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return CSA_OK;
    if (e == cudaErrorInvalidValue || e == cudaErrorInvalidConfiguration) return CSA_ERR_UNSUPPORTED;
    return CSA_ERR_CUDA;
}

csa_status_t check_layout(const csa_layout *L, bool need_csa, bool need_hca)
{
    if (!L || L->reserved != 0 || L->batch <= 0) return CSA_ERR_INVALID_ARG;
    if (!L->cu_kv || !L->cu_q) return CSA_ERR_INVALID_ARG;
    if (need_csa && !L->cu_csa) return CSA_ERR_INVALID_ARG;
    if (need_hca && !L->cu_hca) return CSA_ERR_INVALID_ARG;
    if (L->max_kv_len <= 0 || L->max_q_len < 0 || L->max_q_len > L->max_kv_len) return CSA_ERR_INVALID_ARG;
    if (L->total_kv < 0 || L->total_q < 0 || L->total_csa < 0 || L->total_hca < 0) return CSA_ERR_INVALID_ARG;
    if (L->total_q > (int64_t)L->batch * L->max_q_len) return CSA_ERR_INVALID_ARG;
    if (L->total_kv > (int64_t)L->batch * L->max_kv_len) return CSA_ERR_INVALID_ARG;
    if (L->total_q > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
    return CSA_OK;
}

csa_status_t check_ptr(const void *p, bool needed)
{
    if (!needed) return CSA_OK;
    if (!p) return CSA_ERR_INVALID_ARG;
    return aligned16(p) ? CSA_OK : CSA_ERR_INVALID_ARG;
}

#define CSA_TRY(x)                                  \
    do {                                            \
        const csa_status_t s_ = (x);                \
        if (s_ != CSA_OK) return s_;                \
    } while (0)

constexpr size_t kWsAlign = 256;
inline size_t align_ws(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

IndexArgs index_args(const csa_layout *L, const csa_bf16 *q_idx, const csa_bf16 *k_idx, int hi, int di, int ratio,
                     int top_k, int32_t *idx_out, float *score_out, void *ws, size_t ws_bytes, int *err)
{
    IndexArgs a;
    a.compress = nullptr;
    a.batch = L->batch;
    a.max_kv_len = L->max_kv_len;
    a.max_q_len = L->max_q_len;
    a.total_q = L->total_q;
    a.total_csa = L->total_csa;
    a.pdl = false;
    a.scan_done = nullptr;
    a.cu_kv = L->cu_kv;
    a.cu_q = L->cu_q;
    a.cu_csa = L->cu_csa;
    a.q_idx = q_idx;
    a.k_idx = k_idx;
    a.fp8 = false;
    a.k_fp8 = nullptr;
    a.k_scale = nullptr;
    a.n_heads_idx = hi;
    a.d_idx = di;
    a.ratio = ratio;
    a.top_k = top_k;
    a.idx_out = idx_out;
    a.score_out = score_out;
    a.ws = ws;
    a.ws_bytes = ws_bytes;
    a.err = err;
    return a;
}

AttendArgs attend_args(const csa_layout *L, bool csa_side, const csa_bf16 *q, const csa_bf16 *entries,
                       const csa_bf16 *kv, const int32_t *idx, int H, int d, int ratio, int top_k, float scale,
                       csa_bf16 *out, float *lse, void *ws, size_t ws_bytes, int *err, int num_sms, int sm_share)
{
    AttendArgs a;
    a.batch = L->batch;
    a.max_kv_len = L->max_kv_len;
    a.max_q_len = L->max_q_len;
    a.total_q = L->total_q;
    a.cu_kv = L->cu_kv;
    a.cu_q = L->cu_q;
    a.cu_ent = csa_side ? L->cu_csa : L->cu_hca;
    a.n_ent_rows = csa_side ? L->total_csa : L->total_hca;
    a.n_kv_rows = L->total_kv;
    a.q = q;
    a.entries = entries;
    a.kv = kv;
    a.idx = idx;
    a.n_heads = H;
    a.d = d;
    a.ratio = ratio;
    a.top_k = top_k;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    a.ws = ws;
    a.ws_bytes = ws_bytes;
    a.err = err;
    a.pdl = false;
    a.num_sms = num_sms;
    a.sm_share = sm_share;
    return a;
}

csa_status_t check_index(const csa_layout *L, const csa_bf16 *q_idx, const csa_bf16 *k_idx, int hi, int di,
                         int ratio, int top_k, const int32_t *idx_out, const float *score_out)
{
    CSA_TRY(check_layout(L, true, false));
    if (ratio <= 0 || ratio > 1024 || top_k <= 0) return CSA_ERR_INVALID_ARG;
    if (!index_supported(hi, di, top_k)) return CSA_ERR_UNSUPPORTED;
    CSA_TRY(check_ptr(q_idx, L->total_q > 0));
    CSA_TRY(check_ptr(k_idx, L->total_csa > 0));
    if (L->total_q > 0 && !idx_out) return CSA_ERR_INVALID_ARG;
    if (score_out && (reinterpret_cast<uintptr_t>(score_out) & 3u)) return CSA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(idx_out) & 3u) return CSA_ERR_INVALID_ARG;
    return CSA_OK;
}

// The FP8 indexer's key arrays (codes [total_csa, d_idx] bytes, scales
// [total_csa] fp32) and its row-length limit.
csa_status_t check_fp8_keys(const csa_layout *L, const uint8_t *k_fp8, const float *k_scale, int ratio)
{
    const bool any = L->total_csa > 0;
    CSA_TRY(check_ptr(k_fp8, any));
    if (any && (!k_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3u))) return CSA_ERR_INVALID_ARG;
    if (L->max_kv_len / ratio > index_fp8_max_n()) return CSA_ERR_UNSUPPORTED;
    return CSA_OK;
}

csa_status_t check_attend(const csa_layout *L, bool sparse, const csa_bf16 *q, const csa_bf16 *entries,
                          const csa_bf16 *kv, const int32_t *idx, int H, int d, int ratio, int top_k,
                          const csa_bf16 *out, const float *lse)
{
    CSA_TRY(check_layout(L, sparse, !sparse));
    if (ratio <= 0 || ratio > 1024) return CSA_ERR_INVALID_ARG;
    if (sparse && top_k <= 0) return CSA_ERR_INVALID_ARG;
    if (!attend_supported(H, d)) return CSA_ERR_UNSUPPORTED;
    const bool any_q = L->total_q > 0;
    CSA_TRY(check_ptr(q, any_q));
    CSA_TRY(check_ptr(out, any_q));
    CSA_TRY(check_ptr(kv, any_q));
    CSA_TRY(check_ptr(entries, any_q && (sparse ? L->total_csa : L->total_hca) > 0));
    if (sparse && any_q && (!idx || (reinterpret_cast<uintptr_t>(idx) & 3u))) return CSA_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return CSA_ERR_INVALID_ARG;
    return CSA_OK;
}

// Sliding-window attention over the raw tokens: the dense attention with
// every raw token as its own entry (entries = kv, ratio 1, so no raw tail)
// and only the most recent `window` entries visible.
AttendArgs swa_args(const csa_layout *L, const csa_bf16 *q, const csa_bf16 *kv, int H, int d, int window,
                           float scale, csa_bf16 *out, float *lse, void *ws, size_t ws_bytes, int *err, int num_sms)
{
    AttendArgs a = attend_args(L, false, q, kv, kv, nullptr, H, d, 1, window, scale, out, lse, ws, ws_bytes, err,
                               num_sms, num_sms);
    a.cu_ent = L->cu_kv;
    a.n_ent_rows = L->total_kv;
    return a;
}

csa_status_t check_swa(const csa_layout *L, const csa_bf16 *q, const csa_bf16 *kv, int H, int d, int window,
                              const csa_bf16 *out, const float *lse)
{
    CSA_TRY(check_layout(L, false, false));
    if (window <= 0) return CSA_ERR_INVALID_ARG;
    if (!attend_supported(H, d)) return CSA_ERR_UNSUPPORTED;
    const bool any_q = L->total_q > 0;
    CSA_TRY(check_ptr(q, any_q));
    CSA_TRY(check_ptr(out, any_q));
    CSA_TRY(check_ptr(kv, any_q));
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return CSA_ERR_INVALID_ARG;
    return CSA_OK;
}

csa_status_t compress_impl(const csa_layout *L, bool csa_side, const csa_bf16 *kv, const float *gate, int d,
                           int ratio, csa_bf16 *out, cudaStream_t st)
{
    CSA_TRY(check_layout(L, csa_side, !csa_side));
    if (!pow2(ratio) || ratio > 128) return CSA_ERR_UNSUPPORTED;
    if (d != 128 && d != 512) return CSA_ERR_UNSUPPORTED;
    CSA_TRY(check_ptr(kv, L->total_kv > 0));
    if (L->total_kv > 0 && (!gate || (reinterpret_cast<uintptr_t>(gate) & 3u))) return CSA_ERR_INVALID_ARG;
    CSA_TRY(check_ptr(out, (csa_side ? L->total_csa : L->total_hca) > 0));
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    CompressArgs a;
    std::memset(&a, 0, sizeof a);
    a.batch = L->batch;
    a.max_kv_len = L->max_kv_len;
    a.max_q_len = L->max_q_len;
    a.cu_kv = L->cu_kv;
    a.cu_q = L->cu_q;
    a.d = d;
    a.kv = kv;
    a.gate = gate;
    a.err = ds->err;
    const int64_t *cu = csa_side ? L->cu_csa : L->cu_hca;
    if (ratio <= 32) {
        a.ratio_small = ratio;
        a.cu_small = cu;
        a.out_small = out;
    } else {
        a.ratio_big = ratio;
        a.cu_big = cu;
        a.out_big = out;
    }
    if (!compress_supported(d, a.ratio_small, a.ratio_big)) return CSA_ERR_UNSUPPORTED;
    if (L->total_q == 0) return CSA_OK;
    return from_cuda(launch_compress(a, st));
}

// SMs of the two attention branches, which run at the same time in a decode
// step: in proportion to their largest key counts, the sparse branch's keys
// counted twice (it starts only after the top-k selection, while the dense
// branch starts after the key scan), so that both split-KV grids fit on the
// GPU together and finish at about the same time.
void hybrid_shares(const csa_hybrid_params *p, int num_sms, int *sparse_share, int *dense_share)
{
    const csa_layout *L = &p->layout;
    const int64_t Lmax = L->max_kv_len;
    int64_t ks = Lmax / p->ratio_csa;
    if (ks > p->top_k) ks = p->top_k;
    ks += p->ratio_csa - 1;
    int64_t kd = Lmax / p->ratio_hca + p->ratio_hca - 1;
    ks = ks < Lmax ? ks : Lmax;
    kd = kd < Lmax ? kd : Lmax;
    ks *= 2;
    const int n = num_sms > 0 ? num_sms : 148;
    int64_t d = ks + kd > 0 ? (int64_t)n * kd / (ks + kd) : n / 2;
    // The dense branch starts while the top-k select runs.  For rows longer
    // than 131072 entries (decode-sized batches) the select takes 16 CTAs of
    // 1024 threads per query, each filling an SM's registers: the dense
    // branch gets the SMs they leave.
    const int64_t max_n = Lmax / p->ratio_csa;
    if (L->total_q < 1024 && max_n > 131072 && max_n <= 262144) {
        const int64_t free_sms = (int64_t)n - 16 * L->total_q;
        if (d > free_sms) d = free_sms;
    }
    if (d < n / 8) d = n / 8;
    if (d > n - n / 8) d = n - n / 8;
    *dense_share = (int)d;
    *sparse_share = n - (int)d;
}

size_t hybrid_ws_parts(const csa_hybrid_params *p, size_t *idx_ws, size_t *sp_ws, size_t *hc_ws, int num_sms)
{
    int sh_s = 0, sh_d = 0;
    hybrid_shares(p, num_sms, &sh_s, &sh_d);
    const csa_layout *L = &p->layout;
    IndexArgs ia = index_args(L, p->q_idx, p->k_idx, p->n_heads_idx, p->d_idx, p->ratio_csa, p->top_k, nullptr,
                              nullptr, nullptr, 0, nullptr);
    AttendArgs sa = attend_args(L, true, p->q, p->csa_cache, p->kv, p->idx_out, p->n_heads, p->d,
                                p->ratio_csa, p->top_k, p->scale, nullptr, nullptr, nullptr, 0, nullptr, num_sms,
                                sh_s);
    sa.idx = reinterpret_cast<const int32_t *>(1);   // sparse plan
    AttendArgs ha = attend_args(L, false, p->q, p->hca_cache, p->kv, nullptr, p->n_heads, p->d, p->ratio_hca,
                                0, p->scale, nullptr, nullptr, nullptr, 0, nullptr, num_sms, sh_d);
    *idx_ws = align_ws((p->flags & CSA_INDEX_FP8) ? index_fp8_workspace_bytes(ia) : index_workspace_bytes(ia));
    *sp_ws = align_ws(attend_workspace_bytes(sa));
    *hc_ws = align_ws(attend_workspace_bytes(ha));
    return *idx_ws + *sp_ws + *hc_ws;
}

}  // namespace

bool timing_enabled() { return g_timing.load(std::memory_order_relaxed); }

void timing_record(const char *name, cudaEvent_t start, cudaEvent_t stop)
{
    std::lock_guard<std::mutex> lock(g_timing_mu);
    g_pending.push_back(Pending{name, start, stop});
}

cudaError_t ensure_smem_fn(const void *kern, size_t smem)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_smem_mu);
    auto key = std::make_pair(dev, kern);
    auto it = g_smem.find(key);
    if (it != g_smem.end() && it->second >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) g_smem[key] = smem;
    return e;
}

}  // namespace csa

using namespace csa;

extern "C" {

csa_status_t csa_compress(const csa_layout *layout, const csa_bf16 *kv, const float *gate, int d, int ratio,
                          csa_bf16 *out, csa_stream_t stream)
{
    return compress_impl(layout, true, kv, gate, d, ratio, out, reinterpret_cast<cudaStream_t>(stream));
}

csa_status_t hca_compress(const csa_layout *layout, const csa_bf16 *kv, const float *gate, int d, int ratio,
                          csa_bf16 *out, csa_stream_t stream)
{
    return compress_impl(layout, false, kv, gate, d, ratio, out, reinterpret_cast<cudaStream_t>(stream));
}

csa_status_t csa_quantize_index_keys(const csa_layout *layout, const csa_bf16 *k_idx, int d_idx, uint8_t *k_fp8,
                                     float *k_scale, csa_stream_t stream)
{
    CSA_TRY(check_layout(layout, true, false));
    if (d_idx != 32 && d_idx != 64 && d_idx != 128) return CSA_ERR_UNSUPPORTED;
    const int64_t rows = layout->total_csa;
    CSA_TRY(check_ptr(k_idx, rows > 0));
    CSA_TRY(check_ptr(k_fp8, rows > 0));
    if (rows > 0 && (!k_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3u))) return CSA_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    return from_cuda(launch_quantize_index_keys(k_idx, rows, d_idx, k_fp8, k_scale,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

csa_status_t csa_quantize_index_keys_closed(const csa_layout *layout, const csa_bf16 *k_idx, int d_idx, int ratio,
                                            uint8_t *k_fp8, float *k_scale, csa_stream_t stream)
{
    CSA_TRY(check_layout(layout, true, false));
    if (ratio <= 0 || ratio > 1024) return CSA_ERR_INVALID_ARG;
    if (d_idx != 32 && d_idx != 64 && d_idx != 128) return CSA_ERR_UNSUPPORTED;
    const bool any = layout->total_q > 0 && layout->total_csa > 0;
    CSA_TRY(check_ptr(k_idx, any));
    CSA_TRY(check_ptr(k_fp8, any));
    if (any && (!k_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3u))) return CSA_ERR_INVALID_ARG;
    if (!any) return CSA_OK;
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    return from_cuda(launch_quantize_closed_keys(layout->batch, layout->cu_kv, layout->cu_q, layout->cu_csa,
                                                 layout->total_q, ratio, k_idx, d_idx, k_fp8, k_scale, ds->err,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

csa_status_t lightning_index_topk_fp8(const csa_layout *layout, const csa_bf16 *q_idx, const uint8_t *k_fp8,
                                      const float *k_scale, int n_heads_idx, int d_idx, int ratio, int top_k,
                                      int32_t *idx_out, float *score_out, void *ws, size_t ws_bytes,
                                      csa_stream_t stream)
{
    CSA_TRY(check_index(layout, q_idx, reinterpret_cast<const csa_bf16 *>(k_fp8), n_heads_idx, d_idx, ratio, top_k,
                        idx_out, score_out));
    CSA_TRY(check_fp8_keys(layout, k_fp8, k_scale, ratio));
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    IndexArgs a = index_args(layout, q_idx, nullptr, n_heads_idx, d_idx, ratio, top_k, idx_out, score_out, ws,
                             ws_bytes, ds->err);
    a.fp8 = true;
    a.k_fp8 = k_fp8;
    a.k_scale = k_scale;
    const size_t need = index_fp8_workspace_bytes(a);
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return CSA_ERR_WORKSPACE;
    return from_cuda(launch_index_topk(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status_t csa_index_fp8_workspace_size(const csa_layout *layout, int n_heads_idx, int d_idx, int ratio, int top_k,
                                          size_t *bytes)
{
    if (!bytes) return CSA_ERR_INVALID_ARG;
    CSA_TRY(check_layout(layout, true, false));
    if (ratio <= 0 || top_k <= 0) return CSA_ERR_INVALID_ARG;
    if (!index_supported(n_heads_idx, d_idx, top_k)) return CSA_ERR_UNSUPPORTED;
    if (layout->max_kv_len / ratio > index_fp8_max_n()) return CSA_ERR_UNSUPPORTED;
    IndexArgs a = index_args(layout, nullptr, nullptr, n_heads_idx, d_idx, ratio, top_k, nullptr, nullptr, nullptr,
                             0, nullptr);
    *bytes = align_ws(index_fp8_workspace_bytes(a));
    return CSA_OK;
}

csa_status_t csa_index_workspace_size(const csa_layout *layout, int n_heads_idx, int d_idx, int ratio, int top_k,
                                      size_t *bytes)
{
    if (!bytes) return CSA_ERR_INVALID_ARG;
    CSA_TRY(check_layout(layout, true, false));
    if (ratio <= 0 || top_k <= 0) return CSA_ERR_INVALID_ARG;
    if (!index_supported(n_heads_idx, d_idx, top_k)) return CSA_ERR_UNSUPPORTED;
    IndexArgs a = index_args(layout, nullptr, nullptr, n_heads_idx, d_idx, ratio, top_k, nullptr, nullptr, nullptr,
                             0, nullptr);
    *bytes = align_ws(index_workspace_bytes(a));
    return CSA_OK;
}

csa_status_t lightning_index_topk(const csa_layout *layout, const csa_bf16 *q_idx, const csa_bf16 *k_idx,
                                  int n_heads_idx, int d_idx, int ratio, int top_k, int32_t *idx_out,
                                  float *score_out, void *ws, size_t ws_bytes, csa_stream_t stream)
{
    CSA_TRY(check_index(layout, q_idx, k_idx, n_heads_idx, d_idx, ratio, top_k, idx_out, score_out));
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    IndexArgs a = index_args(layout, q_idx, k_idx, n_heads_idx, d_idx, ratio, top_k, idx_out, score_out, ws,
                             ws_bytes, ds->err);
    const size_t need = index_workspace_bytes(a);
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return CSA_ERR_WORKSPACE;
    return from_cuda(launch_index_topk(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status_t lightning_index_topk_static(const csa_layout *layout, const csa_bf16 *q_idx, const csa_bf16 *k_idx,
                                         int n_heads_idx, int d_idx, int ratio, int top_k, int32_t *idx_out,
                                         float *score_out, csa_stream_t stream)
{
    CSA_TRY(check_index(layout, q_idx, k_idx, n_heads_idx, d_idx, ratio, top_k, idx_out, score_out));
    IndexArgs a = index_args(layout, q_idx, k_idx, n_heads_idx, d_idx, ratio, top_k, idx_out, score_out, nullptr, 0,
                             nullptr);
    // the problem must fit the library-owned scratch (checked before any CUDA call)
    if (index_static_need_bytes(a) > kIndexStaticScratchBytes) return CSA_ERR_WORKSPACE;
    int *err = nullptr;
    CSA_TRY(error_word(&err));
    void *scratch = nullptr;
    if (index_static_scratch(&scratch) != cudaSuccess) return CSA_ERR_CUDA;
    a.ws = scratch;
    a.ws_bytes = kIndexStaticScratchBytes;
    a.err = err;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // histograms and counters start at zero whatever an earlier (possibly failed) call left there
    const size_t zero = index_static_zero_bytes(a);
    if (zero > 0 && cudaMemsetAsync(scratch, 0, zero, st) != cudaSuccess) return CSA_ERR_CUDA;
    return from_cuda(launch_index_topk(a, st));
}

csa_status_t csa_attend_workspace_size(const csa_layout *layout, int n_heads, int d, int ratio, int top_k,
                                       size_t *bytes)
{
    if (!bytes) return CSA_ERR_INVALID_ARG;
    const bool sparse = top_k > 0;
    CSA_TRY(check_layout(layout, sparse, !sparse));
    if (ratio <= 0 || top_k < 0) return CSA_ERR_INVALID_ARG;
    if (!attend_supported(n_heads, d)) return CSA_ERR_UNSUPPORTED;
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    AttendArgs a = attend_args(layout, sparse, nullptr, nullptr, nullptr,
                               sparse ? reinterpret_cast<const int32_t *>(1) : nullptr, n_heads, d, ratio, top_k,
                               1.f, nullptr, nullptr, nullptr, 0, nullptr, ds->num_sms, ds->num_sms);
    *bytes = align_ws(attend_workspace_bytes(a));
    return CSA_OK;
}

csa_status_t sparse_mqa_attend(const csa_layout *layout, const csa_bf16 *q, const csa_bf16 *csa_entries,
                               const csa_bf16 *kv, const int32_t *idx, int n_heads, int d, int ratio, int top_k,
                               float scale, csa_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                               csa_stream_t stream)
{
    CSA_TRY(check_attend(layout, true, q, csa_entries, kv, idx, n_heads, d, ratio, top_k, out, lse));
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    AttendArgs a = attend_args(layout, true, q, csa_entries, kv, idx, n_heads, d, ratio, top_k, scale,
                               out, lse, ws, ws_bytes, ds->err, ds->num_sms, ds->num_sms);
    const size_t need = attend_workspace_bytes(a);
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return CSA_ERR_WORKSPACE;
    return from_cuda(launch_attend(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status_t hca_dense_attend(const csa_layout *layout, const csa_bf16 *q, const csa_bf16 *hca_entries,
                              const csa_bf16 *kv, int n_heads, int d, int ratio, float scale, csa_bf16 *out,
                              float *lse, void *ws, size_t ws_bytes, csa_stream_t stream)
{
    CSA_TRY(check_attend(layout, false, q, hca_entries, kv, nullptr, n_heads, d, ratio, 0, out, lse));
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    AttendArgs a = attend_args(layout, false, q, hca_entries, kv, nullptr, n_heads, d, ratio, 0, scale,
                               out, lse, ws, ws_bytes, ds->err, ds->num_sms, ds->num_sms);
    const size_t need = attend_workspace_bytes(a);
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return CSA_ERR_WORKSPACE;
    return from_cuda(launch_attend(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status_t swa_workspace_size(const csa_layout *layout, int n_heads, int d, int window, size_t *bytes)
{
    if (!bytes) return CSA_ERR_INVALID_ARG;
    CSA_TRY(check_layout(layout, false, false));
    if (window <= 0) return CSA_ERR_INVALID_ARG;
    if (!attend_supported(n_heads, d)) return CSA_ERR_UNSUPPORTED;
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    const AttendArgs a = swa_args(layout, nullptr, nullptr, n_heads, d, window, 1.f, nullptr, nullptr, nullptr, 0,
                                  nullptr, ds->num_sms);
    *bytes = align_ws(attend_workspace_bytes(a));
    return CSA_OK;
}

csa_status_t swa_attend(const csa_layout *layout, const csa_bf16 *q, const csa_bf16 *kv, int n_heads, int d,
                        int window, float scale, csa_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                        csa_stream_t stream)
{
    CSA_TRY(check_swa(layout, q, kv, n_heads, d, window, out, lse));
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    const AttendArgs a = swa_args(layout, q, kv, n_heads, d, window, scale, out, lse, ws, ws_bytes, ds->err,
                                  ds->num_sms);
    const size_t need = attend_workspace_bytes(a);
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return CSA_ERR_WORKSPACE;
    return from_cuda(launch_attend(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status_t csa_inverse_rope(const csa_layout *layout, csa_bf16 *out, int n_heads, int d, int d_rope, float base,
                              csa_stream_t stream)
{
    CSA_TRY(check_layout(layout, false, false));
    if (n_heads <= 0 || !(base > 0.f) || !std::isfinite(base)) return CSA_ERR_INVALID_ARG;
    if (!inverse_rope_supported(d, d_rope)) return CSA_ERR_UNSUPPORTED;
    CSA_TRY(check_ptr(out, layout->total_q > 0));
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    RopeArgs a;
    a.batch = layout->batch;
    a.total_q = layout->total_q;
    a.cu_kv = layout->cu_kv;
    a.cu_q = layout->cu_q;
    a.n_heads = n_heads;
    a.d = d;
    a.d_rope = d_rope;
    a.base = (double)base;
    a.out = reinterpret_cast<uint16_t *>(out);
    a.err = ds->err;
    a.num_sms = ds->num_sms;
    return from_cuda(launch_inverse_rope(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status_t csa_workspace_size(const csa_hybrid_params *p, size_t *bytes)
{
    if (!p || !bytes) return CSA_ERR_INVALID_ARG;
    CSA_TRY(check_layout(&p->layout, true, true));
    if (p->ratio_csa <= 0 || p->ratio_hca <= 0 || p->top_k <= 0) return CSA_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    size_t a, b, c;
    *bytes = hybrid_ws_parts(p, &a, &b, &c, ds->num_sms);
    return CSA_OK;
}

csa_status_t hybrid_attend(const csa_hybrid_params *p, csa_stream_t stream_)
{
    if (!p || p->reserved != 0) return CSA_ERR_INVALID_ARG;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
    const csa_layout *L = &p->layout;
    const bool fp8 = (p->flags & CSA_INDEX_FP8) != 0;
    if (p->flags & ~(CSA_SKIP_COMPRESS | CSA_INDEX_FP8)) return CSA_ERR_INVALID_ARG;
    // with FP8 keys the bf16 keys are not read (a non-null placeholder passes the shared checks)
    CSA_TRY(check_index(L, p->q_idx, fp8 ? reinterpret_cast<const csa_bf16 *>(p->k_idx_fp8) : p->k_idx,
                        p->n_heads_idx, p->d_idx, p->ratio_csa, p->top_k, p->idx_out, p->score_out));
    if (fp8) CSA_TRY(check_fp8_keys(L, p->k_idx_fp8, p->k_idx_scale, p->ratio_csa));
    CSA_TRY(check_attend(L, true, p->q, p->csa_cache, p->kv, p->idx_out, p->n_heads, p->d, p->ratio_csa, p->top_k,
                         p->o_csa, p->lse_csa));
    CSA_TRY(check_attend(L, false, p->q, p->hca_cache, p->kv, nullptr, p->n_heads, p->d, p->ratio_hca, 0, p->o_hca,
                         p->lse_hca));
    const bool compress = !(p->flags & CSA_SKIP_COMPRESS);
    if (compress) {
        if (!pow2(p->ratio_csa) || p->ratio_csa > 128 || !pow2(p->ratio_hca) || p->ratio_hca > 128)
            return CSA_ERR_UNSUPPORTED;
        CSA_TRY(check_ptr(p->kv, L->total_kv > 0));
        if (L->total_kv > 0 && !p->gate) return CSA_ERR_INVALID_ARG;
        CSA_TRY(check_ptr(p->csa_cache, L->total_csa > 0));
        CSA_TRY(check_ptr(p->hca_cache, L->total_hca > 0));
    }
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    size_t w_idx, w_sp, w_hc;
    const size_t need = hybrid_ws_parts(p, &w_idx, &w_sp, &w_hc, ds->num_sms);
    if (need > 0 && (!p->ws || p->ws_bytes < need || !aligned16(p->ws))) return CSA_ERR_WORKSPACE;
    if (L->total_q == 0) return CSA_OK;
    char *ws = static_cast<char *>(p->ws);

    Helper *hp = nullptr;
    CSA_TRY(helper_for(st, &hp));
    std::unique_lock<std::mutex> issue_lock;
    if (hp) issue_lock = std::unique_lock<std::mutex>(hp->mu);

    // Streams.  The caller's stream `st` runs the compression and the CSA
    // branch (indexer, top-k, sparse attention) as one chain of dependent
    // launches: the key scan reads no compressed entry and overlaps the
    // compression, each later kernel starts while its predecessor finishes.
    // The helper stream of (device, st) runs the HCA branch once the key scan
    // (the part of the indexer that fills the GPU) is done, so it overlaps the
    // top-k selection and the sparse attention.  Without a helper (the table
    // is full) the HCA branch follows the CSA branch on `st`.
    if (hp) {
        if (cudaEventRecord(hp->fork, st) != cudaSuccess) return CSA_ERR_CUDA;
        if (cudaStreamWaitEvent(hp->aux, hp->fork, 0) != cudaSuccess) return CSA_ERR_CUDA;
    }

    // a1: compression of the blocks closed by this call's query positions.  The
    // fused kernel runs inside the index call (after the key scan on the
    // key-scan paths, ahead of the indexer otherwise); the fallback runs first.
    csa_status_t s_c = CSA_OK;
    CompressArgs ca;
    std::memset(&ca, 0, sizeof ca);
    const bool fused = compress && compress_supported(p->d, p->ratio_csa, p->ratio_hca);
    if (fused) {
        ca.batch = L->batch;
        ca.max_kv_len = L->max_kv_len;
        ca.max_q_len = L->max_q_len;
        ca.cu_kv = L->cu_kv;
        ca.cu_q = L->cu_q;
        ca.d = p->d;
        ca.kv = p->kv;
        ca.gate = p->gate;
        ca.err = ds->err;
        ca.ratio_small = p->ratio_csa;
        ca.cu_small = L->cu_csa;
        ca.out_small = p->csa_cache;
        ca.ratio_big = p->ratio_hca;
        ca.cu_big = L->cu_hca;
        ca.out_big = p->hca_cache;
    } else if (compress) {
        s_c = compress_impl(L, true, p->kv, p->gate, p->d, p->ratio_csa, p->csa_cache, st);
        if (s_c == CSA_OK) s_c = compress_impl(L, false, p->kv, p->gate, p->d, p->ratio_hca, p->hca_cache, st);
    }

    // a2 + a3 (records sdone once every key is scored and the compression is done)
    if (s_c == CSA_OK) {
        IndexArgs ia = index_args(L, p->q_idx, p->k_idx, p->n_heads_idx, p->d_idx, p->ratio_csa, p->top_k,
                                  p->idx_out, p->score_out, w_idx ? ws : nullptr, w_idx, ds->err);
        ia.scan_done = hp ? hp->sdone : nullptr;
        ia.pdl = compress && !fused;   // behind the fallback compression
        ia.compress = fused ? &ca : nullptr;
        if (fp8) {
            ia.fp8 = true;
            ia.k_fp8 = p->k_idx_fp8;
            ia.k_scale = p->k_idx_scale;
        }
        s_c = from_cuda(launch_index_topk(ia, st));
    } else if (hp) {
        cudaEventRecord(hp->sdone, st);
    }

    // the SM shares that sized the workspace (kept when the branches run one after the other)
    int sh_s = 0, sh_d = 0;
    hybrid_shares(p, ds->num_sms, &sh_s, &sh_d);
    const AttendArgs ha = attend_args(L, false, p->q, p->hca_cache, p->kv, nullptr, p->n_heads, p->d, p->ratio_hca,
                                      0, p->scale, p->o_hca, p->lse_hca, w_hc ? ws + w_idx + w_sp : nullptr, w_hc,
                                      ds->err, ds->num_sms, sh_d);

    // a5 on the helper stream, behind the compression and the key scan
    bool c1 = true;
    csa_status_t s_h = s_c;
    if (hp) {
        c1 = cudaStreamWaitEvent(hp->aux, hp->sdone, 0) == cudaSuccess;
        if (s_h == CSA_OK) s_h = from_cuda(launch_attend(ha, hp->aux));
    }

    // a4, launched behind the selection
    if (s_c == CSA_OK) {
        AttendArgs sa = attend_args(L, true, p->q, p->csa_cache, p->kv, p->idx_out, p->n_heads, p->d,
                                    p->ratio_csa, p->top_k, p->scale, p->o_csa, p->lse_csa,
                                    w_sp ? ws + w_idx : nullptr, w_sp, ds->err, ds->num_sms, sh_s);
        sa.pdl = true;
        s_c = from_cuda(launch_attend(sa, st));
    }
    if (!hp) {
        // a5 after a4 on the caller's stream
        if (s_c == CSA_OK) s_h = from_cuda(launch_attend(ha, st));
        if (s_c != CSA_OK) return s_c;
        return s_h;
    }
    // join (always, so the helper stream never dangles inside a capture)
    const bool j1 = cudaEventRecord(hp->join, hp->aux) == cudaSuccess;
    const bool j2 = cudaStreamWaitEvent(st, hp->join, 0) == cudaSuccess;
    if (s_c != CSA_OK) return s_c;
    if (s_h != CSA_OK) return s_h;
    return (c1 && j1 && j2) ? CSA_OK : CSA_ERR_CUDA;
}

csa_status_t csa_workspace_init(void *ws, size_t ws_bytes, csa_stream_t stream)
{
    if (ws_bytes == 0) return CSA_OK;
    if (!ws) return CSA_ERR_INVALID_ARG;
    return cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? CSA_OK
                                                                                                  : CSA_ERR_CUDA;
}

const char *csa_status_string(csa_status_t s)
{
    switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported size";
    case CSA_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA_ERR_CUDA: return "CUDA error";
    case CSA_ERR_TIMEOUT: return "device wait timed out";
    case CSA_ERR_DEVICE: return "device-side layout or index error";
    default: return "unknown status";
    }
}

csa_status_t csa_check_device_error(csa_stream_t stream, csa_status_t *device_status)
{
    if (!device_status) return CSA_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    CSA_TRY(device_state(&ds));
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return CSA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ds->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return CSA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(ds->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return CSA_ERR_CUDA;
    *device_status = static_cast<csa_status_t>(v);
    return CSA_OK;
}

int csa_version(void) { return 130; }   // 1.1: FP8 indexer keys (.1: the closed-rows quantiser); 1.2: swa_attend; 1.3: csa_inverse_rope

csa_status_t csa_timing_enable(int enable)
{
    g_timing.store(enable != 0);
    return CSA_OK;
}

int csa_timing_read(int cap, const char **names, int64_t *launches, double *total_ms)
{
    std::lock_guard<std::mutex> lock(g_timing_mu);
    for (auto &pd : g_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(pd.b) == cudaSuccess && cudaEventElapsedTime(&ms, pd.a, pd.b) == cudaSuccess) {
            auto &acc = g_timing_acc[pd.name];
            acc.first += 1;
            acc.second += ms;
        }
        cudaEventDestroy(pd.a);
        cudaEventDestroy(pd.b);
    }
    g_pending.clear();
    int i = 0;
    for (auto &kv : g_timing_acc) {
        if (i < cap) {
            if (names) names[i] = kv.first.c_str();
            if (launches) launches[i] = kv.second.first;
            if (total_ms) total_ms[i] = kv.second.second;
        }
        i++;
    }
    return i;
}

void csa_timing_reset(void)
{
    std::lock_guard<std::mutex> lock(g_timing_mu);
    for (auto &pd : g_pending) {
        cudaEventDestroy(pd.a);
        cudaEventDestroy(pd.b);
    }
    g_pending.clear();
    g_timing_acc.clear();
}

}  // extern "C"
