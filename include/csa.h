/*
 * csa.h -- C ABI of the B300 (sm_103a) CSA + HCA hybrid compressed attention.
 *
 * The operations follow the DeepSeek-V4 hybrid attention as described in
 * "DeepSeek-V4 core architecture" (gitcode.csdn.net article):
 *   §2.2 "CSA: compressed sparse attention"
 *        step 1  token-level compression: every m adjacent tokens' KV become
 *                one entry, weighted by learnable softmax-normalised weights;
 *        step 2  lightning indexer: a light scorer rates each query against
 *                every compressed entry and only the top-k entries are kept;
 *        step 3  multi-query attention with shared KV: each selected entry is
 *                both key and value, and all query heads share it;
 *   §2.3 "HCA: heavily compressed attention": 128 tokens per entry, dense
 *        attention over all entries, no selection; CSA and HCA alternate
 *        across layers.
 * and "DeepSeek V4's architecture debt chain" (vendordeep.com),
 * "Constraint 1 -> Innovation 1" (many tokens' KV weighted into one
 * compressed token at up to 128x; the "reverse RoPE" correction of the
 * attention output: csa_inverse_rope).  Sliding-window attention over the
 * raw tokens (swa_attend) follows §3.2 "SWA sliding-window attention" of the
 * bjdmk.com.cn DeepSeek-V4 walkthrough.
 *
 * Where the pages leave a step open this library takes these readings:
 *   - one scalar gate logit per token; the weights of a block are the
 *     softmax of its tokens' logits; blocks are non-overlapping and aligned
 *     at position 0; a trailing partial block has no entry;
 *   - the indexer score of entry j for the query at t is the fp32 sum over
 *     indexer heads h of q_{t,h} . k_j, with one indexer key per entry;
 *   - an entry becomes visible only once its block is complete: entry j of
 *     ratio m is visible to position t iff (j+1)*m <= t+1;
 *   - each query also attends to the raw tokens of its own incomplete
 *     block: r(t) = (t+1) mod m tokens, positions t-r(t)+1 .. t;
 *   - top-k keeps the min(k, n(t)) highest scores, ties to the lower entry
 *     index, and returns them in ascending index order padded with -1.
 *
 * Conventions shared by every call:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, row-major,
 *     contiguous and 16-byte aligned.  bf16 tensors are passed as their raw
 *     16-bit patterns (csa_bf16).  Rows of all sequences are packed.
 *   - The library allocates no device memory.  Scratch space is the caller's
 *     workspace (ws, ws_bytes), sized by the *_workspace_size calls.  It must
 *     be zero-filled once before its first use (csa_workspace_init does
 *     that).  It holds counters and histograms, which every call that
 *     returns CSA_OK leaves at zero again (or which the call resets itself),
 *     and scratch (candidate lists, partial outputs), which calls overwrite
 *     and leave as they are.  Scratch of an indexer call with 1024 or more
 *     queries lies where a call with fewer keeps its histograms: after such
 *     a call (lightning_index_topk, or hybrid_attend), zero the workspace
 *     again before a call with fewer queries uses it, and zero it again
 *     after any call that failed.  Calls on the same side of that divide
 *     (every decode step of a serving loop, say) reuse it as it is.
 *   - Every call is asynchronous on the given stream and does not
 *     synchronise.  Calls that share one workspace must not overlap in time.
 *   - Every call returns a csa_status_t.  Argument errors are detected on the
 *     host before anything is launched.  Layout inconsistencies that can only
 *     be seen on the device (for example an entry count that does not equal
 *     floor(L/m), or an index that is not visible) set the device error word,
 *     which csa_check_device_error reads; the offending rows are skipped.
 *   - hybrid_attend runs its two branches concurrently on the caller's
 *     stream and one helper stream.  The first hybrid_attend call on a given
 *     (device, stream) pair creates that pair's helper stream and three
 *     events, kept until the process exits; make that first call outside
 *     any CUDA graph capture.  Calls on different streams (or captured into
 *     different graphs) use different helpers and do not interfere; calls
 *     on one stream are issued one at a time (the library holds a host lock
 *     per pair while it issues a call).  Past 256 pairs, a call on a new
 *     pair runs the two branches one after the other on its own stream.
 *   - The library keeps per-device state (the device error word's address,
 *     the static scratch's address, the helper streams).  It must not be
 *     used across a device reset (cudaDeviceReset or a primary-context
 *     reset) in the same process.
 *   - Inside a call, kernels that follow another kernel of the same call may
 *     be launched with programmatic dependent launch (they start early and
 *     wait on the device for their predecessor).  The first kernel of every
 *     call waits for all earlier work on the caller's stream in the ordinary
 *     way.
 */
#ifndef CSA_H
#define CSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *csa_stream_t;

/* Raw bf16 bit pattern. */
typedef uint16_t csa_bf16;

typedef enum csa_status {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARG = 1,   /* bad pointer, size or layout value (host check) */
    CSA_ERR_UNSUPPORTED = 2,   /* a size this build has no kernel for */
    CSA_ERR_WORKSPACE = 3,     /* ws missing or smaller than required */
    CSA_ERR_CUDA = 4,          /* a CUDA runtime call or a launch failed */
    CSA_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out */
    CSA_ERR_DEVICE = 6         /* device: layout inconsistency / invalid index */
} csa_status_t;

/*
 * Packed variable-length batch.  Sequence b (0 <= b < batch) has
 * L_b = cu_kv[b+1] - cu_kv[b] tokens at rows cu_kv[b] .. of the token
 * tensors, n_q,b = cu_q[b+1] - cu_q[b] queries at rows cu_q[b] .. of the
 * query tensors, and its compressed entries at rows cu_csa[b] .. and
 * cu_hca[b] .. of the entry tensors.  The queries of a sequence are its
 * LAST n_q,b positions: L_b - n_q,b .. L_b - 1 (n_q,b = L_b for a prefill,
 * 1 for a decode step).  cu_csa[b+1] - cu_csa[b] must equal floor(L_b /
 * ratio_csa) and likewise for cu_hca with ratio_hca.  The cu_* arrays are
 * int64 device arrays of batch+1 elements starting at 0; the totals and
 * maxima are host copies of what they imply (used to size grids without a
 * device read).  A call that does not use a given array may pass NULL.
 */
typedef struct csa_layout {
    int32_t batch;
    int32_t max_kv_len;        /* max over b of L_b */
    int32_t max_q_len;         /* max over b of n_q,b */
    int32_t reserved;          /* must be 0 */
    const int64_t *cu_kv;
    const int64_t *cu_q;
    const int64_t *cu_csa;
    const int64_t *cu_hca;
    int64_t total_kv;          /* cu_kv[batch] */
    int64_t total_q;           /* cu_q[batch] */
    int64_t total_csa;         /* cu_csa[batch] */
    int64_t total_hca;         /* cu_hca[batch] */
} csa_layout;

/* ---------------------------------------------------------------------------
 * Token-level compression (§2.2 step 1 with ratio m = 4; §2.3 with m = 128).
 *
 * For every block j whose last token is a query position of its sequence
 * (position >= L_b - n_q,b), writes
 *     out[cu_*[b] + j] = sum_{t in block j} softmax_block(gate)_t * kv[t]
 * computed in fp32 and rounded to bf16 once.  With n_q = L (prefill) that is
 * every complete block; with n_q = 1 (decode) it is the block completed by
 * the newest token, if any.  Rows of `out` for other blocks are not touched.
 *   kv    [total_kv, d] bf16     per-token KV vectors
 *   gate  [total_kv]    fp32     per-token gate logits
 *   out   [total_csa, d] bf16 (csa_compress, packed by cu_csa)
 *         [total_hca, d] bf16 (hca_compress, packed by cu_hca)
 *   d     128 or 512;  ratio a power of two in 1 .. 128.
 * ------------------------------------------------------------------------- */
csa_status_t csa_compress(const csa_layout *layout, const csa_bf16 *kv, const float *gate,
                          int d, int ratio, csa_bf16 *out, csa_stream_t stream);
csa_status_t hca_compress(const csa_layout *layout, const csa_bf16 *kv, const float *gate,
                          int d, int ratio, csa_bf16 *out, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Lightning indexer + top-k (§2.2 step 2).
 *
 * For each query row i (position t of sequence b) over the visible entries
 * j < n(t) = floor((t+1)/ratio):
 *     s(i, j) = fp32 sum_{h < n_heads_idx} q_idx[i, h, :] . k_idx[cu_csa[b] + j, :]
 * and writes the top min(top_k, n(t)) entries by (score desc, index asc) to
 * idx_out[i, 0 .. top_k) as sequence-local entry indices in ascending
 * order, padded with -1.  score_out (nullable) receives the fp32 score of
 * each returned index (padding slots: -inf).
 *   q_idx  [total_q, n_heads_idx, d_idx] bf16
 *   k_idx  [total_csa, d_idx]            bf16   one key per CSA entry
 *   (n_heads_idx, d_idx) in {(2,32), (4,64)} or any n_heads_idx <= 16 with
 *   d_idx in {32, 64, 128};  1 <= top_k <= 2048.
 * The full score matrix is never written out: decode-sized batches keep one
 * score row per query in the workspace; prefill-sized batches stream the
 * keys once per 16 queries and keep only candidate entries (about 2k per
 * query) in the workspace.
 * ------------------------------------------------------------------------- */
csa_status_t lightning_index_topk(const csa_layout *layout, const csa_bf16 *q_idx,
                                  const csa_bf16 *k_idx, int n_heads_idx, int d_idx,
                                  int ratio, int top_k, int32_t *idx_out, float *score_out,
                                  void *ws, size_t ws_bytes, csa_stream_t stream);
csa_status_t csa_index_workspace_size(const csa_layout *layout, int n_heads_idx, int d_idx,
                                      int ratio, int top_k, size_t *bytes);

/* ---------------------------------------------------------------------------
 * lightning_index_topk without a caller workspace.  The paper has no
 * counterpart: this is a library convenience, not a step of the method.
 *
 * Some callers cannot allocate device memory.  Examples are a plug-in host
 * that hands a custom operation only its input and output buffers (no
 * allocator, no workspace), and a latency-critical loop that may not call
 * cudaMalloc, which can synchronise the whole device.  For them this entry
 * point computes exactly what lightning_index_topk computes (same kernels,
 * same results) and takes its scratch from a library-owned device array of
 * CSA_INDEX_STATIC_SCRATCH_BYTES (32 MiB).  That array lives in every GPU
 * that loads the library until the process exits.  This call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 *   - Arguments, layout and outputs are those of lightning_index_topk; the
 *     caller still provides q_idx, k_idx, idx_out and score_out.
 *   - A decode-sized problem whose workspace (csa_index_workspace_size)
 *     exceeds CSA_INDEX_STATIC_SCRATCH_BYTES is rejected with
 *     CSA_ERR_WORKSPACE before anything is launched.  Prefill-sized batches
 *     (total_q >= 1024, at most 32768 entries per sequence, top_k <= 1024)
 *     run with as many candidate buffers as the scratch holds (fewer CTAs
 *     than with a full workspace; the same results).
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current).  Make that first call before
 *     any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents.
 *     Each call therefore clears the histograms and counters it needs first:
 *     one cudaMemsetAsync of about 16 KiB per query of the call (a per-query
 *     histogram and counters; never more than the array) on `stream`, a
 *     memset node when the call is captured into a graph.  The workspace
 *     calls above need no such clear: their caller zero-fills the workspace
 *     once.
 *     Calls that overlap on the GPU (on different streams or host threads)
 *     race on the array and must not be issued.
 * ------------------------------------------------------------------------- */
#define CSA_INDEX_STATIC_SCRATCH_BYTES (32u << 20)
csa_status_t lightning_index_topk_static(const csa_layout *layout, const csa_bf16 *q_idx,
                                         const csa_bf16 *k_idx, int n_heads_idx, int d_idx,
                                         int ratio, int top_k, int32_t *idx_out, float *score_out,
                                         csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * FP8 indexer keys: a low-precision lightning indexer ("DeepSeek-V4 core
 * architecture", §9 "key innovations summary", table row 5: the indexer's
 * QK product is quantised, there to FP4 through quantisation-aware
 * training).  This library takes the inference-side form of that idea with
 * FP8 E4M3 keys and one scale per key row.  It is an option next to the
 * bf16 indexer above, for callers that keep the indexer keys in FP8, and
 * reads half the bytes per entry, the dominant traffic of a decode step.
 *
 * csa_quantize_index_keys turns each indexer key row j (d_idx bf16 values)
 * into FP8 E4M3 codes with one fp32 scale, all arithmetic in fp32 (IEEE
 * division and multiplication, round to nearest even):
 *     a_j = max_i |k_ji|,  inv_j = 448 / a_j,
 *     code_ji = e4m3(k_ji * inv_j)   round to nearest even, saturating at +-448,
 *     scale_j = a_j / 448            (a_j = 0: every code 0 and scale 0)
 *   k_idx   [total_csa, d_idx] bf16
 *   k_fp8   [total_csa, d_idx] E4M3 bytes;   k_scale [total_csa] fp32
 *
 * lightning_index_topk_fp8 is lightning_index_topk on the dequantised keys:
 *     s(t, j) = scale_j * sum_i (sum_h q^I_{t,h,i}) * e4m3_value(code_ji)   (fp32)
 * with the same selection rules, outputs and padding.  Rows of up to 262144
 * entries (longer: CSA_ERR_UNSUPPORTED).  Workspace from
 * csa_index_fp8_workspace_size, zero-filled, as for lightning_index_topk.
 * ------------------------------------------------------------------------- */
csa_status_t csa_quantize_index_keys(const csa_layout *layout, const csa_bf16 *k_idx, int d_idx,
                                     uint8_t *k_fp8, float *k_scale, csa_stream_t stream);
/* csa_quantize_index_keys_closed is the incremental form for decode and
 * chunked prefill: it quantises, with the same arithmetic, only the rows of
 * the entries that the layout's query positions close (the query at position
 * t closes entry (t+1)/ratio - 1 of its sequence when (t+1) is a multiple of
 * ratio; "DeepSeek-V4 core architecture", §2.2 step 1: an entry exists once
 * its m tokens do) and leaves every other row of k_fp8 and k_scale as it is.
 * ratio is the CSA ratio (1 .. 1024).  An entry count that is not L/ratio
 * sets the device error word (CSA_ERR_DEVICE) and that query's row is not
 * written. */
csa_status_t csa_quantize_index_keys_closed(const csa_layout *layout, const csa_bf16 *k_idx, int d_idx, int ratio,
                                            uint8_t *k_fp8, float *k_scale, csa_stream_t stream);
csa_status_t lightning_index_topk_fp8(const csa_layout *layout, const csa_bf16 *q_idx,
                                      const uint8_t *k_fp8, const float *k_scale,
                                      int n_heads_idx, int d_idx, int ratio, int top_k,
                                      int32_t *idx_out, float *score_out, void *ws, size_t ws_bytes,
                                      csa_stream_t stream);
csa_status_t csa_index_fp8_workspace_size(const csa_layout *layout, int n_heads_idx, int d_idx,
                                          int ratio, int top_k, size_t *bytes);

/* ---------------------------------------------------------------------------
 * Sparse shared-KV multi-query attention (§2.2 step 3).
 *
 * Query row i at position t of sequence b attends, with every one of its
 * n_heads heads, over the key set
 *     { csa_entries[cu_csa[b] + idx[i, s]] : idx[i, s] >= 0 }
 *   U { kv[cu_kv[b] + u] : t - r(t) < u <= t },  r(t) = (t+1) mod ratio,
 * each key serving as its own value:
 *     out[i, h] = sum_x softmax_x(scale * q[i, h] . x) x,
 *     lse[i, h] = ln sum_x exp(scale * q[i, h] . x)
 * idx rows are laid out as lightning_index_topk writes them: at most
 * min(top_k, n(t)) valid entries first, then -1.  An index >= n(t) is not
 * visible: it sets CSA_ERR_DEVICE and is skipped.
 *   q      [total_q, n_heads, d] bf16
 *   out    [total_q, n_heads, d] bf16;  lse [total_q, n_heads] fp32 (nullable)
 *   d in {128, 512};  n_heads in {1 .. 16} or a multiple of 64 up to 256.
 * ------------------------------------------------------------------------- */
csa_status_t sparse_mqa_attend(const csa_layout *layout, const csa_bf16 *q,
                               const csa_bf16 *csa_entries, const csa_bf16 *kv,
                               const int32_t *idx, int n_heads, int d, int ratio, int top_k,
                               float scale, csa_bf16 *out, float *lse,
                               void *ws, size_t ws_bytes, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * HCA dense shared-KV multi-query attention (§2.3).
 *
 * Like sparse_mqa_attend with the key set
 *     { hca_entries[cu_hca[b] + j] : j < floor((t+1)/ratio) }
 *   U { kv[cu_kv[b] + u] : t - r(t) < u <= t },  r(t) = (t+1) mod ratio.
 * ------------------------------------------------------------------------- */
csa_status_t hca_dense_attend(const csa_layout *layout, const csa_bf16 *q,
                              const csa_bf16 *hca_entries, const csa_bf16 *kv, int n_heads,
                              int d, int ratio, float scale, csa_bf16 *out, float *lse,
                              void *ws, size_t ws_bytes, csa_stream_t stream);

/* Workspace for one attention call (sparse: top_k > 0; dense: top_k = 0). */
csa_status_t csa_attend_workspace_size(const csa_layout *layout, int n_heads, int d, int ratio,
                                       int top_k, size_t *bytes);

/* ---------------------------------------------------------------------------
 * Sliding-window shared-KV multi-query attention over the raw tokens (the
 * bjdmk.com.cn DeepSeek-V4 walkthrough, §3.2 "SWA sliding-window attention":
 * each token attends only to a fixed window of the tokens before it, 4096 in
 * its example).  Reading: the window holds the
 * query's own token and the window - 1 tokens before it.  Query row i at
 * position t of sequence b attends over
 *     { kv[cu_kv[b] + u] : max(0, t - window + 1) <= u <= t }
 * with the output and lse of sparse_mqa_attend (each token serves as its own
 * key and value; all heads share them).  Only cu_kv and cu_q of the layout
 * are read (cu_csa / cu_hca may be NULL).
 *   q      [total_q, n_heads, d] bf16;  kv [total_kv, d] bf16
 *   out    [total_q, n_heads, d] bf16;  lse [total_q, n_heads] fp32 (nullable)
 *   window >= 1 (CSA_ERR_INVALID_ARG otherwise); d and n_heads as for
 *   sparse_mqa_attend.  The workspace (swa_workspace_size) holds split
 *   partial results; the caller owns it, and it needs no clearing.
 * ------------------------------------------------------------------------- */
csa_status_t swa_attend(const csa_layout *layout, const csa_bf16 *q, const csa_bf16 *kv,
                        int n_heads, int d, int window, float scale, csa_bf16 *out, float *lse,
                        void *ws, size_t ws_bytes, csa_stream_t stream);
csa_status_t swa_workspace_size(const csa_layout *layout, int n_heads, int d, int window,
                                size_t *bytes);

/* ---------------------------------------------------------------------------
 * Inverse-RoPE correction of an attention output ("DeepSeek V4's
 * architecture debt chain", Constraint 1 -> Innovation 1: the compressed
 * entries carry no per-token position, so the attention output is corrected
 * by an inverse rotary embedding).  The pages fix no convention; readings:
 * the last d_rope dims of each head turn, paired as (2i, 2i+1) within that
 * slice, pair i at theta_i = base^(-2i/d_rope), and the output row of the
 * query at position t (of its sequence, from cu_kv / cu_q) turns by
 * -t * theta_i:
 *     (x, y) -> (x cos phi + y sin phi, -x sin phi + y cos phi),  phi = t theta_i
 * in fp32 with the angle reduced modulo 2 pi in double precision, rounded to
 * bf16 once; every other dim is left as it is.
 *   out    [total_q, n_heads, d] bf16, corrected in place (any attention
 *          output of this library, e.g. o_hca)
 *   d % 8 == 0; d_rope % 8 == 0, 8 <= d_rope <= min(d, 512) (else
 *   CSA_ERR_UNSUPPORTED); base > 0 and finite, n_heads >= 1 (else
 *   CSA_ERR_INVALID_ARG).  No workspace.  Only cu_kv and cu_q of the layout
 *   are read.
 * ------------------------------------------------------------------------- */
csa_status_t csa_inverse_rope(const csa_layout *layout, csa_bf16 *out, int n_heads, int d, int d_rope,
                              float base, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Hybrid step (§2.3: CSA and HCA layers alternate): runs, on the same
 * inputs, compression into both caches (unless CSA_SKIP_COMPRESS), then the
 * CSA branch (indexer, top-k, sparse attention) and the HCA branch (dense
 * attention) concurrently, and returns both branches' outputs.
 * ------------------------------------------------------------------------- */
#define CSA_SKIP_COMPRESS 0x1   /* caches already hold every needed entry */
#define CSA_INDEX_FP8 0x2       /* index with k_idx_fp8 / k_idx_scale (see csa_quantize_index_keys);
                                   the codes of every entry the step can see, including those its own
                                   positions close, must be in place before the call (a decode loop runs
                                   csa_quantize_index_keys_closed on the step's layout first); k_idx
                                   is then not read */

typedef struct csa_hybrid_params {
    csa_layout layout;
    int32_t d, n_heads, n_heads_idx, d_idx;
    int32_t ratio_csa, ratio_hca, top_k, flags;
    float scale;
    int32_t reserved;          /* must be 0 */
    const csa_bf16 *kv;        /* [total_kv, d] */
    const float *gate;         /* [total_kv] */
    const csa_bf16 *q_idx;     /* [total_q, n_heads_idx, d_idx] */
    const csa_bf16 *k_idx;     /* [total_csa, d_idx] */
    const csa_bf16 *q;         /* [total_q, n_heads, d] */
    csa_bf16 *csa_cache;       /* [total_csa, d]  written by compression */
    csa_bf16 *hca_cache;       /* [total_hca, d]  written by compression */
    int32_t *idx_out;          /* [total_q, top_k] */
    float *score_out;          /* [total_q, top_k] or NULL */
    csa_bf16 *o_csa;           /* [total_q, n_heads, d] */
    float *lse_csa;            /* [total_q, n_heads] or NULL */
    csa_bf16 *o_hca;           /* [total_q, n_heads, d] */
    float *lse_hca;            /* [total_q, n_heads] or NULL */
    void *ws;
    size_t ws_bytes;
    const uint8_t *k_idx_fp8;  /* [total_csa, d_idx] E4M3 codes, with CSA_INDEX_FP8 (else NULL) */
    const float *k_idx_scale;  /* [total_csa] fp32 scales, with CSA_INDEX_FP8 (else NULL) */
} csa_hybrid_params;

csa_status_t hybrid_attend(const csa_hybrid_params *params, csa_stream_t stream);
csa_status_t csa_workspace_size(const csa_hybrid_params *params, size_t *bytes);

/* Zero-fill a workspace (cudaMemsetAsync on `stream`). */
csa_status_t csa_workspace_init(void *ws, size_t ws_bytes, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Diagnostics.
 * csa_check_device_error synchronises `stream`, then reads and clears the
 * current device's error word (CSA_OK if no kernel reported anything).
 * csa_timing_* time each kernel launch with CUDA events on the stream it
 * runs on (disabled by default; only for eager, non-captured calls).
 * ------------------------------------------------------------------------- */
const char *csa_status_string(csa_status_t status);
csa_status_t csa_check_device_error(csa_stream_t stream, csa_status_t *device_status);
int csa_version(void);

csa_status_t csa_timing_enable(int enable);
/* Per kernel name: launches and total milliseconds since the last reset.
 * Returns the number of distinct kernels; fills at most `cap` entries. */
int csa_timing_read(int cap, const char **names, int64_t *launches, double *total_ms);
void csa_timing_reset(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H */
