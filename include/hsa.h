/*
 * hsa.h -- C ABI of the B300 (sm_103a) hybrid compressed/sparse attention library.
 *
 * One attention layer of DeepSeek-V4-style long-context attention, as the
 * QbitAI article "DeepSeek V4报告太详尽了！484天换代之路全公开" describes it in
 * its section 混合注意力机制 ("hybrid attention"):
 *   - CSA: every m tokens' K/V are compressed into one entry, a light indexer
 *     scores each query against every entry, the top-k entries are attended
 *     (Multi-Query Attention, one KV head);
 *   - HCA: heavier compression (m' = 128), dense attention over all entries;
 *   - both add a sliding-window branch over the most recent raw tokens, and
 *     compressed attention is strictly causal: only complete blocks count.
 * The pages leave the compressor and the indexer open; this library fixes
 * them: an entry is a fixed weighted sum of its block (weights w[0..m-1]), the
 * indexer score is the int32 dot product of int8 vectors, top-k orders by
 * (score desc, index asc), and the selected entries and the window share one
 * softmax with logit scale `scale` (normally 1/sqrt(d)).
 *
 * Conventions (all entry points):
 *   - Every buffer argument is caller-owned DEVICE memory of the current CUDA
 *     device (or managed memory) unless stated otherwise.  Each call classifies
 *     its pointers with cudaPointerGetAttributes before it enqueues anything and
 *     refuses host memory (pageable or pinned) and other devices' memory with
 *     HSA_ERR_INVALID_ARG.  The library never allocates, frees or
 *     synchronises (except hsa_check); all work is enqueued on `stream`
 *     (a cudaStream_t; NULL is the legacy default stream).
 *   - Strides are in ELEMENTS.  The innermost (channel) dimension is
 *     contiguous.  Vector loads need 16-byte aligned base pointers and row
 *     strides that are multiples of 16 bytes; otherwise HSA_ERR_UNSUPPORTED.
 *   - Sequence lengths and positions live in device arrays, so a captured CUDA
 *     graph can be replayed with new lengths.  Host-side size arguments
 *     (N_cap, E_cap, ...) are buffer CAPACITIES and bound the launch grids.
 *   - A call returns HSA_OK once its kernels are enqueued.  Argument errors
 *     return before anything is enqueued and leave the stream untouched.
 *     Asynchronous CUDA errors surface on the next call or through hsa_check.
 *     Device-side range violations (a position or index outside its buffer)
 *     never fault: the offending access is skipped, the output for that item
 *     is unspecified, and a sticky device flag is raised that hsa_check
 *     reports as HSA_ERR_DEVICE_FLAG.
 *   - hsa_last_error() returns a thread-local message for the last failing
 *     call on this thread.
 *   - Workspaces are caller-owned device scratch sized by the matching
 *     *_workspace_size call.  A workspace must be zero-filled once before its
 *     first use (cudaMemset); every successful call leaves it zero-filled
 *     again.  Calls that share a workspace must not run concurrently.
 */
#ifndef HSA_H
#define HSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define HSA_API __attribute__((visibility("default")))
#else
#define HSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *hsa_stream_t; /* identical to cudaStream_t */

typedef enum {
    HSA_OK = 0,
    HSA_ERR_INVALID_ARG = 1, /* a size, pointer or stride is invalid */
    HSA_ERR_UNSUPPORTED = 2, /* valid but not supported: dtype, head dim, alignment, device */
    HSA_ERR_WORKSPACE = 3,   /* workspace missing or too small */
    HSA_ERR_CUDA = 4,        /* a CUDA runtime call failed (message in hsa_last_error) */
    HSA_ERR_DEVICE_FLAG = 5  /* a kernel raised its range-violation flag (hsa_check) */
} hsa_status_t;

typedef enum {
    HSA_F32 = 0, /* IEEE fp32 */
    HSA_BF16 = 1 /* bfloat16 */
} hsa_dtype_t;

/* Thread-local, NUL-terminated message describing the last failure on this
 * thread ("" if none).  The pointer stays valid until the next call on this
 * thread. */
HSA_API const char *hsa_last_error(void);

/* Library ABI version (major*10000 + minor*100 + patch). */
HSA_API int hsa_version(void);

/* Synchronises `stream`, then reports (and clears) any pending asynchronous
 * CUDA error and the device range-violation flag of the current device. */
HSA_API hsa_status_t hsa_check(hsa_stream_t stream);

/* The pointer classification every entry point applies to its buffers (no
 * counterpart in the pages: a guard of this library's boundary).  HSA_OK if
 * `p` is device memory of the current device or managed memory;
 * HSA_ERR_INVALID_ARG (with the reason in hsa_last_error) for NULL, host memory
 * (pageable or pinned) and another device's memory.  Enqueues nothing. */
HSA_API hsa_status_t hsa_check_pointer(const void *p);

/*
 * hsa_compress -- KV compression (QbitAI article, 混合注意力机制: CSA step 1
 * "every m tokens' KV entries are merged into one"; HCA "every m' = 128 tokens
 * into one, no overlap").
 *   kc[b, j, :] = sum_{r<m} w[r] * k[b, j*m + r, :]   (and vc from v)
 * for every block j in [tok_begin[b] / m, tok_end[b] / m) (integer division),
 * accumulated in fp32 in the order r = 0..m-1 and rounded once (RNE) to `dt`.
 *   k, v       [B, N_cap, d] of `dt`, strides (in_sb, in_st), unit channel stride
 *   tok_begin, tok_end  device int64 [B]; 0 <= tok_begin <= tok_end <= N_cap
 *   max_blocks host bound on tok_end/m - tok_begin/m over all b (grid size)
 *   w          device fp32 [m]; weights (normally summing to 1)
 *   kc, vc     [B, E_cap, d] of `dt`, strides (out_sb, out_se); may alias
 *              nothing that k/v reads
 * m in [1, 4096], d a multiple of 8 (bf16) or 4 (fp32), d <= 512.
 * Blocks beyond N_cap or E_cap are skipped and raise the device flag.
 */
HSA_API hsa_status_t hsa_compress(const void *k, const void *v, hsa_dtype_t dt, int B, int d,
                          int64_t in_sb, int64_t in_st, int64_t N_cap,
                          const int64_t *tok_begin, const int64_t *tok_end, int64_t max_blocks,
                          const float *w, int m,
                          void *kc, void *vc, int64_t out_sb, int64_t out_se, int64_t E_cap,
                          hsa_stream_t stream);

/*
 * hsa_compress_v4 -- hsa_compress for V4's shared key/value entries, with the
 * entry's preparation as it is written (QbitAI article, 混合注意力机制: the
 * KV normalisation and partial RoPE paragraphs; one entry serves as key and
 * value):  kc[b, j] = R((j+1)m - 1) N(sum_{r<m} w[r] k[b, j*m + r])
 * with N RMSNorm (gamma, eps) and R the rotation of the last rope_dims
 * channels as in hsa_rmsnorm_rope; the sum runs in fp32 in the order
 * r = 0..m-1 and the result is rounded once to `dt`.  Arguments as
 * hsa_compress for the one tensor k -> kc, plus gamma (device fp32 [d] or
 * NULL), eps >= 0, rope_dims (even, <= min(d, 128)) and theta > 0.
 * d a multiple of 64, d <= 512.  The result equals hsa_compress followed by
 * hsa_rmsnorm_rope on the new entries up to that call's rounding of the
 * intermediate entry.
 */
HSA_API hsa_status_t hsa_compress_v4(const void *k, hsa_dtype_t dt, int B, int d, int64_t in_sb, int64_t in_st,
                                     int64_t N_cap, const int64_t *tok_begin, const int64_t *tok_end,
                                     int64_t max_blocks, const float *w, int m, void *kc, int64_t out_sb,
                                     int64_t out_se, int64_t E_cap, const float *gamma, float eps, int rope_dims,
                                     float theta, hsa_stream_t stream);

/*
 * hsa_compress_learned -- attention-like compression with learned weights
 * (QbitAI article, 混合注意力机制: CSA step 1 merges every m tokens "through an
 * attention-like mechanism with learned weights"; the HCA paragraph: m' = 128
 * and no overlap, unlike CSA).  The pages give no formula; this library reads
 * it as: entry j pools the L tokens t_r = (j+1)*m - L + r, r = 0..L-1
 * (t_r >= 0; L = 2m for CSA, the block and the one before it; L = m for HCA):
 *   s_r = <u, k[b, t_r]> + bias[r],  a = softmax_r(s)  (fp32),
 *   kc[b, j] = sum_r a_r k[b, t_r],   vc[b, j] = sum_r a_r v[b, t_r]
 * rounded once to `dt`, for blocks j in [tok_begin[b] / m, tok_end[b] / m).
 * Entry j still ends at token (j+1)*m - 1, so visibility is unchanged.
 *   u          device fp32 [d];  bias  device fp32 [L]
 * Other arguments as hsa_compress; d a multiple of 32 up to 512, 1 <= L <= 1024.
 */
HSA_API hsa_status_t hsa_compress_learned(const void *k, const void *v, hsa_dtype_t dt, int B, int d,
                                          int64_t in_sb, int64_t in_st, int64_t N_cap,
                                          const int64_t *tok_begin, const int64_t *tok_end, int64_t max_blocks,
                                          const float *u, const float *bias, int m, int L,
                                          void *kc, void *vc, int64_t out_sb, int64_t out_se, int64_t E_cap,
                                          hsa_stream_t stream);

/*
 * hsa_compress_append -- decode-time compression with a partial-block state
 * cache, the incremental form of hsa_compress (the yage.ai essay
 * "deepseek-v4-agentic-workload", paragraph on what hybrid attention costs:
 * V4 manages a state cache beside the classical KV cache; here the state is
 * the running weighted sum of each sequence's incomplete block).
 * For each sequence b and new token t = 0..T-1 at position p = pos0[b] + t,
 * with r = p mod m:
 *   state[b] = (r == 0 ? 0 : state[b]) + w[r] * x[b, t]   (fp32, fused multiply-add)
 *   if r == m - 1:  c[b, p / m] = round_to_dt(state[b])
 * for K (state_k -> kc) and V (state_v -> vc).  The entries are bit-identical
 * to hsa_compress over the same tokens; earlier tokens are never re-read, so
 * the raw cache only needs the attention window.  After the call the states
 * hold the partial sums of each sequence's incomplete block; a state whose
 * block starts inside the call needs no initial value.
 *   k_new, v_new  [B, T, d] of `dt`, strides (new_sb, new_st), unit channel stride
 *   pos0          device int64 [B], >= 0
 *   w             device fp32 [m]
 *   state_k, state_v  device fp32 [B, d], sequence stride state_sb (elements),
 *                 16-byte aligned
 *   kc, vc        [B, E_cap, d] of `dt`, strides (out_sb, out_se)
 * The indexer key of a new entry comes from the model's indexer projection,
 * which this library does not hold: the caller writes it into k_idx.
 * d a multiple of 8 (bf16) or 4 (fp32), d <= 512; m in [1, 4096].  Entries
 * beyond E_cap or a negative position raise the device flag.
 */
HSA_API hsa_status_t hsa_compress_append(const void *k_new, const void *v_new, hsa_dtype_t dt, int B, int T, int d,
                                         int64_t new_sb, int64_t new_st, const int64_t *pos0, const float *w, int m,
                                         float *state_k, float *state_v, int64_t state_sb, void *kc, void *vc,
                                         int64_t out_sb, int64_t out_se, int64_t E_cap, hsa_stream_t stream);

/*
 * hsa_index_topk -- lightning indexer and exact top-k (QbitAI article,
 * 混合注意力机制: CSA step 2 "a light indexer scores each query token against
 * every compressed block, the top-k blocks are kept"; k = 512 for V4-Flash and
 * 1024 for V4-Pro per the yage.ai essay on agentic workloads).
 * For query t of sequence b at position p = q_pos0[b] + t:
 *   s_j = sum_c q_idx[b, t, c] * k_idx[b, j, c]   (exact int32)
 * for the E(p) = floor((p+1)/m) visible entries; the first min(topk, E(p)) of
 * j ordered by (s_j desc, j asc) are written to idx_out[b, t, :] in ASCENDING
 * index order, padded with -1; cnt_out[b, t] = min(topk, E(p)).
 *   q_idx      int8 [B, T, DI], strides (q_sb, q_st)
 *   k_idx      int8 [B, E_cap, DI], strides (k_sb, k_se); E(p) <= E_cap required
 *   q_pos0     device int64 [B]
 *   idx_out    int32 [B, T, topk] contiguous;  cnt_out int32 [B, T] contiguous
 *   ws         workspace of hsa_index_topk_workspace_size bytes
 * DI a multiple of 16 in [16, 128]; 1 <= topk <= 4096; m >= 1.
 * Results are bit-identical for every input (ties included) and independent
 * of B, T and the launch configuration.  B * T <= 2^24.
 */
HSA_API hsa_status_t hsa_index_topk_workspace_size(int B, int T, int DI, int64_t E_cap, int topk,
                                           size_t *bytes);
HSA_API hsa_status_t hsa_index_topk(const int8_t *q_idx, int64_t q_sb, int64_t q_st,
                            const int8_t *k_idx, int64_t k_sb, int64_t k_se, int64_t E_cap,
                            int B, int T, int DI, const int64_t *q_pos0, int m, int topk,
                            int32_t *idx_out, int32_t *cnt_out, void *ws, size_t ws_bytes,
                            hsa_stream_t stream);

/*
 * hsa_index_topk_noalloc -- hsa_index_topk for callers that cannot allocate
 * device memory.  The paper has no counterpart: this is a convenience of the
 * library, not a step of the method.
 *
 * Some callers own every byte of device memory through their own pool (an
 * inference server that reserves HBM up front, a framework whose caching
 * allocator must see every allocation) or run where host code may not call
 * cudaMalloc at all, and their interface hands this library only inputs and
 * outputs, so they cannot pass the workspace hsa_index_topk needs.  This entry
 * point takes the same arguments minus the workspace and computes the same
 * result (bit-identical) in a scratch buffer built into the library: a static
 * device array of HSA_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU which loads
 * the library holds until the process exits.  It calls no cudaMalloc, cudaFree
 * or allocating library routine.
 *   - Calls whose scratch need (the value hsa_index_topk_workspace_size would
 *     return for the same sizes) exceeds HSA_NOALLOC_SCRATCH_BYTES are rejected
 *     with HSA_ERR_WORKSPACE and a message giving both sizes; use
 *     hsa_index_topk with your own workspace for those.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before capturing a stream.
 *   - Every call on a device shares the one array and it keeps the previous
 *     call's contents; the call clears the part that must start at zero on its
 *     stream before its kernels run.  Calls that overlap on the GPU (other
 *     streams, other threads) race on the array: serialise them.
 */
#define HSA_NOALLOC_SCRATCH_BYTES (16u << 20)
HSA_API hsa_status_t hsa_index_topk_noalloc(const int8_t *q_idx, int64_t q_sb, int64_t q_st,
                                            const int8_t *k_idx, int64_t k_sb, int64_t k_se,
                                            int64_t E_cap, int B, int T, int DI,
                                            const int64_t *q_pos0, int m, int topk,
                                            int32_t *idx_out, int32_t *cnt_out,
                                            hsa_stream_t stream);

/*
 * hsa_attn_decode -- one new query token per sequence (QbitAI article,
 * 混合注意力机制: CSA step 3, MQA over the selected compressed entries; HCA,
 * dense over all entries; the sliding-window paragraph: the most recent
 * `window` raw tokens, current one included, join the same softmax).
 * Sequence b's query sits at p = ctx_len[b] - 1 and attends, per head h, to
 *   S = {kc/vc[b, j] : j in idx[b, :cnt[b]]}  (CSA)  or  {j < E(p)}  (HCA: idx == NULL)
 *     + {k_raw/v_raw[b, t] : max(0, p-window+1) <= t <= p}
 * with logits scale * <q[b,h], k_x> and one softmax; out[b, h] is the
 * softmax-weighted sum of v_x and lse[b, h] its natural-log normaliser
 * (-inf and out = 0 for an empty set).  Work is split over the set and the
 * parts are combined with the log-sum-exp rule.  CSA (idx given): the split of
 * a sequence depends only on its own set size, so its output is bit-identical
 * whatever else is in the batch.  HCA (idx == NULL), bf16, d = 128, H a
 * multiple of 64, B <= 1024: the batch's 128-item tiles are split evenly over
 * the SMs, so outputs are deterministic for a given batch but may differ in the
 * last bits from the same sequence decoded in another batch.
 *   q          [B, H, d] of `dt`, contiguous
 *   kc, vc     [B, E_cap, d] of `dt`, strides (c_sb, c_se)
 *   idx, cnt   int32 [B, topk] (ascending or not; entries < 0 are skipped)
 *              and int32 [B] (NULL: all topk slots are scanned), or idx = NULL
 *              for dense HCA
 *   k_raw, v_raw [B, N_cap, d] of `dt`, strides (r_sb, r_st)
 *   ctx_len    device int64 [B]; 1 <= ctx_len <= N_cap
 *   out        [B, H, d] of `dt`, contiguous;  lse fp32 [B, H] or NULL
 *   ws         workspace of hsa_attn_decode_workspace_size bytes (may be 0):
 *              the parts' partial results.  For bf16 CSA with d = 128, H a
 *              multiple of 64 and topk + window <= 2048 the parts are tiles of
 *              128 slots, one thread-block cluster per (sequence, 64 heads), and
 *              the workspace holds their fp32 partials, about B * H/64 *
 *              ceil((topk + window) / 128) * 33,280 bytes; for bf16 HCA
 *              (d = 128, H a multiple of 64) about B * H/64 * (ceil(E_cap / 128)
 *              + ceil(window / 128)) * 33,280 bytes.
 * Every pointer is a device pointer; host memory, pinned or not, is refused
 * with HSA_ERR_INVALID_ARG before anything is enqueued.
 * bf16: d in {64, 128}, H a multiple of 16 up to 128.  fp32: d a multiple of
 * 32 up to 256, any H.
 */
HSA_API hsa_status_t hsa_attn_decode_workspace_size(hsa_dtype_t dt, int B, int H, int d, int64_t E_cap,
                                            int m, int topk, int window, size_t *bytes);
HSA_API hsa_status_t hsa_attn_decode(const void *q, hsa_dtype_t dt, int B, int H, int d,
                             const void *kc, const void *vc, int64_t c_sb, int64_t c_se,
                             int64_t E_cap, int m, const int32_t *idx, const int32_t *cnt, int topk,
                             const void *k_raw, const void *v_raw, int64_t r_sb, int64_t r_st,
                             int64_t N_cap, int window, const int64_t *ctx_len, float scale,
                             void *out, float *lse, void *ws, size_t ws_bytes, hsa_stream_t stream);

/*
 * hsa_decode_csa -- one CSA decode step in one launch: the indexer and exact
 * top-k of hsa_index_topk followed by the attention of hsa_attn_decode over the
 * selected entries plus the window (QbitAI article, 混合注意力机制: CSA steps 2
 * and 3 and the sliding-window paragraph).  For sequence b with its query at
 * p = ctx_len[b] - 1 (so q_pos0 = ctx_len - 1 for the indexer):
 *   idx_out[b, :], cnt_out[b]   exactly as hsa_index_topk (bit-identical)
 *   out[b, h], lse[b, h]        as hsa_attn_decode with idx = idx_out, cnt = cnt_out
 * The CTAs that score a sequence's entries also attend to the entries they
 * select and meet at three barriers inside one cooperative launch, instead of
 * a grid-wide hand-off between two kernels.  The split of the attention follows
 * the launch's chunks, which depend on B: outputs are deterministic for a given
 * batch (not bit-identical across batches).
 *   q_idx      int8 [B, DI], row stride qi_sb;  k_idx int8 [B, E_cap, DI] with
 *              k_se == DI (contiguous rows), sequence stride k_sb
 *   idx_out    int32 [B, topk];  cnt_out int32 [B]
 *   q          [B, H, d] bf16 contiguous;  kc, vc [B, E_cap, d] (c_sb, c_se);
 *              k_raw, v_raw [B, N_cap, d] (r_sb, r_st);  out [B, H, d];  lse [B, H]
 *              fp32 or NULL
 *   ws         workspace of hsa_decode_csa_workspace_size bytes, zero-filled
 *              once before first use (left zero by every call)
 * bf16, d = 128, H in {64, 128}, DI in {16, 32, 64, 128}, 1 <= topk <= 4096,
 * E_cap >= 1.  Sizes whose chunks cannot all be resident at once return
 * HSA_ERR_UNSUPPORTED (use the two calls).
 */
HSA_API hsa_status_t hsa_decode_csa_workspace_size(int B, int H, int d, int DI, int64_t E_cap, size_t *bytes);
HSA_API hsa_status_t hsa_decode_csa(const int8_t *q_idx, int64_t qi_sb, const int8_t *k_idx, int64_t k_sb,
                                    int64_t k_se, int64_t E_cap, int DI, int m, int topk, int32_t *idx_out,
                                    int32_t *cnt_out, const void *q, hsa_dtype_t dt, int B, int H, int d,
                                    const void *kc, const void *vc, int64_t c_sb, int64_t c_se, const void *k_raw,
                                    const void *v_raw, int64_t r_sb, int64_t r_st, int64_t N_cap, int window,
                                    const int64_t *ctx_len, float scale, void *out, float *lse, void *ws,
                                    size_t ws_bytes, hsa_stream_t stream);

/*
 * hsa_attn_prefill -- T query tokens per sequence at positions
 * q_pos0[b] .. q_pos0[b]+T-1, each with its own set S as in hsa_attn_decode
 * (causal within the chunk through E(p) and the window bound; the raw cache
 * already holds every query token).
 *   q          [B, T, H, d] of `dt`, contiguous
 *   idx, cnt   int32 [B, T, topk] and [B, T] (cnt may be NULL), or idx = NULL (HCA)
 *   out        [B, T, H, d] of `dt`;  lse fp32 [B, T, H] or NULL
 * Other arguments as hsa_attn_decode.
 */
HSA_API hsa_status_t hsa_attn_prefill_workspace_size(hsa_dtype_t dt, int B, int T, int H, int d,
                                             int64_t E_cap, int m, int topk, int window,
                                             size_t *bytes);
HSA_API hsa_status_t hsa_attn_prefill(const void *q, hsa_dtype_t dt, int B, int T, int H, int d,
                              const void *kc, const void *vc, int64_t c_sb, int64_t c_se,
                              int64_t E_cap, int m, const int32_t *idx, const int32_t *cnt, int topk,
                              const void *k_raw, const void *v_raw, int64_t r_sb, int64_t r_st,
                              int64_t N_cap, int window, const int64_t *q_pos0, float scale,
                              void *out, float *lse, void *ws, size_t ws_bytes,
                              hsa_stream_t stream);

/*
 * V4's per-layer attention details (QbitAI article, 混合注意力机制, the
 * paragraphs after the CSA/HCA description: Q/KV normalisation, partial RoPE,
 * one KV entry as key and value with the output rotated back by the query's
 * position, attention sink).  They run on the same attention kernels: prepare
 * the query, the compressed entries and the raw window tokens with
 * hsa_rmsnorm_rope, pass one buffer as both kc and vc (and as both k_raw and
 * v_raw), request lse from the attention call, then apply hsa_attn_finalize.
 * For CSA decode, hsa_compress_v4 prepares each entry as it is written and
 * hsa_attn_decode_v4 takes the raw query and applies the sink and the inverse
 * rotation itself (below), so only the window tokens need hsa_rmsnorm_rope.
 * The result is
 *   q~ = R(p) N_q(q),  e~_x = R(t_x) N_kv(e_x),  logit_x = scale <q~, e~_x>,
 *   out = R(-p) sum_x softmax'(logit)_x e~_x,  lse = ln(sum_x e^logit_x + e^z_h)
 * where softmax' includes the sink logit z_h in its denominator, N is RMSNorm
 * x * gamma / sqrt(mean(x^2) + eps), and R(t) turns channel pair k of the last
 * rope_dims channels (channels d - rope_dims + 2k, + 1) by t * theta^(-2k /
 * rope_dims).  A compressed entry j sits at its block's last token, (j+1)*m - 1.
 *
 * hsa_rmsnorm_rope -- x <- R(pos) N(x), in place, for the rows
 * n in [n_begin[b], n_end[b]) of every sequence b and all H heads:
 *   x          [B, n_cap, H, d] of `dt`, strides (x_sb, x_sn) in elements,
 *              heads contiguous (stride d)
 *   n_begin, n_end  device int64 [B];  max_rows host bound on n_end - n_begin
 *   pos        (pos_base ? pos_base[b] : 0) + n * pos_stride + pos_offset
 *              (queries: pos_base = q_pos0, stride 1; entries: stride m,
 *              offset m - 1; raw tokens: stride 1)
 *   gamma      device fp32 [d] or NULL (ones);  rope_dims even, <= min(d, 128)
 * d a multiple of 64, d <= 512.  Rows outside [0, n_cap) raise the device flag.
 *
 * hsa_attn_finalize -- sink and inverse rotation on the (out, lse) of an
 * attention call over prepared vectors, in place:
 *   lse' = ln(e^lse + e^sink[h]),  out' = R(-p) e^(lse - lse') out
 * with p = q_pos0[b] + t (decode: q_pos0 = ctx_len - 1, T = 1).
 *   out        [B, T, H, d] of `dt`, contiguous;  lse fp32 [B, T, H]
 *   sink       device fp32 [H] or NULL (no sink: lse unchanged)
 */
/*
 * hsa_attn_decode_v4 -- the same V4 decode attention with the query's
 * preparation and the finalization inside the attention kernel (QbitAI
 * article, 混合注意力机制, the Q/KV normalisation, partial RoPE, shared
 * key/value and attention-sink paragraphs): q is the raw query; the kernel
 * forms R(p) N_q(q) in shared memory (N_q with gamma_q and eps, R turning the
 * last rope_dims channels by p * theta^(-2k / rope_dims), p = ctx_len - 1),
 * attends to the selected entries and the window exactly as hsa_attn_decode,
 * and writes out = R(-p) sum_x softmax'(logit)_x v_x and lse = ln(sum_x
 * e^logit_x + e^sink[h]) -- the result of hsa_rmsnorm_rope on q, then
 * hsa_attn_decode, then hsa_attn_finalize, in one launch.  The entries and
 * window tokens must already be prepared (hsa_rmsnorm_rope when they are
 * written).  Arguments as hsa_attn_decode (workspace of
 * hsa_attn_decode_workspace_size bytes), plus:
 *   gamma_q    device fp32 [d] or NULL (ones);  eps >= 0
 *   rope_dims  even, 0 <= rope_dims <= d;  theta > 0
 *   sink       device fp32 [H] or NULL (no sink)
 * Runs on the tensor-core CSA decode path only: bf16, d = 128, H a multiple of
 * 64, idx non-NULL, topk + window <= 2048; other shapes return
 * HSA_ERR_UNSUPPORTED.  q is not modified.
 */
HSA_API hsa_status_t hsa_attn_decode_v4(const void *q, hsa_dtype_t dt, int B, int H, int d, const void *kc,
                                        const void *vc, int64_t c_sb, int64_t c_se, int64_t E_cap, int m,
                                        const int32_t *idx, const int32_t *cnt, int topk, const void *k_raw,
                                        const void *v_raw, int64_t r_sb, int64_t r_st, int64_t N_cap, int window,
                                        const int64_t *ctx_len, float scale, const float *gamma_q, float eps,
                                        int rope_dims, float theta, const float *sink, void *out, float *lse,
                                        void *ws, size_t ws_bytes, hsa_stream_t stream);

HSA_API hsa_status_t hsa_rmsnorm_rope(void *x, hsa_dtype_t dt, int B, int H, int d, int64_t x_sb, int64_t x_sn,
                                      int64_t n_cap, const int64_t *n_begin, const int64_t *n_end,
                                      int64_t max_rows, const int64_t *pos_base, int64_t pos_stride,
                                      int64_t pos_offset, const float *gamma, float eps, int rope_dims,
                                      float theta, hsa_stream_t stream);
HSA_API hsa_status_t hsa_attn_finalize(void *out, float *lse, hsa_dtype_t dt, int B, int T, int H, int d,
                                       const int64_t *q_pos0, const float *sink, int rope_dims, float theta,
                                       hsa_stream_t stream);

/*
 * Context-parallel exchange of one long sequence (no counterpart in the pages:
 * the pages describe one GPU's attention; these three calls let several ranks
 * that each hold a contiguous range of a sequence's compressed entries produce
 * the same result).  Per decode step each rank runs hsa_index_topk on its own
 * range, ships its local top-k as (score, global index) pairs, every rank
 * merges the gathered pairs with hsa_topk_merge (the global top-k is the
 * top-k of the union of the local top-k lists), attends to the selected
 * entries it holds (the rank holding the newest raw tokens adds the window),
 * and the ranks' partial (out, lse) are combined with hsa_lse_merge.
 *
 * hsa_index_scores -- exact indexer scores of listed entries (the score of
 * hsa_index_topk: s_j = sum_c q_idx[b, t, c] * k_idx[b, j, c], int32).
 *   idx        int32 [B, T, topk] entry indices (local to k_idx); slots with
 *              j < 0 or at or beyond cnt[b, t] get INT32_MIN
 *   cnt        int32 [B, T] or NULL (all topk slots)
 *   scores     int32 [B, T, topk] contiguous
 * Other arguments as hsa_index_topk.  j >= E_cap raises the device flag.
 */
HSA_API hsa_status_t hsa_index_scores(const int8_t *q_idx, int64_t q_sb, int64_t q_st,
                                      const int8_t *k_idx, int64_t k_sb, int64_t k_se, int64_t E_cap,
                                      int B, int T, int DI, const int32_t *idx, const int32_t *cnt, int topk,
                                      int32_t *scores, hsa_stream_t stream);

/*
 * hsa_topk_merge -- exact top-k over explicit (score, index) pairs.
 *   scores, idx  int32 [rows, n] contiguous; idx < 0 marks an empty slot.
 *                The non-empty indices of a row must be distinct and in
 *                ascending order (the rank-major concatenation of per-rank
 *                ascending lists over increasing entry ranges is).
 *   idx_out      int32 [rows, topk]: the first min(topk, non-empty) indices
 *                under (score desc, index asc), in ascending index order,
 *                padded with -1;  cnt_out int32 [rows] their count.
 * 1 <= n <= 1 << 20, 1 <= topk <= 4096.
 */
HSA_API hsa_status_t hsa_topk_merge(const int32_t *scores, const int32_t *idx, int rows, int n, int topk,
                                    int32_t *idx_out, int32_t *cnt_out, hsa_stream_t stream);

/*
 * hsa_lse_merge -- combine S partial attention results of the same queries
 * over disjoint item sets: lse = ln sum_s exp(lse_s) and
 * out = sum_s exp(lse_s - lse) * out_s (a part with lse_s = -inf is empty and
 * weighs 0; all parts empty give out = 0, lse = -inf).
 *   parts_o    [S, rows, H, d] of `dt`, contiguous
 *   parts_lse  fp32 [S, rows, H], contiguous
 *   out        [rows, H, d] of `dt`;  lse_out fp32 [rows, H] or NULL
 * d a multiple of 4 (fp32) or 8 (bf16), d <= 1024; S >= 1.
 */
HSA_API hsa_status_t hsa_lse_merge(const void *parts_o, const float *parts_lse, hsa_dtype_t dt, int S, int rows,
                                   int H, int d, void *out, float *lse_out, hsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HSA_H */
