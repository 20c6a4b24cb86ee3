// Internal launch interface between the C-ABI layer (hsa_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace hsa {

struct CompressArgs {
    const void *k, *v;
    int B, d;
    int64_t in_sb, in_st, N_cap;
    const int64_t *tok_begin, *tok_end;
    int64_t max_blocks;
    const float *w;
    int m;
    void *kc, *vc;
    int64_t out_sb, out_se, E_cap;
};
cudaError_t launch_compress(const CompressArgs &a, bool bf16, int num_sms, cudaStream_t s);
// V4: the entries of one tensor (one entry is both key and value) normalised with
// gamma (RMSNorm) and turned by R((j+1)m - 1) as they are written.
struct CompressV4Args {
    const float *gamma;  // [d] or null (ones)
    float eps;
    int rope_dims;
    double inv_freq[64];
};
cudaError_t launch_compress_v4(const CompressArgs &a, const CompressV4Args &v, bool bf16, cudaStream_t s);
struct CompressAppendArgs {
    const void *k_new, *v_new;  // [B, T, d]
    int B, T, d;
    int64_t new_sb, new_st;
    const int64_t *pos0;        // [B]
    const float *w;
    int m;
    float *state_k, *state_v;   // [B, d] fp32
    int64_t state_sb;
    void *kc, *vc;
    int64_t out_sb, out_se, E_cap;
};
cudaError_t launch_compress_append(const CompressAppendArgs &a, bool bf16, cudaStream_t s);
struct CompressLearnedArgs {
    const void *k, *v;
    int B, d;
    int64_t in_sb, in_st, N_cap;
    const int64_t *tok_begin, *tok_end;
    int64_t max_blocks;
    const float *u;      // [d]
    const float *bias;   // [L]
    int m, L;
    void *kc, *vc;
    int64_t out_sb, out_se, E_cap;
};
cudaError_t launch_compress_learned(const CompressLearnedArgs &a, bool bf16, cudaStream_t s);

// ---------------------------------------------------------------- indexer
struct IndexArgs {
    const int8_t *q;
    int64_t q_sb, q_st;
    const int8_t *k;
    int64_t k_sb, k_se, E_cap;
    int B, T, DI;
    const int64_t *q_pos0;
    int m, topk;
    int32_t *idx_out, *cnt_out;
};
// Workspace layout of the decode-shaped indexer (all offsets 256-byte aligned).
struct IndexPlan {
    int rows;          // rows handled by one launch group
    int chunk;         // entries per CTA
    int nchunks;       // max chunks per row (grid.x)
    int key_bits;      // bits of the biased score key
    int shift1;        // level-1 histogram uses key >> shift1 (256 bins)
    int cap;           // candidate capacity per row
    size_t off_keys, off_hist1, off_tick, off_sel, off_runs, off_cand_u, off_cand_j, total;
};
IndexPlan plan_index(int rows, int DI, int64_t E_cap, int topk, int num_sms);
cudaError_t launch_index_topk(const IndexArgs &a, const IndexPlan &p, void *ws, int row_begin,
                              cudaStream_t s);

// Decode-shaped indexer: one cooperative launch (index_fused.cu).
struct FusedIndexPlan {
    bool ok;           // false: the rows do not fit one resident launch
    int rows, ctas_per_row, chunk, key_bits, shift1, nb2;
    int off_stage_smem;  // byte offset of the copy stages in dynamic shared memory
    size_t smem;
    size_t off_hist1, off_bar, off_rec, off_cand, total;
    size_t zero_bytes;   // the leading part that must be zero before a launch (histograms, counters)
};
FusedIndexPlan plan_index_fused(int rows, int DI, int64_t E_cap, int num_sms);
cudaError_t launch_index_fused(const IndexArgs &a, const FusedIndexPlan &p, void *ws, cudaStream_t s);

// One CSA decode step (indexer, exact top-k, attention) in one cooperative launch
// (decode_fused.cu): bf16, d = 128, H in {64, 128}, indexer keys contiguous.
struct DecodeStepPlan {
    bool ok;
    int rows, ctas_per_row, chunk, key_bits, shift1, nb2;
    size_t smem;
    size_t off_hist, off_bar, off_rec, off_b1, off_po, off_pml, zero_bytes, total;
};
DecodeStepPlan plan_decode_step(int B, int H, int DI, int64_t E_cap, int num_sms);
struct DecodeStepCall {
    const int8_t *qi;
    int64_t qi_sb;
    const int8_t *ki;
    int64_t ki_sb, E_cap;
    int B, DI, m, topk, H, window;
    int32_t *idx_out, *cnt_out;
    const void *q, *kc, *vc, *k_raw, *v_raw;
    int64_t c_sb, c_se, r_sb, r_st, N_cap;
    const int64_t *ctx;
    float scale;
    void *out;
    float *lse;
};
cudaError_t launch_decode_step(const DecodeStepCall &c, const DecodeStepPlan &p, void *ws, cudaStream_t s);

// Many-row indexer on tcgen05 tensor cores (index_prefill_tc.cu).
struct PrefillIndexPlan {
    bool ok;
    int n_qtiles, n_seg, seg_tiles, cap_seg, sample_split;
    size_t off_q16, off_k16, off_hist, off_counts, off_lists, total;
};
PrefillIndexPlan plan_index_prefill(int B, int T, int DI, int64_t E_cap, int topk, int num_sms);
cudaError_t launch_index_prefill(const IndexArgs &a, const PrefillIndexPlan &p, void *ws, int num_sms,
                                 cudaStream_t s);

// ------------------------------------------- context-parallel exchange (cp_merge.cu)
struct IndexScoreArgs {
    const int8_t *q;
    int64_t q_sb, q_st;
    const int8_t *k;
    int64_t k_sb, k_se, E_cap;
    int B, T, DI;
    const int32_t *idx;  // [B*T, topk]
    const int32_t *cnt;  // [B*T] or null
    int topk;
    int32_t *scores;     // [B*T, topk]
};
cudaError_t launch_index_scores(const IndexScoreArgs &a, cudaStream_t s);
struct TopkMergeArgs {
    const int32_t *scores, *idx;  // [rows, n]; idx < 0 marks an empty slot
    int rows, n, topk;
    int32_t *idx_out, *cnt_out;   // [rows, topk], [rows]
};
cudaError_t launch_topk_merge(const TopkMergeArgs &a, cudaStream_t s);
struct LseMergeArgs {
    const void *parts_o;      // [S, rows, H, d]
    const float *parts_lse;   // [S, rows, H]
    int S, rows, H, d;
    void *out;                // [rows, H, d]
    float *lse_out;           // [rows, H] or null
};
cudaError_t launch_lse_merge(const LseMergeArgs &a, bool bf16, cudaStream_t s);

// ------------------------------------------- V4 attention details (v4_extras.cu)
constexpr int kMaxRopeDims = 128;
struct NormRopeArgs {
    void *x;                  // [B, n_cap, H, d], strides (x_sb, x_sn), heads contiguous
    int B, H, d;
    int64_t x_sb, x_sn, n_cap;
    const int64_t *n_begin, *n_end;  // [B]
    int64_t max_rows;
    const int64_t *pos_base;  // [B] or null (0)
    int64_t pos_stride, pos_offset;
    const float *gamma;       // [d] or null (1)
    float eps;
    int rope_dims;
    double inv_freq[kMaxRopeDims / 2];  // theta^(-2k/rope_dims)
};
cudaError_t launch_rmsnorm_rope(const NormRopeArgs &a, bool bf16, cudaStream_t s);
struct FinalizeArgs {
    void *out;                // [B*T, H, d]
    float *lse;               // [B*T, H]
    int B, T, H, d;
    const int64_t *q_pos0;    // [B]
    const float *sink;        // [H] or null
    int rope_dims;
    double inv_freq[kMaxRopeDims / 2];
};
cudaError_t launch_attn_finalize(const FinalizeArgs &a, bool bf16, cudaStream_t s);

// -------------------------------------------------------------- attention
struct AttnArgs {
    const void *q;      // [rows, H, d]
    int rows;           // B * T
    int T;              // queries per sequence (row r -> b = r / T, t = r % T)
    int H, d;
    const void *kc, *vc;
    int64_t c_sb, c_se, E_cap;
    int m;
    const int32_t *idx;  // [rows, topk] or null (dense)
    const int32_t *cnt;  // [rows] or null
    int topk;
    const void *k_raw, *v_raw;
    int64_t r_sb, r_st, N_cap;
    int window;
    const int64_t *pos;  // decode: ctx_len[b] (p = ctx_len - 1); prefill: q_pos0[b] (p = q_pos0 + t)
    int pos_is_ctx;
    int shared_kv;      // kc == vc and k_raw == v_raw: one entry is both key and value
    float scale;
    void *out;          // [rows, H, d]
    float *lse;         // [rows, H] or null
    // split-KV partials (decode)
    int split;          // items per split; <= 0 -> one split per row
    int max_splits;
    float *part_o;      // [rows, max_splits, H, d]
    float *part_lse;    // [rows, max_splits, H]
    // V4 details fused into the tcgen05 CSA decode attention (v4 != 0): RMSNorm
    // (gamma_q) and partial RoPE of the query in shared memory, attention sink and
    // inverse rotation of the output in the merge
    int v4;
    const float *gamma_q;  // [d] or null (ones)
    const float *sink;     // [H] or null (no sink)
    float eps;
    int rope_dims;
    double inv_freq[kMaxRopeDims / 2];
};
int attn_split_size(bool bf16, bool dense, int H, int rows, int64_t max_items, int num_sms);
cudaError_t launch_attn_bf16(const AttnArgs &a, cudaStream_t s);
cudaError_t launch_attn_f32(const AttnArgs &a, cudaStream_t s);
cudaError_t launch_attn_merge(const AttnArgs &a, bool bf16, cudaStream_t s);
// bf16 decode with H in {16, 32, 64, 128}: one cluster per sequence, no workspace.
bool decode_cluster_supported(int H, int d);
cudaError_t launch_attn_decode_cluster(const AttnArgs &a, cudaStream_t s);
// bf16 CSA decode with d = 128, H a multiple of 64, 0 < topk, topk + window <= 2048:
// one cluster of 128-item tiles per (sequence, 64-head group), tcgen05 MMAs; the
// tiles' partials go through a workspace (part_o: O, part_lse: maximum and sum).
bool decode_tc_shape(int H, int d, int topk, int window);
struct DecodeTcWorkspace {
    size_t off_o, off_ml, total;
};
DecodeTcWorkspace decode_tc_workspace(int B, int H, int topk, int window);
bool decode_tc_supported(const AttnArgs &a);
cudaError_t launch_attn_decode_tc(const AttnArgs &a, cudaStream_t s);
// bf16 dense (HCA) decode with d = 128, H a multiple of 64, B <= 1024: one unit per
// 128-item tile of each (sequence, 64-head group), persistent tcgen05 + TMA kernel, the
// tiles' partials (part_o: O, part_lse: maximum and sum) merged in tile order.
bool decode_dense_tc_shape(int B, int H, int d);
struct DecodeDenseWorkspace {
    size_t off_o, off_ml, off_cum, total;  // part_o at off_o, part_lse at off_ml, tile prefix at off_cum
};
DecodeDenseWorkspace decode_dense_workspace(int B, int H, int64_t E_cap, int window);
cudaError_t launch_attn_decode_dense_tc(const AttnArgs &a, int num_sms, cudaStream_t s);
// bf16 dense (HCA) prefill with d = 128 and T*H a multiple of 128: tcgen05 + TMA kernel.
bool prefill_tc_supported(const AttnArgs &a);
cudaError_t launch_attn_prefill_tc(const AttnArgs &a, int num_sms, cudaStream_t s);
// bf16 CSA prefill with H = 64 and d = 128: per-token gathers, tcgen05 M = 64 MMAs.
bool gather_tc_supported(const AttnArgs &a);
cudaError_t launch_attn_gather_tc(const AttnArgs &a, int num_sms, cudaStream_t s);

}  // namespace hsa
