// Kernels for the context-parallel exchange of one long sequence whose
// compressed entries are sharded over ranks (each rank holds a contiguous
// range of entries):
//   index_scores  exact int32 indexer scores of listed entries, so a rank can
//                 ship its local top-k as (score, global index) pairs;
//   topk_merge    exact top-k over the gathered pairs of every rank, ordered by
//                 (score desc, index asc), written in ascending index order
//                 (QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制,
//                 CSA step 2: keep the top-k of the scored entries);
//   lse_merge     o = sum_s exp(lse_s - lse) o_s with lse = ln sum_s exp(lse_s),
//                 the log-sum-exp combination of per-rank partial attention.
// The global top-k of the whole sequence is the top-k of the union of the
// ranks' local top-k lists: an entry outside its own rank's top-k has k
// entries of that rank ranked above it.
#include "block_scan.cuh"
#include "common.cuh"
#include "internal.h"

namespace hsa {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int dot16(const int4 &x, const int4 &y) {
    int s = __dp4a(x.x, y.x, 0);
    s = __dp4a(x.y, y.y, s);
    s = __dp4a(x.z, y.z, s);
    return __dp4a(x.w, y.w, s);
}

// ------------------------------------------------------------ index_scores
__global__ void __launch_bounds__(kThreads) index_scores_kernel(IndexScoreArgs a) {
    const int row = blockIdx.y;
    const int i = blockIdx.x * kThreads + threadIdx.x;
    if (i >= a.topk) return;
    const int b = row / a.T, t = row - (row / a.T) * a.T;
    int32_t *out = a.scores + (int64_t)row * a.topk;
    const int n = a.cnt ? a.cnt[row] : a.topk;
    const int32_t j = a.idx[(int64_t)row * a.topk + i];
    if (i >= n || j < 0) {
        out[i] = INT32_MIN;
        return;
    }
    if (j >= a.E_cap) {
        raise_flag(FLAG_INDEX_RANGE);
        out[i] = INT32_MIN;
        return;
    }
    const int4 *qp = reinterpret_cast<const int4 *>(a.q + b * a.q_sb + (int64_t)t * a.q_st);
    const int4 *kp = reinterpret_cast<const int4 *>(a.k + b * a.k_sb + (int64_t)j * a.k_se);
    int s = 0;
    for (int c = 0; c < a.DI / 16; ++c) s += dot16(__ldg(qp + c), __ldg(kp + c));
    out[i] = s;
}

// -------------------------------------------------------------- topk_merge
// The bin of hist[0 .. nb) (bin index grows with the key) where the count from the
// top first reaches `want`: s_out[0] = bin, s_out[1] = count above it.
__device__ void find_bin(const unsigned *hist, int nb, int want, int *s_scan, int *s_out) {
    const int per = nb / kThreads, top = nb - 1 - threadIdx.x * per;
    int local = 0;
    for (int q = 0; q < per; ++q) local += (int)hist[top - q];
    int tot;
    const int before = block_exclusive_sum(local, s_scan, tot);
    if (before < want && before + local >= want) {
        int cum = before;
        for (int q = 0; q < per; ++q) {
            const int hv = (int)hist[top - q];
            if (cum + hv >= want) {
                s_out[0] = top - q;
                s_out[1] = cum;
                break;
            }
            cum += hv;
        }
    }
    __syncthreads();
}

// order-preserving map of int32 scores to unsigned keys
__device__ __forceinline__ uint32_t key_of(int32_t s) { return (uint32_t)s ^ 0x80000000u; }

__global__ void __launch_bounds__(kThreads) topk_merge_kernel(TopkMergeArgs a) {
    __shared__ unsigned hist[2048];
    __shared__ int s_scan[33];
    __shared__ int s_out[2];
    __shared__ int s_w[2 * (kThreads / 32)];
    const int row = blockIdx.x;
    const int32_t *sc = a.scores + (int64_t)row * a.n;
    const int32_t *ix = a.idx + (int64_t)row * a.n;
    int32_t *out = a.idx_out + (int64_t)row * a.topk;

    int nv = 0;
    for (int i = threadIdx.x; i < a.n; i += kThreads) nv += ix[i] >= 0;
    int n_valid;
    block_exclusive_sum(nv, s_scan, n_valid);
    const int kk = n_valid < a.topk ? n_valid : a.topk;
    for (int i = kk + threadIdx.x; i < a.topk; i += kThreads) out[i] = -1;
    if (threadIdx.x == 0) a.cnt_out[row] = kk;
    if (kk == 0) return;

    // three radix levels over the 32-bit key: bits 31..21, 20..10, 9..0
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    uint32_t prefix = 0, prefix_mask = 0;
    int need = kk;
    for (int lv = 0; lv < 3; ++lv) {
        const int nb = 1 << widths[lv];
        for (int i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < a.n; i += kThreads) {
            if (ix[i] < 0) continue;
            const uint32_t u = key_of(sc[i]);
            if ((u & prefix_mask) == prefix) atomicAdd(&hist[(u >> shifts[lv]) & (uint32_t)(nb - 1)], 1u);
        }
        __syncthreads();
        find_bin(hist, nb, need, s_scan, s_out);
        prefix |= (uint32_t)s_out[0] << shifts[lv];
        prefix_mask |= (uint32_t)(nb - 1) << shifts[lv];
        need -= s_out[1];
        __syncthreads();
    }
    const uint32_t T = prefix;  // the kk-th largest key
    const int n_eq_need = need;  // items equal to T to take, lowest index first

    // ordered compaction: each warp owns one contiguous run of items
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kWarps = kThreads / 32;
    const int run = ((a.n + kWarps - 1) / kWarps + 31) & ~31;
    const int w0 = min(a.n, warp * run), w1 = min(a.n, w0 + run);
    int gt = 0, eq = 0;
    for (int i = w0 + lane; i < w1; i += 32) {
        if (ix[i] < 0) continue;
        const uint32_t u = key_of(sc[i]);
        gt += u > T;
        eq += u == T;
    }
    gt = __reduce_add_sync(0xffffffffu, gt);
    eq = __reduce_add_sync(0xffffffffu, eq);
    if (lane == 0) {
        s_w[warp] = gt;
        s_w[kWarps + warp] = eq;
    }
    __syncthreads();
    int eq_run = 0, sel_run = 0;
    for (int v = 0; v < warp; ++v) {
        const int ev = s_w[kWarps + v];
        int tk = n_eq_need - eq_run;
        tk = tk < 0 ? 0 : (tk > ev ? ev : tk);
        sel_run += s_w[v] + tk;
        eq_run += ev;
    }
    const uint32_t lt = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const int32_t j = i < w1 ? ix[i] : -1;
        const bool valid = j >= 0;
        const uint32_t u = valid ? key_of(sc[i]) : 0u;
        const bool is_eq = valid && u == T;
        const uint32_t em = __ballot_sync(0xffffffffu, is_eq);
        const bool take = (valid && u > T) || (is_eq && eq_run + __popc(em & lt) < n_eq_need);
        const uint32_t tm = __ballot_sync(0xffffffffu, take);
        if (take) {
            const int o = sel_run + __popc(tm & lt);
            if (o < kk) out[o] = j;
        }
        eq_run += __popc(em);
        sel_run += __popc(tm);
    }
}

// --------------------------------------------------------------- lse_merge
template <typename T>
__device__ __forceinline__ float4 load4(const T *p);
template <>
__device__ __forceinline__ float4 load4<float>(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u), __uint_as_float(v.y << 16),
                       __uint_as_float(v.y & 0xffff0000u));
}

template <typename T>
__global__ void __launch_bounds__(128) lse_merge_kernel(LseMergeArgs a) {
    // one warp per (row, head)
    const int row = blockIdx.y;
    const int h = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (h >= a.H) return;
    const int64_t rh = (int64_t)row * a.H + h;
    const int64_t part_lse = (int64_t)a.rows * a.H, part_o = part_lse * a.d;
    float M = -INFINITY;
    for (int s = lane; s < a.S; s += 32) M = fmaxf(M, a.parts_lse[s * part_lse + rh]);
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 8));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
    float L = 0.f;
    if (M != -INFINITY)
        for (int s = lane; s < a.S; s += 32) {
            const float ls = a.parts_lse[s * part_lse + rh];
            L += ls == -INFINITY ? 0.f : expf(ls - M);
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const bool empty = M == -INFINITY;
    const float invL = empty ? 0.f : 1.f / L;
    const T *po = static_cast<const T *>(a.parts_o);
    T *out = static_cast<T *>(a.out) + rh * a.d;
    for (int c4 = lane; c4 < a.d / 4; c4 += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!empty)
            for (int s = 0; s < a.S; ++s) {
                const float ls = a.parts_lse[s * part_lse + rh];
                if (ls == -INFINITY) continue;
                const float wgt = expf(ls - M) * invL;
                const float4 v = load4<T>(po + s * part_o + rh * a.d + c4 * 4);
                acc.x = fmaf(wgt, v.x, acc.x);
                acc.y = fmaf(wgt, v.y, acc.y);
                acc.z = fmaf(wgt, v.z, acc.z);
                acc.w = fmaf(wgt, v.w, acc.w);
            }
        if constexpr (sizeof(T) == 2) {
            uint2 pk;
            pk.x = pack_bf16x2(acc.x, acc.y);
            pk.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2 *>(out + c4 * 4) = pk;
        } else {
            *reinterpret_cast<float4 *>(out + c4 * 4) = acc;
        }
    }
    if (a.lse_out && lane == 0) a.lse_out[rh] = empty ? -INFINITY : M + logf(L);
}

}  // namespace

cudaError_t launch_index_scores(const IndexScoreArgs &a, cudaStream_t s) {
    const int rows = a.B * a.T;
    dim3 grid((a.topk + kThreads - 1) / kThreads, rows);
    index_scores_kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_topk_merge(const TopkMergeArgs &a, cudaStream_t s) {
    topk_merge_kernel<<<a.rows, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_lse_merge(const LseMergeArgs &a, bool bf16, cudaStream_t s) {
    dim3 grid((a.H + 3) / 4, a.rows);
    if (bf16)
        lse_merge_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a);
    else
        lse_merge_kernel<float><<<grid, 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace hsa
