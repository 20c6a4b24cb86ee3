// Lightning indexer + exact top-k for few queries per sequence (decode).
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制, CSA step 2: each
// query scores every visible compressed entry and keeps the top-k.  Scores are
// exact int32 dot products of int8 vectors (dp4a), the order is (score desc,
// index asc), so the selected set is unique and the result bit-exact.
//
// Scores are biased to a non-negative key u = s + DI*16256 < DI*32640, which has
// `key_bits` bits.  Selection is a two-level radix threshold:
//   1. scan  (grid: chunks x rows): dp4a scores of one chunk of entries, keys
//      stored to the workspace, a 256-bin histogram of u >> shift1 merged into a
//      per-row global histogram.  The last CTA of a row (atomic ticket, no
//      waiting) finds the bin b1 that holds the k-th largest key.
//   2. collect (same grid): each chunk compacts its keys with bin >= b1, in
//      index order, into a per-row candidate list (one atomic per CTA).  The
//      last CTA of the row resolves the exact threshold key T inside bin b1
//      with a level-2 histogram over the low bits, breaks ties at T by
//      ascending index, and writes the result in ascending index order.
//      If the candidates overflow their capacity (heavily tied scores) the
//      same CTA falls back to an exact pass over all of the row's keys.
// Every workspace counter that a call uses is returned to zero by that call.
#include "block_scan.cuh"
#include "common.cuh"
#include "internal.h"

namespace hsa {

namespace {

constexpr int kThreads = 256;
constexpr int kBins1 = 256;

struct RowSel {
    int b1, count_above, n_cand, kE;
};

__device__ __forceinline__ uint32_t *keys_of(void *ws, const IndexPlan &p, int r) {
    return reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + p.off_keys) + (size_t)r * p.nchunks * p.chunk;
}
__device__ __forceinline__ uint32_t *hist1_of(void *ws, const IndexPlan &p, int r) {
    return reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + p.off_hist1) + (size_t)r * kBins1;
}
__device__ __forceinline__ uint32_t *tick_of(void *ws, const IndexPlan &p, int r) {
    return reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + p.off_tick) + (size_t)r * 4;
}
__device__ __forceinline__ RowSel *sel_of(void *ws, const IndexPlan &p, int r) {
    return reinterpret_cast<RowSel *>(static_cast<char *>(ws) + p.off_sel) + r;
}
__device__ __forceinline__ uint2 *runs_of(void *ws, const IndexPlan &p, int r) {
    return reinterpret_cast<uint2 *>(static_cast<char *>(ws) + p.off_runs) + (size_t)r * p.nchunks;
}
__device__ __forceinline__ uint32_t *cand_u_of(void *ws, const IndexPlan &p, int r) {
    return reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + p.off_cand_u) + (size_t)r * p.cap;
}
__device__ __forceinline__ int32_t *cand_j_of(void *ws, const IndexPlan &p, int r) {
    return reinterpret_cast<int32_t *>(static_cast<char *>(ws) + p.off_cand_j) + (size_t)r * p.cap;
}

// Row bookkeeping shared by both kernels.
struct RowInfo {
    int b, t;
    int64_t E;
};
__device__ __forceinline__ RowInfo row_info(const IndexArgs &a, int row) {
    RowInfo ri;
    ri.b = row / a.T;
    ri.t = row - ri.b * a.T;
    const int64_t p = a.q_pos0[ri.b] + ri.t;
    ri.E = num_entries(p, a.m);
    if (ri.E > a.E_cap) ri.E = a.E_cap;  // flagged by the scan kernel
    return ri;
}

__device__ __forceinline__ int dot16(const int4 &x, const int4 &y) {
    int s = __dp4a(x.x, y.x, 0);
    s = __dp4a(x.y, y.y, s);
    s = __dp4a(x.z, y.z, s);
    return __dp4a(x.w, y.w, s);
}

template <int LPE>  // lanes per entry = DI / 16
__global__ void __launch_bounds__(kThreads) index_scan_kernel(IndexArgs a, IndexPlan p, void *ws, int row_begin) {
    __shared__ unsigned s_hist[kBins1];
    __shared__ int s_scan[33];
    __shared__ int s_last;
    __shared__ int s_b1;

    const int lrow = blockIdx.y;
    const int row = row_begin + lrow;
    const RowInfo ri = row_info(a, row);
    {
        const int64_t p_ = a.q_pos0[ri.b] + ri.t;
        if (num_entries(p_, a.m) > a.E_cap && blockIdx.x == 0 && threadIdx.x == 0) raise_flag(FLAG_INDEX_RANGE);
    }
    const int64_t c0 = (int64_t)blockIdx.x * p.chunk;
    if (c0 >= ri.E) return;
    const int n = (int)(int)(ri.E - c0 < p.chunk ? ri.E - c0 : p.chunk);
    const int nch = (int)((ri.E + p.chunk - 1) / p.chunk);

    for (int i = threadIdx.x; i < kBins1; i += kThreads) s_hist[i] = 0;

    const int lane_e = threadIdx.x % LPE;
    const int grp = threadIdx.x / LPE;
    constexpr int kGroups = kThreads / LPE;
    const int4 qv = *reinterpret_cast<const int4 *>(a.q + ri.b * a.q_sb + (int64_t)ri.t * a.q_st + lane_e * 16);
    const int bias = a.DI * 16256;
    const char *kbase = reinterpret_cast<const char *>(a.k + ri.b * a.k_sb) + lane_e * 16;
    uint32_t *keys = keys_of(ws, p, lrow) + c0;
    __syncthreads();

    constexpr int U = 8;
    for (int e0 = 0; e0 < n; e0 += kGroups * U) {
        int4 kv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * kGroups + grp;
            if (e < n) kv[u] = ld_nc_v4(kbase + (c0 + e) * a.k_se);
            else kv[u] = make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            int s = dot16(qv, kv[u]);
#pragma unroll
            for (int o = 1; o < LPE; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            const int e = e0 + u * kGroups + grp;
            if (lane_e == 0 && e < n) {
                const uint32_t key = (uint32_t)(s + bias);
                keys[e] = key;
                atomicAdd(&s_hist[key >> p.shift1], 1u);
            }
        }
    }
    __syncthreads();
    uint32_t *gh = hist1_of(ws, p, lrow);
    for (int i = threadIdx.x; i < kBins1; i += kThreads)
        if (s_hist[i]) atomicAdd(&gh[i], s_hist[i]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned tk = atomicAdd(&tick_of(ws, p, lrow)[0], 1u);
        s_last = (tk == (unsigned)(nch - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // Last CTA of the row: find bin b1 of the kE-th largest key.
    const int kE = (int)(ri.E < a.topk ? ri.E : a.topk);
    const int bin = kBins1 - 1 - threadIdx.x;  // thread i owns bin 255-i (descending)
    const int h = (int)__ldcg(&gh[bin]);
    int tot;
    const int before = block_exclusive_sum(h, s_scan, tot);  // keys in bins above `bin`
    if (threadIdx.x == 0) s_b1 = -1;
    __syncthreads();
    if (before < kE && before + h >= kE) {
        s_b1 = bin;
        RowSel rs;
        rs.b1 = bin;
        rs.count_above = before;
        rs.n_cand = before + h;
        rs.kE = kE;
        *sel_of(ws, p, lrow) = rs;
    }
    __syncthreads();
    gh[bin] = 0;  // leave the workspace zeroed for the next call
    if (threadIdx.x == 0) tick_of(ws, p, lrow)[0] = 0;
}

// Find T2 = the largest level-2 bin whose suffix count reaches `need` and the
// number of keys of bin b1 strictly above it.  hist has nb bins (multiple of kThreads).
__device__ __forceinline__ void find_level2(const unsigned *hist, int nb, int need, int *s_scan, int *s_out) {
    const int per = nb / kThreads;
    // thread i owns bins [nb-1-i*per, nb-1-(i+1)*per+1], visited in descending order
    const int top = nb - 1 - threadIdx.x * per;
    int local = 0;
    for (int q = 0; q < per; ++q) local += (int)hist[top - q];
    int tot;
    const int before = block_exclusive_sum(local, s_scan, tot);
    if (before < need && before + local >= need) {
        int cum = before;
        for (int q = 0; q < per; ++q) {
            const int hv = (int)hist[top - q];
            if (cum + hv >= need) {
                s_out[0] = top - q;  // T2
                s_out[1] = cum;      // keys of bin b1 above T2
                break;
            }
            cum += hv;
        }
    }
    __syncthreads();
}

template <int LPE>
__global__ void __launch_bounds__(kThreads) index_collect_kernel(IndexArgs a, IndexPlan p, void *ws, int row_begin) {
    extern __shared__ unsigned s_dyn[];  // level-2 histogram (1 << shift1 bins), then candidates
    __shared__ int s_scan[33];
    __shared__ int s_last;
    __shared__ int s_thr[2];
    __shared__ int s_base[2];

    const int lrow = blockIdx.y;
    const int row = row_begin + lrow;
    const RowInfo ri = row_info(a, row);
    int32_t *idx_out = a.idx_out + (size_t)row * a.topk;
    if (ri.E == 0) {
        if (blockIdx.x == 0) {
            for (int i = threadIdx.x; i < a.topk; i += kThreads) idx_out[i] = -1;
            if (threadIdx.x == 0) a.cnt_out[row] = 0;
        }
        return;
    }
    const int64_t c0 = (int64_t)blockIdx.x * p.chunk;
    if (c0 >= ri.E) return;
    const int n = (int)(int)(ri.E - c0 < p.chunk ? ri.E - c0 : p.chunk);
    const int nch = (int)((ri.E + p.chunk - 1) / p.chunk);
    RowSel rs;
    {
        const int4 v = __ldcg(reinterpret_cast<const int4 *>(sel_of(ws, p, lrow)));
        rs.b1 = v.x;
        rs.count_above = v.y;
        rs.n_cand = v.z;
        rs.kE = v.w;
    }
    const bool overflow = rs.n_cand > p.cap;
    const uint32_t *keys_row = keys_of(ws, p, lrow);
    uint32_t *tick = tick_of(ws, p, lrow);

    // ---- 1. per-chunk ordered compaction of keys in bin >= b1
    if (!overflow) {
        // stage the chunk's keys in shared memory with coalesced 16-byte loads
        uint32_t *s_keys = s_dyn;
        const uint4 *src4 = reinterpret_cast<const uint4 *>(keys_row + c0);
        for (int i = threadIdx.x; i < p.chunk / 4; i += kThreads)
            reinterpret_cast<uint4 *>(s_keys)[i] = __ldcg(&src4[i]);
        __syncthreads();
        const int per = p.chunk / kThreads;  // consecutive keys per thread
        const int my0 = threadIdx.x * per;
        int cntl = 0;
        for (int q = 0; q < per; ++q) {
            const int e = my0 + q;
            if (e < n && (int)(s_keys[e] >> p.shift1) >= rs.b1) ++cntl;
        }
        int tot;
        const int pre = block_exclusive_sum(cntl, s_scan, tot);
        if (threadIdx.x == 0) {
            const unsigned off = tot ? atomicAdd(&tick[2], (unsigned)tot) : 0u;
            s_base[0] = (int)off;
            runs_of(ws, p, lrow)[blockIdx.x] = make_uint2(off, (unsigned)tot);
        }
        __syncthreads();
        const int base = s_base[0] + pre;
        uint32_t *cu = cand_u_of(ws, p, lrow);
        int32_t *cj = cand_j_of(ws, p, lrow);
        int w = 0;
        for (int q = 0; q < per; ++q) {
            const int e = my0 + q;
            if (e < n) {
                const uint32_t u = s_keys[e];
                if ((int)(u >> p.shift1) >= rs.b1) {
                    if (base + w < p.cap) {
                        cu[base + w] = u;
                        cj[base + w] = (int32_t)(c0 + e);
                    }
                    ++w;
                }
            }
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned tk = atomicAdd(&tick[1], 1u);
        s_last = (tk == (unsigned)(nch - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- 2. last CTA of the row: exact threshold and ordered output
    const int nb2 = 1 << p.shift1;
    unsigned *hist2 = s_dyn;
    for (int i = threadIdx.x; i < nb2; i += kThreads) hist2[i] = 0;
    const int need = rs.kE - rs.count_above;  // >= 1 by the choice of b1
    const uint32_t mask2 = (uint32_t)nb2 - 1u;
    __syncthreads();

    if (!overflow) {
        // Gather the candidates in ascending index order (runs are per chunk, chunks ascend).
        int *s_runpre = reinterpret_cast<int *>(hist2 + nb2);       // [nch + 1]
        uint32_t *s_u = reinterpret_cast<uint32_t *>(s_runpre + p.nchunks + 1);
        int32_t *s_j = reinterpret_cast<int32_t *>(s_u + p.cap);
        const uint2 *runs = runs_of(ws, p, lrow);
        // prefix over runs (nch may exceed the thread count)
        int carry = 0;
        for (int c_ = 0; c_ < nch; c_ += kThreads) {
            const int c = c_ + threadIdx.x;
            const int v = c < nch ? (int)__ldcg(&runs[c].y) : 0;
            int tot;
            const int pre = block_exclusive_sum(v, s_scan, tot);
            if (c < nch) s_runpre[c] = carry + pre;
            carry += tot;
        }
        if (threadIdx.x == 0) s_runpre[nch] = carry;
        __syncthreads();
        const int ncand = carry;  // == rs.n_cand
        const uint32_t *cu = cand_u_of(ws, p, lrow);
        const int32_t *cj = cand_j_of(ws, p, lrow);
        for (int g = threadIdx.x; g < ncand; g += kThreads) {
            int lo = 0, hi = nch - 1;  // last run with s_runpre[run] <= g
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_runpre[mid] <= g) lo = mid;
                else hi = mid - 1;
            }
            const int src = (int)__ldcg(&runs[lo].x) + (g - s_runpre[lo]);
            const uint32_t u = __ldcg(&cu[src]);
            s_u[g] = u;
            s_j[g] = __ldcg(&cj[src]);
            if ((int)(u >> p.shift1) == rs.b1) atomicAdd(&hist2[u & mask2], 1u);
        }
        __syncthreads();
        find_level2(hist2, nb2, need, s_scan, s_thr);
        const uint32_t T = ((uint32_t)rs.b1 << p.shift1) | (uint32_t)s_thr[0];
        const int n_eq_need = need - s_thr[1];
        // ordered compaction over the candidates
        const int per = (ncand + kThreads - 1) / kThreads;
        const int my0 = threadIdx.x * per;
        int eq = 0;
        for (int q = 0; q < per; ++q) {
            const int g = my0 + q;
            if (g < ncand && s_u[g] == T) ++eq;
        }
        int tot;
        int eqrank = block_exclusive_sum(eq, s_scan, tot);
        int nsel = 0;
        {
            int er = eqrank;
            for (int q = 0; q < per; ++q) {
                const int g = my0 + q;
                if (g >= ncand) break;
                const uint32_t u = s_u[g];
                if (u > T) ++nsel;
                else if (u == T) { if (er < n_eq_need) ++nsel; ++er; }
            }
        }
        int pos = block_exclusive_sum(nsel, s_scan, tot);
        for (int q = 0; q < per; ++q) {
            const int g = my0 + q;
            if (g >= ncand) break;
            const uint32_t u = s_u[g];
            bool take = false;
            if (u > T) take = true;
            else if (u == T) { take = eqrank < n_eq_need; ++eqrank; }
            if (take) idx_out[pos++] = s_j[g];
        }
    } else {
        // Exact fallback: two passes over every key of the row, in index order.
        for (int64_t e = threadIdx.x; e < ri.E; e += kThreads) {
            const uint32_t u = __ldcg(&keys_row[e]);
            if ((int)(u >> p.shift1) == rs.b1) atomicAdd(&hist2[u & mask2], 1u);
        }
        __syncthreads();
        find_level2(hist2, nb2, need, s_scan, s_thr);
        const uint32_t T = ((uint32_t)rs.b1 << p.shift1) | (uint32_t)s_thr[0];
        const int n_eq_need = need - s_thr[1];
        constexpr int PER = 16;
        int eq_base = 0, pos_base = 0;
        for (int64_t t0 = 0; t0 < ri.E; t0 += (int64_t)kThreads * PER) {
            const int64_t my0 = t0 + (int64_t)threadIdx.x * PER;
            uint32_t uu[PER];
            int eq = 0;
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int64_t e = my0 + q;
                uu[q] = e < ri.E ? __ldcg(&keys_row[e]) : 0u;
                if (e < ri.E && uu[q] == T) ++eq;
            }
            int tot_eq;
            int eqrank = eq_base + block_exclusive_sum(eq, s_scan, tot_eq);
            int nsel = 0;
            {
                int er = eqrank;
#pragma unroll
                for (int q = 0; q < PER; ++q) {
                    const int64_t e = my0 + q;
                    if (e >= ri.E) break;
                    if (uu[q] > T) ++nsel;
                    else if (uu[q] == T) { if (er < n_eq_need) ++nsel; ++er; }
                }
            }
            int tot_sel;
            int pos = pos_base + block_exclusive_sum(nsel, s_scan, tot_sel);
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int64_t e = my0 + q;
                if (e >= ri.E) break;
                bool take = false;
                if (uu[q] > T) take = true;
                else if (uu[q] == T) { take = eqrank < n_eq_need; ++eqrank; }
                if (take) idx_out[pos++] = (int32_t)e;
            }
            eq_base += tot_eq;
            pos_base += tot_sel;
        }
    }
    for (int i = rs.kE + threadIdx.x; i < a.topk; i += kThreads) idx_out[i] = -1;
    if (threadIdx.x == 0) {
        a.cnt_out[row] = rs.kE;
        tick[1] = 0;
        tick[2] = 0;
    }
}

int key_bits_for(int DI) {
    const long long maxkey = (long long)DI * 32640;  // (127 + 128) * 128 per channel, exclusive bound
    int kb = 0;
    while ((1ll << kb) <= maxkey) ++kb;
    return kb;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

IndexPlan plan_index(int rows, int DI, int64_t E_cap, int topk, int num_sms) {
    IndexPlan p{};
    p.rows = rows;
    // entries per CTA: aim for >= 2 waves of CTAs over the SMs, 1024..8192 entries each
    int64_t per = (E_cap * rows) / (2ll * num_sms);
    int chunk = 1024;
    while (chunk < 8192 && chunk < per) chunk <<= 1;
    p.chunk = chunk;
    p.nchunks = (int)((E_cap + chunk - 1) / chunk);
    if (p.nchunks < 1) p.nchunks = 1;
    p.key_bits = key_bits_for(DI);
    p.shift1 = p.key_bits - 8;
    p.cap = 4096;
    size_t off = 0;
    p.off_keys = off;
    off = align256(off + sizeof(uint32_t) * (size_t)rows * p.nchunks * p.chunk);
    p.off_hist1 = off;
    off = align256(off + sizeof(uint32_t) * (size_t)rows * kBins1);
    p.off_tick = off;
    off = align256(off + sizeof(uint32_t) * 4 * (size_t)rows);
    p.off_sel = off;
    off = align256(off + sizeof(int) * 4 * (size_t)rows);
    p.off_runs = off;
    off = align256(off + sizeof(uint2) * (size_t)rows * p.nchunks);
    p.off_cand_u = off;
    off = align256(off + sizeof(uint32_t) * (size_t)rows * p.cap);
    p.off_cand_j = off;
    off = align256(off + sizeof(int32_t) * (size_t)rows * p.cap);
    p.total = off;
    (void)topk;
    return p;
}

static size_t collect_smem(const IndexPlan &p) {
    const size_t fin = sizeof(unsigned) * ((size_t)1 << p.shift1) + sizeof(int) * (p.nchunks + 1) +
                       (sizeof(uint32_t) + sizeof(int32_t)) * (size_t)p.cap;
    const size_t stage = sizeof(uint32_t) * (size_t)p.chunk;
    return fin > stage ? fin : stage;
}

template <int LPE>
static cudaError_t launch_lpe(const IndexArgs &a, const IndexPlan &p, void *ws, int row_begin, int rows,
                              cudaStream_t s) {
    dim3 grid(p.nchunks, rows);
    index_scan_kernel<LPE><<<grid, kThreads, 0, s>>>(a, p, ws, row_begin);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = collect_smem(p);
    static unsigned long long done = 0;
    e = smem_limit_once(index_collect_kernel<LPE>, 200 * 1024, done);
    if (e != cudaSuccess) return e;
    index_collect_kernel<LPE><<<grid, kThreads, smem, s>>>(a, p, ws, row_begin);
    return cudaGetLastError();
}

cudaError_t launch_index_topk(const IndexArgs &a, const IndexPlan &p, void *ws, int row_begin,
                              cudaStream_t s) {
    const int rows = min(p.rows, a.B * a.T - row_begin);
    switch (a.DI / 16) {
        case 1: return launch_lpe<1>(a, p, ws, row_begin, rows, s);
        case 2: return launch_lpe<2>(a, p, ws, row_begin, rows, s);
        case 4: return launch_lpe<4>(a, p, ws, row_begin, rows, s);
        case 8: return launch_lpe<8>(a, p, ws, row_begin, rows, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace hsa
