// Lightning indexer + exact top-k, decode-shaped: one cooperative launch.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制, CSA step 2 (score every
// visible compressed entry against the query, keep the top-k).  Same result as
// the two-kernel path in index_topk.cu, in one launch whose CTAs of a row meet
// at two row barriers (the launch is cooperative, so all CTAs are resident and
// every barrier completes; each wait is still bounded and raises the device
// flag if it ever gives up):
//   phase 1  dp4a scores of this CTA's chunk, kept in shared memory as biased
//            keys u = s + DI*16256; a 2048-bin histogram of u >> shift1 is
//            merged into the row's global histogram.               -- barrier
//   phase 2  every CTA reads the row histogram and finds the bin b1 holding
//            the k-th largest key; it publishes its count of keys above b1
//            and appends its keys inside b1 to the row's in-bin list.  -- barrier
//   phase 3  every CTA resolves the exact threshold key T and the number of
//            ties at T to take (by ascending index) from the small in-bin list,
//            then writes its own chunk's winners, in index order, at the
//            offset given by the earlier chunks.  The last CTA to finish
//            returns the row's histogram and counters to zero.
// If the in-bin list overflows its capacity (heavily tied scores) the keys are
// spilled to the workspace and the first CTA of the row does an exact
// row-wide pass instead.
#include "block_scan.cuh"
#include "common.cuh"
#include "internal.h"

namespace hsa {

namespace {

constexpr int kThreads = 256;
constexpr int kNB1 = 2048;
constexpr unsigned long long kSpinLimit = 1ull << 24;
constexpr int kStages = 3;
constexpr int kSlot = 7;     // in-bin (key, index) pairs carried by a chunk record
constexpr int kBrute = 512;  // in-bin lists up to this size are ranked by brute force
constexpr int kStageBytes = 16384;

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Row barrier: every participating CTA adds one, then waits for `target`.
// Returns false (and raises the device flag) if the wait gives up.
__device__ __forceinline__ bool row_barrier(unsigned *ctr, unsigned target, int *s_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
        unsigned long long it = 0;
        int ok = 1;
        while (ld_acquire(ctr) < target) {
            if (++it > kSpinLimit) {
                raise_flag(FLAG_INDEX_RANGE | 0x100u);
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
        *s_flag = ok;
    }
    __syncthreads();
    return *s_flag != 0;
}

__device__ __forceinline__ int dot16(const int4 &x, const int4 &y) {
    int s = __dp4a(x.x, y.x, 0);
    s = __dp4a(x.y, y.y, s);
    s = __dp4a(x.z, y.z, s);
    return __dp4a(x.w, y.w, s);
}

struct Ws {
    unsigned *hist1;  // [rows][kNB1]
    unsigned *bar;    // [rows][4]: barrier, in-bin count, exit count, pad
    uint32_t *in_u;   // [rows][cap_in]
    int32_t *in_j;    // [rows][cap_in]
    uint32_t *keys;   // [rows][C*chunk] (heavy ties only)
    int *rec;         // [rows][C][16] chunk records
};
__device__ __forceinline__ Ws carve(void *ws, const FusedIndexPlan &p, int r) {
    char *b = static_cast<char *>(ws);
    Ws w;
    w.hist1 = reinterpret_cast<unsigned *>(b + p.off_hist1) + (size_t)r * kNB1;
    w.bar = reinterpret_cast<unsigned *>(b + p.off_bar) + (size_t)r * 4;
    w.in_u = reinterpret_cast<uint32_t *>(b + p.off_in_u) + (size_t)r * p.cap_in;
    w.in_j = reinterpret_cast<int32_t *>(b + p.off_in_j) + (size_t)r * p.cap_in;
    w.keys = reinterpret_cast<uint32_t *>(b + p.off_keys) + (size_t)r * p.ctas_per_row * p.chunk;
    w.rec = reinterpret_cast<int *>(b + p.off_rec) + (size_t)r * p.ctas_per_row * 16;
    return w;
}

// T2 = largest level-2 bin whose suffix count reaches `need`; out[1] = keys above it.
__device__ __forceinline__ void find_threshold(const unsigned *hist, int nb, int need, int *s_scan, int *s_out) {
    const int per = nb / kThreads;
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
                s_out[0] = top - q;
                s_out[1] = cum;
                break;
            }
            cum += hv;
        }
    }
    __syncthreads();
}

template <int LPE>
__global__ void __launch_bounds__(kThreads) index_fused_kernel(IndexArgs a, FusedIndexPlan p, void *ws) {
    // a kernel launched after this one with programmatic stream serialization (the
    // decode attention) may be scheduled now; it waits for this grid's completion
    // before it reads anything
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t *s_keys = reinterpret_cast<uint32_t *>(smem);          // [chunk], kept over all phases
    unsigned *s_h = reinterpret_cast<unsigned *>(smem + (size_t)p.chunk * 4);  // [max(kNB1, nb2)]
    __shared__ int s_scan[33];
    __shared__ int s_misc[8];

    const int row = blockIdx.y;
    const int b = row / a.T, t = row - (row / a.T) * a.T;
    const int64_t pos = a.q_pos0[b] + t;
    int64_t E = num_entries(pos, a.m);
    if (E > a.E_cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_flag(FLAG_INDEX_RANGE);
        E = a.E_cap;
    }
    int32_t *idx_out = a.idx_out + (size_t)row * a.topk;
    const int kE = (int)(E < a.topk ? E : a.topk);
    if (blockIdx.x == 0) {
        for (int i = kE + threadIdx.x; i < a.topk; i += kThreads) idx_out[i] = -1;
        if (threadIdx.x == 0) a.cnt_out[row] = kE;
    }
    if (E == 0) return;
    const int nch = (int)((E + p.chunk - 1) / p.chunk);
    const int c = blockIdx.x;
    if (c >= nch) return;
    const int64_t c0 = (int64_t)c * p.chunk;
    const int n = (int)(E - c0 < p.chunk ? E - c0 : p.chunk);
    const Ws w = carve(ws, p, row);

    // ---------------------------------------------------------------- phase 1
    for (int i = threadIdx.x; i < kNB1; i += kThreads) s_h[i] = 0;
    const int lane_e = threadIdx.x % LPE, grp = threadIdx.x / LPE;
    constexpr int kGroups = kThreads / LPE;
    const int4 qv = *reinterpret_cast<const int4 *>(a.q + b * a.q_sb + (int64_t)t * a.q_st + lane_e * 16);
    const int bias = a.DI * 16256;
    auto score_one = [&](const int4 &kv, int e, bool valid) {
        int s = dot16(qv, kv);
#pragma unroll
        for (int o = 1; o < LPE; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane_e == 0 && valid) {
            const uint32_t key = (uint32_t)(s + bias);
            s_keys[e] = key;
            atomicAdd(&s_h[key >> p.shift1], 1u);
        }
    };
    if (a.k_se == a.DI) {
        // Contiguous chunk: stream it through a ring of shared-memory stages with
        // bulk asynchronous copies (one thread issues, mbarriers count bytes).
        unsigned char *s_stage = smem + p.off_stage_smem;
        __shared__ __align__(8) uint64_t s_bar[kStages];
        const int eps = kStageBytes / a.DI;  // entries per stage
        const int nst = (n + eps - 1) / eps;
        const char *src = reinterpret_cast<const char *>(a.k + b * a.k_sb + c0 * a.k_se);
        if (threadIdx.x == 0) {
            for (int st = 0; st < kStages; ++st) mbar_init(&s_bar[st], 1);
            fence_mbar_init();
        }
        __syncthreads();
        auto issue = [&](int it) {
            const int st = it % kStages;
            const int ne = min(eps, n - it * eps);
            const unsigned bytes = (unsigned)(ne * a.DI);
            mbar_expect_tx(&s_bar[st], bytes);
            bulk_g2s(s_stage + st * kStageBytes, src + (int64_t)it * kStageBytes, bytes, &s_bar[st]);
        };
        if (threadIdx.x == 0)
            for (int it = 0; it < nst && it < kStages; ++it) issue(it);
        bool ok = true;
        int it = 0;
        for (; it < nst; ++it) {
            const int st = it % kStages;
            if (!mbar_wait(&s_bar[st], (unsigned)((it / kStages) & 1))) {
                ok = false;
                break;
            }
            const int ne = min(eps, n - it * eps);
            const unsigned char *base = s_stage + st * kStageBytes + lane_e * 16;
            for (int el0 = 0; el0 < ne; el0 += kGroups) {
                const int el = el0 + grp;
                const bool valid = el < ne;
                const int4 kv = valid ? *reinterpret_cast<const int4 *>(base + el * a.DI) : make_int4(0, 0, 0, 0);
                score_one(kv, it * eps + el, valid);
            }
            __syncthreads();  // stage consumed by every thread
            if (threadIdx.x == 0 && it + kStages < nst) issue(it + kStages);
        }
        if (!ok) {
            // an mbarrier wait gave up: flag it, let the copies already issued land, leave
            raise_flag(FLAG_INDEX_RANGE | 0x200u);
            for (int j = it; j < nst && j < it + kStages; ++j) mbar_wait(&s_bar[j % kStages], (unsigned)((j / kStages) & 1));
            __syncthreads();
            return;
        }
    } else {
        const char *kbase = reinterpret_cast<const char *>(a.k + b * a.k_sb) + lane_e * 16;
        __syncthreads();
        constexpr int U = 8;
        for (int e0 = 0; e0 < n; e0 += kGroups * U) {
            int4 kv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = e0 + u * kGroups + grp;
                kv[u] = e < n ? ld_nc_v4(kbase + (c0 + e) * a.k_se) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = e0 + u * kGroups + grp;
                score_one(kv[u], e, e < n);
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kNB1; i += kThreads)
        if (s_h[i]) atomicAdd(&w.hist1[i], s_h[i]);
    if (!row_barrier(&w.bar[0], (unsigned)nch, &s_misc[7])) return;

    // ---------------------------------------------------------------- phase 2
    // One read of the row histogram gives b1; this chunk publishes a fixed-size
    // record {keys above b1, keys in b1, up to kSlot (key, index) pairs in b1}
    // with plain stores; in-bin keys beyond kSlot go to the row overflow list.
    __shared__ int s_cnt_above, s_cnt_in, s_list_n, s_above_before, s_sel_before;
    __shared__ uint32_t s_slot_u[kSlot];
    __shared__ int32_t s_slot_j[kSlot];
    constexpr int PB = kNB1 / kThreads;  // bins per thread, descending
    if (threadIdx.x == 0) {
        s_cnt_above = 0;
        s_cnt_in = 0;
        s_list_n = 0;
        s_above_before = 0;
        s_sel_before = 0;
    }
    {
        const int top = kNB1 - 1 - threadIdx.x * PB;
        int hv[PB];
        int local = 0;
#pragma unroll
        for (int q = 0; q < PB; ++q) {
            hv[q] = (int)__ldcg(&w.hist1[top - q]);
            local += hv[q];
        }
        int tot;
        const int before = block_exclusive_sum(local, s_scan, tot);
        if (before < kE && before + local >= kE) {
            int cum = before;
#pragma unroll
            for (int q = 0; q < PB; ++q) {
                if (cum + hv[q] >= kE) {
                    s_misc[0] = top - q;  // b1
                    s_misc[1] = cum;      // keys in bins above b1
                    s_misc[2] = hv[q];    // keys in b1
                    break;
                }
                cum += hv[q];
            }
        }
        __syncthreads();
    }
    const int b1 = s_misc[0], count_above = s_misc[1], n_in = s_misc[2];
    const bool spill = n_in > p.cap_in;  // heavily tied scores: exact pass over spilled keys
    const int per = (p.chunk + kThreads - 1) / kThreads;
    const int my0 = threadIdx.x * per;
    {
        int above = 0;
        for (int q = 0; q < per; ++q) {
            const int e = my0 + q;
            if (e < n) {
                const uint32_t u = s_keys[e];
                const int bin = (int)(u >> p.shift1);
                above += bin > b1;
                if (bin == b1) {
                    const int k = atomicAdd(&s_cnt_in, 1);
                    if (k < kSlot) {
                        s_slot_u[k] = u;
                        s_slot_j[k] = (int32_t)(c0 + e);
                    } else if (!spill) {
                        const unsigned o = atomicAdd(&w.bar[1], 1u);
                        if (o < (unsigned)p.cap_in) {
                            w.in_u[o] = u;
                            w.in_j[o] = (int32_t)(c0 + e);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
        if ((threadIdx.x & 31) == 0 && above) atomicAdd(&s_cnt_above, above);
    }
    __syncthreads();
    if (threadIdx.x < 16) {
        // record layout: {above, n_in, (u0, j0), ..., (u6, j6)}; unused pairs carry j = -1
        int v;
        if (threadIdx.x == 0) v = s_cnt_above;
        else if (threadIdx.x == 1) v = s_cnt_in;
        else {
            const int k = (threadIdx.x - 2) >> 1;
            const bool has = k < s_cnt_in && k < kSlot;
            v = (threadIdx.x & 1) == 0 ? (has ? (int)s_slot_u[k] : 0) : (has ? s_slot_j[k] : -1);
        }
        w.rec[(size_t)c * 16 + threadIdx.x] = v;
    }
    if (spill)
        for (int e = threadIdx.x; e < n; e += kThreads) w.keys[c0 + e] = s_keys[e];
    if (!row_barrier(&w.bar[0], 2u * (unsigned)nch, &s_misc[7])) return;

    // ---------------------------------------------------------------- phase 3
    const int need = kE - count_above;  // >= 1
    if (!spill) {
        // One read of every chunk's record (and of the overflow count) builds the
        // in-bin list in shared memory (the copy stages are free by now).
        uint2 *s_l = reinterpret_cast<uint2 *>(smem + p.off_stage_smem);  // [cap_in] (key, index)
        const int4 *rec4 = reinterpret_cast<const int4 *>(w.rec);
        int above_before = 0;
        for (int r = threadIdx.x; r < nch * 4; r += kThreads) {
            const int4 v = __ldcg(&rec4[r]);
            const int cc = r >> 2, qq = r & 3;
            if (qq == 0 && cc < c) above_before += v.x;
            if (qq != 0 && v.y >= 0) {
                const int k = atomicAdd(&s_list_n, 1);
                if (k < p.cap_in) s_l[k] = make_uint2((uint32_t)v.x, (uint32_t)v.y);
            }
            if (v.w >= 0) {
                const int k = atomicAdd(&s_list_n, 1);
                if (k < p.cap_in) s_l[k] = make_uint2((uint32_t)v.z, (uint32_t)v.w);
            }
        }
        const int n_ovf = (int)min(__ldcg(&w.bar[1]), (unsigned)p.cap_in);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) above_before += __shfl_xor_sync(0xffffffffu, above_before, o);
        if ((threadIdx.x & 31) == 0 && above_before) atomicAdd(&s_above_before, above_before);
        for (int i = threadIdx.x; i < n_ovf; i += kThreads) {
            const int k = atomicAdd(&s_list_n, 1);
            if (k < p.cap_in) s_l[k] = make_uint2(__ldcg(&w.in_u[i]), (uint32_t)__ldcg(&w.in_j[i]));
        }
        __syncthreads();
        const int nl = min(s_list_n, p.cap_in);  // == n_in
        // Decide every in-bin key; count the selected ones that precede this chunk
        // and mark those inside it (bit 31 of its shared-memory key; keys < 2^23).
        int sel_before = 0;
        auto settle = [&](uint32_t j, bool take) {
            if (!take) return;
            if ((int64_t)j < c0) ++sel_before;
            else if ((int64_t)j < c0 + n) s_keys[j - c0] |= 0x80000000u;
        };
        if (nl <= kBrute) {
            // rank = in-bin keys that beat key i under (key desc, index asc)
            for (int i = threadIdx.x; i < nl; i += kThreads) {
                const uint2 me = s_l[i];
                int rank = 0;
#pragma unroll 8
                for (int k = 0; k < nl; ++k) {
                    const uint2 o = s_l[k];
                    rank += (o.x > me.x) | ((o.x == me.x) & (o.y < me.y));
                }
                settle(me.y, rank < need);
            }
        } else {
            // level-2 histogram over the low bits of the in-bin keys
            unsigned *s_h2 = s_h;
            const uint32_t mask2 = (uint32_t)p.nb2 - 1u;
            for (int i = threadIdx.x; i < p.nb2; i += kThreads) s_h2[i] = 0;
            __syncthreads();
            for (int i = threadIdx.x; i < nl; i += kThreads) atomicAdd(&s_h2[s_l[i].x & mask2], 1u);
            __syncthreads();
            find_threshold(s_h2, p.nb2, need, s_scan, &s_misc[4]);
            const uint32_t T = ((uint32_t)b1 << p.shift1) | (uint32_t)s_misc[4];
            const int n_eq_need = need - s_misc[5];
            for (int i = threadIdx.x; i < nl; i += kThreads) {
                const uint2 me = s_l[i];
                bool take = me.x > T;
                if (me.x == T) {
                    int er = 0;
                    for (int k = 0; k < nl; ++k) er += (s_l[k].x == T) & (s_l[k].y < me.y);
                    take = er < n_eq_need;
                }
                settle(me.y, take);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sel_before += __shfl_xor_sync(0xffffffffu, sel_before, o);
        if ((threadIdx.x & 31) == 0 && sel_before) atomicAdd(&s_sel_before, sel_before);
        __syncthreads();
        const int base = s_above_before + s_sel_before;
        // this chunk, in index order
        auto taken = [&](uint32_t u) {
            return (int)((u & 0x7fffffffu) >> p.shift1) > b1 || (u & 0x80000000u);
        };
        int nsel = 0;
        for (int q = 0; q < per; ++q) {
            const int e = my0 + q;
            if (e < n) nsel += taken(s_keys[e]);
        }
        int tot;
        int o = base + block_exclusive_sum(nsel, s_scan, tot);
        for (int q = 0; q < per; ++q) {
            const int e = my0 + q;
            if (e < n && taken(s_keys[e])) idx_out[o++] = (int32_t)(c0 + e);
        }
    } else if (c == 0) {
        // exact row-wide pass over the spilled keys (heavily tied scores)
        unsigned *s_h2 = s_h;
        const uint32_t mask2 = (uint32_t)p.nb2 - 1u;
        for (int i = threadIdx.x; i < p.nb2; i += kThreads) s_h2[i] = 0;
        __syncthreads();
        for (int64_t e = threadIdx.x; e < E; e += kThreads) {
            const uint32_t u = __ldcg(&w.keys[e]);
            if ((int)(u >> p.shift1) == b1) atomicAdd(&s_h2[u & mask2], 1u);
        }
        __syncthreads();
        find_threshold(s_h2, p.nb2, need, s_scan, &s_misc[4]);
        const uint32_t T = ((uint32_t)b1 << p.shift1) | (uint32_t)s_misc[4];
        const int n_eq_need = need - s_misc[5];
        constexpr int PER = 16;
        int eq_base = 0, pos_base = 0;
        for (int64_t t0 = 0; t0 < E; t0 += (int64_t)kThreads * PER) {
            const int64_t m0 = t0 + (int64_t)threadIdx.x * PER;
            uint32_t uu[PER];
            int eq = 0;
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int64_t e = m0 + q;
                uu[q] = e < E ? __ldcg(&w.keys[e]) : 0u;
                eq += (e < E && uu[q] == T);
            }
            int tot_eq, tot_sel;
            int er = eq_base + block_exclusive_sum(eq, s_scan, tot_eq);
            int nsel = 0;
            {
                int er2 = er;
#pragma unroll
                for (int q = 0; q < PER; ++q) {
                    if (m0 + q >= E) break;
                    if (uu[q] > T) ++nsel;
                    else if (uu[q] == T) { nsel += er2 < n_eq_need; ++er2; }
                }
            }
            int o = pos_base + block_exclusive_sum(nsel, s_scan, tot_sel);
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int64_t e = m0 + q;
                if (e >= E) break;
                bool take = uu[q] > T;
                if (uu[q] == T) { take = er < n_eq_need; ++er; }
                if (take) idx_out[o++] = (int32_t)e;
            }
            eq_base += tot_eq;
            pos_base += tot_sel;
        }
    }

    // ---------------------------------------------------------------- exit
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_misc[6] = atomicAdd(&w.bar[2], 1u) == (unsigned)(nch - 1);
    }
    __syncthreads();
    if (s_misc[6]) {
        __threadfence();
        for (int i = threadIdx.x; i < kNB1; i += kThreads) w.hist1[i] = 0;
        if (threadIdx.x == 0) {
            w.bar[0] = 0;
            w.bar[1] = 0;
            w.bar[2] = 0;
        }
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int key_bits_for(int DI) {
    const long long maxkey = (long long)DI * 32640;
    int kb = 0;
    while ((1ll << kb) <= maxkey) ++kb;
    return kb;
}

template <int LPE>
int occupancy(size_t smem) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, index_fused_kernel<LPE>, kThreads, smem) != cudaSuccess)
        return 0;
    return occ;
}

// Occupancy per (indexer dim, shared memory in KiB), cached: the answer depends
// only on the kernel and its shared memory, and planning runs on every call.
int occupancy_for(int DI, size_t smem) {
    static unsigned long long done[4] = {0, 0, 0, 0};
    static int cache[4][232];
    static bool init = false;
    if (!init) {
        for (auto &r : cache)
            for (int &v : r) v = -1;
        init = true;
    }
    const int slot = DI == 16 ? 0 : DI == 32 ? 1 : DI == 64 ? 2 : 3;
    const int kb = (int)((smem + 1023) / 1024);
    if (kb >= 232) return 0;
    if (cache[slot][kb] >= 0) return cache[slot][kb];
    const size_t q = (size_t)kb * 1024;
    int occ = 0;
    switch (slot) {
        case 0: smem_limit_once(index_fused_kernel<1>, 200 * 1024, done[0]); occ = occupancy<1>(q); break;
        case 1: smem_limit_once(index_fused_kernel<2>, 200 * 1024, done[1]); occ = occupancy<2>(q); break;
        case 2: smem_limit_once(index_fused_kernel<4>, 200 * 1024, done[2]); occ = occupancy<4>(q); break;
        default: smem_limit_once(index_fused_kernel<8>, 200 * 1024, done[3]); occ = occupancy<8>(q); break;
    }
    cache[slot][kb] = occ;
    return occ;
}

}  // namespace

FusedIndexPlan plan_index_fused(int rows, int DI, int64_t E_cap, int num_sms) {
    FusedIndexPlan p{};
    p.ok = false;
    if (rows <= 0 || E_cap <= 0) return p;
    p.rows = rows;
    p.key_bits = key_bits_for(DI);
    p.shift1 = p.key_bits - 11;
    p.nb2 = 1 << p.shift1;
    p.cap_in = 4096;
    // Chunks are multiples of 64 entries; pick the smallest chunk whose launch
    // (ceil(E/chunk) CTAs per row) is resident all at once, so every SM streams
    // an equal share.
    for (int chunk = 256; chunk <= 16384; chunk += 64) {
        const int64_t C = (E_cap + chunk - 1) / chunk;
        const size_t base = (size_t)chunk * 4 + (size_t)4 * (kNB1 > p.nb2 ? kNB1 : p.nb2);
        const size_t stage_off = (base + 127) & ~(size_t)127;
        const size_t smem = stage_off + (size_t)kStages * kStageBytes;
        const int occ = occupancy_for(DI, smem);
        if (occ <= 0) return p;
        if (C * rows <= (int64_t)occ * num_sms) {
            p.chunk = chunk;
            p.ctas_per_row = (int)C;
            p.smem = ((smem + 1023) / 1024) * 1024;
            p.off_stage_smem = (int)stage_off;
            p.ok = true;
            break;
        }
    }
    if (!p.ok) return p;
    size_t off = 0;
    p.off_hist1 = off;
    off = align256(off + sizeof(unsigned) * kNB1 * (size_t)rows);
    p.off_bar = off;
    off = align256(off + sizeof(unsigned) * 4 * (size_t)rows);
    p.off_rec = off;
    off = align256(off + sizeof(int) * 16 * (size_t)p.ctas_per_row * rows);
    p.off_in_u = off;
    off = align256(off + sizeof(uint32_t) * (size_t)p.cap_in * rows);
    p.off_in_j = off;
    off = align256(off + sizeof(int32_t) * (size_t)p.cap_in * rows);
    p.off_keys = off;
    off = align256(off + sizeof(uint32_t) * (size_t)p.ctas_per_row * p.chunk * rows);
    p.total = off;
    return p;
}

template <int LPE>
static cudaError_t launch_fused_lpe(const IndexArgs &a, const FusedIndexPlan &p, void *ws, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas_per_row, p.rows);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, index_fused_kernel<LPE>, a, p, ws);
}

cudaError_t launch_index_fused(const IndexArgs &a, const FusedIndexPlan &p, void *ws, cudaStream_t s) {
    switch (a.DI / 16) {
        case 1: return launch_fused_lpe<1>(a, p, ws, s);
        case 2: return launch_fused_lpe<2>(a, p, ws, s);
        case 4: return launch_fused_lpe<4>(a, p, ws, s);
        case 8: return launch_fused_lpe<8>(a, p, ws, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace hsa
