// Lightning indexer + exact top-k, decode-shaped: one cooperative launch.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制, CSA step 2 (score every
// visible compressed entry against the query, keep the top-k).  Same result as
// the two-kernel path in index_topk.cu, in one launch whose CTAs of a row meet
// once at a row barrier (the launch is cooperative, so all CTAs are resident and
// the barrier completes; each wait is still bounded and raises the device flag
// if it ever gives up):
//   phase 1  dp4a scores of this CTA's chunk, kept in shared memory as biased
//            keys u = s + DI*16256; a 1024-bin histogram of u >> shift1 is
//            merged into the row's global histogram.               -- barrier
//   phase 2  every CTA reads the row histogram and finds the bin b1 holding
//            the k-th largest key; it writes its keys in bins >= b1 (key,
//            index), in index order, to its chunk's region of the row's
//            candidate list, and their count.  An atomic counter finds the last
//            CTA of the row to get here; the others leave.
//   phase 3  the last CTA reads the candidate list chunk after chunk (so in
//            index order), resolves the exact threshold key T inside b1 with a
//            level-2 histogram, takes the keys above T and the first ties at T,
//            writes the row's output and returns the row's histogram and
//            counter to zero.
// A chunk's region holds its whole chunk, so heavily tied scores (many keys in
// b1) only make phase 3 longer.
#include "block_scan.cuh"
#include "common.cuh"
#include "internal.h"

namespace hsa {

namespace {

constexpr int kThreads = 256;
constexpr int kNB1 = 1024;                    // level-1 histogram bins
constexpr unsigned long long kSpinLimit = 1ull << 24;
constexpr int kStages = 3;
constexpr int kStageBytes = 16384;

// Stores taken under a predicate without a branch around them (per-key branches
// in these loops cost several times the work they guard).
__device__ __forceinline__ void st_if(uint2 *p, uint2 v, bool pr) {
    asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %3, 0;\n @q st.global.v2.b32 [%0], {%1, %2};\n}\n" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"((int)pr)
                 : "memory");
}
__device__ __forceinline__ void st_if(int32_t *p, int32_t v, bool pr) {
    asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n @q st.global.b32 [%0], %1;\n}\n" ::"l"(p), "r"(v),
                 "r"((int)pr)
                 : "memory");
}

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
    unsigned *bar;    // [rows][4]: row counter, pad
    int *rec;         // [rows][C] candidates per chunk
    uint2 *cand;      // [rows][C * chunk] (key, index) in bins >= b1, chunk c at c * chunk
};
__device__ __forceinline__ Ws carve(void *ws, const FusedIndexPlan &p, int r) {
    char *b = static_cast<char *>(ws);
    Ws w;
    w.hist1 = reinterpret_cast<unsigned *>(b + p.off_hist1) + (size_t)r * kNB1;
    w.bar = reinterpret_cast<unsigned *>(b + p.off_bar) + (size_t)r * 4;
    w.rec = reinterpret_cast<int *>(b + p.off_rec) + (size_t)r * p.ctas_per_row;
    w.cand = reinterpret_cast<uint2 *>(b + p.off_cand) + (size_t)r * p.ctas_per_row * p.chunk;
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
    __shared__ int s_scan[66];
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
    // One read of the row histogram gives b1; this chunk appends its keys in bins
    // >= b1, as (key, index) in index order, to its region of the row's candidate
    // list and records how many.  The last CTA of the row to get here does phase 3;
    // the others leave.
    {
        constexpr int PB = kNB1 / kThreads;  // bins per thread, descending
        if (threadIdx.x == 0) s_misc[0] = s_misc[1] = s_misc[2] = 0;  // set below; defined even if never found
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
    {
        const int per = (p.chunk + kThreads - 1) / kThreads;
        const int my0 = threadIdx.x * per, my1 = min(n, my0 + per);
        int nc = 0;
        for (int e = my0; e < my1; ++e) nc += (int)(s_keys[e] >> p.shift1) >= b1;
        int tot;
        int o = block_exclusive_sum(nc, s_scan, tot);
        uint2 *cand = w.cand + c0;
        for (int e = my0; e < my1; ++e) {
            const uint32_t u = s_keys[e];
            const bool take = (int)(u >> p.shift1) >= b1;
            st_if(cand + o, make_uint2(u, (uint32_t)(c0 + e)), take);
            o += take;
        }
        if (threadIdx.x == 0) w.rec[c] = tot;
    }
    // every thread's candidates are ordered before thread 0's fence by the block
    // barrier; the fence and the counter publish them to the row's last CTA
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_misc[6] = atomicAdd(&w.bar[0], 1u) == 2u * (unsigned)nch - 1u;
    }
    __syncthreads();
    if (!s_misc[6]) return;
    __threadfence();

    // ---------------------------------------------------------------- phase 3
    // (last CTA of the row) The chunks' regions, one after another, list every key
    // in bins >= b1 in index order.  The first `spec` slots of every region are
    // loaded together with the regions' counts (slots past a count are never
    // used), so a typical row needs one round trip to L2; longer regions are read
    // by one flat pass over all threads.  The list is staged in shared memory in
    // index order while a level-2 histogram of the low bits of the keys in b1 is
    // built; it gives the threshold key T and how many keys equal to T to take (the
    // first ones in index order).  One ordered pass writes the winners.
    int *s_off = reinterpret_cast<int *>(smem + p.off_stage_smem);  // [nch + 1] list offsets
    int *s_roff = s_off + (nch + 1);                                 // [nch + 1] offsets past the first spec slots
    const int l_off = (2 * (nch + 1) * 4 + 15) & ~15;
    uint2 *s_l = reinterpret_cast<uint2 *>(smem + p.off_stage_smem + l_off);
    const int l_cap = (kStages * kStageBytes - l_off) / 8 - 1;  // slot l_cap takes the stores of empty slots
    unsigned *s_h2 = s_h;
    const uint32_t mask2 = (uint32_t)p.nb2 - 1u;
    for (int i = threadIdx.x; i < p.nb2; i += kThreads) s_h2[i] = 0;
    if (threadIdx.x == 0) s_misc[4] = s_misc[5] = 0;  // set by find_threshold; defined even if never found
    constexpr int kSpecPer = 16;  // speculative slot loads per thread
    int lg_spec = 5;
    while (lg_spec > 0 && (nch << lg_spec) > kThreads * kSpecPer) --lg_spec;
    const int spec = (nch << lg_spec) <= kThreads * kSpecPer ? 1 << lg_spec : 0;
    uint2 sv[kSpecPer];
#pragma unroll
    for (int q = 0; q < kSpecPer; ++q) {
        const int sp = q * kThreads + threadIdx.x;
        const int cc = spec ? sp >> lg_spec : nch;
        sv[q] = cc < nch ? __ldcg(w.cand + (int64_t)cc * p.chunk + (sp & (spec - 1))) : make_uint2(0u, 0u);
    }
    const int cpt = (nch + kThreads - 1) / kThreads;  // chunks per thread for the scans
    const int i0 = threadIdx.x * cpt;
    {
        int loc = 0, rest = 0;
        for (int q = 0; q < cpt; ++q)
            if (i0 + q < nch) {
                const int v = __ldcg(&w.rec[i0 + q]);
                s_off[i0 + q] = v;
                loc += v;
                rest += v > spec ? v - spec : 0;
            }
        int tot, rtot;
        const int2 orr = block_exclusive_sum2(loc, rest, s_scan, tot, rtot);
        int o = orr.x, ro = orr.y;
        for (int q = 0; q < cpt; ++q)
            if (i0 + q < nch) {
                const int v = s_off[i0 + q];
                s_off[i0 + q] = o;
                s_roff[i0 + q] = ro;
                o += v;
                ro += v > spec ? v - spec : 0;
            }
        if (threadIdx.x == 0) {
            s_off[nch] = tot;
            s_roff[nch] = rtot;
        }
        __syncthreads();
    }
    const int total = s_off[nch], n_rest = s_roff[nch];
    if (total != count_above + n_in && threadIdx.x == 0) raise_flag(FLAG_INDEX_RANGE | 0x400u);
    const bool staged = total <= l_cap;
    const int need = kE - count_above;  // >= 1
    // a key of b1 is counted in the level-2 histogram (rare: a branch)
    auto note_b1 = [&](const uint2 &v) {
        if ((int)(v.x >> p.shift1) == b1) atomicAdd(&s_h2[v.x & mask2], 1u);
    };
    auto take_in = [&](const uint2 &v, int L) {
        if (staged) s_l[L] = v;
        note_b1(v);
    };
#pragma unroll
    for (int q = 0; q < kSpecPer; ++q) {
        const int sp = q * kThreads + threadIdx.x;
        const int cc = spec ? min(sp >> lg_spec, nch) : nch;
        const int i = sp & (spec - 1);
        const int lo = s_off[min(cc, nch - 1)], hi = s_off[min(cc, nch - 1) + 1];
        const bool v = cc < nch && i < hi - lo;
        if (staged) s_l[v ? lo + i : l_cap] = sv[q];  // empty slots store into the spare slot
        if (v) note_b1(sv[q]);
    }
    // last c with off[c] <= L (off ascending over [0, nch])
    auto find_chunk = [&](const int *off, int L) {
        int lo = 0, hi = nch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (off[mid] <= L) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    };
    constexpr int PER = 8;
    for (int t0 = 0; t0 < n_rest; t0 += kThreads * PER) {
        uint2 v[PER];
        int lpos[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int R = t0 + q * kThreads + threadIdx.x;
            lpos[q] = -1;
            if (R < n_rest) {
                const int cc = find_chunk(s_roff, R);
                const int i = spec + (R - s_roff[cc]);
                lpos[q] = s_off[cc] + i;
                v[q] = __ldcg(w.cand + (int64_t)cc * p.chunk + i);
            }
        }
#pragma unroll
        for (int q = 0; q < PER; ++q)
            if (lpos[q] >= 0) take_in(v[q], lpos[q]);
    }
    __syncthreads();
    find_threshold(s_h2, p.nb2, need, s_scan, &s_misc[4]);
    const uint32_t T = ((uint32_t)b1 << p.shift1) | (uint32_t)s_misc[4];
    const int n_eq_need = need - s_misc[5];
    // One block scan per pass of packed per-thread counts (keys above T in the high
    // half, ties at T in the low half) places every winner: a key above T goes
    // after the keys above T and the ties taken before it, the j-th tie (in index
    // order) is taken while j < n_eq_need.
    int a_base = 0, e_base = 0;  // keys above T and ties in the passes before
    for (int t0 = 0; t0 < total; t0 += kThreads * PER) {
        const int m0 = t0 + threadIdx.x * PER;
        uint2 v[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int L = m0 + q;
            if (L >= total) v[q] = make_uint2(0u, 0u);
            else if (staged) v[q] = s_l[L];
            else {
                const int cc = find_chunk(s_off, L);
                v[q] = __ldcg(w.cand + (int64_t)cc * p.chunk + (L - s_off[cc]));
            }
        }
        int cg = 0, ce = 0;
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const bool in = m0 + q < total;
            cg += in && v[q].x > T;
            ce += in && v[q].x == T;
        }
        int tot;
        const int pre = block_exclusive_sum((cg << 16) | ce, s_scan, tot);
        int a_ = a_base + (pre >> 16), e_ = e_base + (pre & 0xffff);
        bool bad = false;
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const bool in = m0 + q < total;
            const bool gt = in && v[q].x > T, eq = in && v[q].x == T;
            const int o = gt ? a_ + min(e_, n_eq_need) : a_ + e_;
            const bool take = gt || (eq && e_ < n_eq_need);
            st_if(idx_out + (o < kE ? o : 0), (int32_t)v[q].y, take && o < kE);
            bad |= take && o >= kE;
            a_ += gt;
            e_ += eq;
        }
        if (bad) raise_flag(FLAG_INDEX_RANGE | 0x400u);
        a_base += tot >> 16;
        e_base += tot & 0xffff;
    }

    // the row's histogram and counter return to zero for the next launch
    for (int i = threadIdx.x; i < kNB1; i += kThreads) w.hist1[i] = 0;
    if (threadIdx.x == 0) w.bar[0] = 0;
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
    p.shift1 = p.key_bits - 10;
    p.nb2 = 1 << p.shift1;
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
    p.zero_bytes = off;
    off = align256(off + sizeof(int) * (size_t)p.ctas_per_row * rows);
    p.off_cand = off;
    off = align256(off + sizeof(uint2) * (size_t)p.ctas_per_row * p.chunk * rows);
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
