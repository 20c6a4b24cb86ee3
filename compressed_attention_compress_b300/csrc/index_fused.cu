// Lightning indexer + exact top-k, decode-shaped: one cooperative launch.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制, CSA step 2 (score every
// visible compressed entry against the query, keep the top-k).  Same result as
// the two-kernel path in index_topk.cu, in one launch whose CTAs are all resident
// (the launch is cooperative, so the waits below complete; each is still bounded
// and raises the device flag if it ever gives up):
//   phase 1  dp4a scores of this CTA's chunk, kept in shared memory as biased
//            keys u = s + DI*16256, and a 2048-bin histogram of u >> shift1.
//   phase 2  the histogram is added into the row's; the chunk writes its
//            candidates -- its keys in bins >= bc, bc the highest bin with at
//            least G of its keys at or above it (found by walking the bins down
//            from its largest key) -- as (key, index) in index order to its
//            region of the row's candidate list, with their count and bc, and
//            arrives at the row counter.  The other chunks then wait for the
//            verdict of the row's finisher (chunk row mod chunks).
//   phase 3  the finisher waits for every chunk, reads the row histogram, the
//            counts, the bc's and the first slots of every region in one round
//            trip, finds the bin b1 holding the k-th largest key and returns the
//            histogram to zero.  If no bc is above b1 the candidates hold every
//            key in bins >= b1: the verdict ("fast") lets the other chunks leave.
//            Else the verdict is b1 and every chunk rewrites its region with its
//            keys in bins >= b1 before the finisher goes on.  The regions, one
//            after another, list the candidates in index order.  The threshold
//            key T comes from the keys in b1; the keys above T and the first ties
//            at T are placed by one block scan of per-thread counts and written.
// G is twice a chunk's even share of the top-k plus 16, so with scores spread
// anything like evenly over the chunks the verdict is fast; scores that pile up
// in a few chunks take the rewrite, one more round trip.  The verdict is one word
// per row: a launch number that the finisher advances (the other chunks read it
// before they arrive) and the verdict, written with a plain store -- nothing is
// ordered after it.  A region holds its whole chunk, so heavily tied scores (many
// keys in b1) only make phase 3 longer (its general pass stages the list in
// shared memory and resolves T with a level-2 histogram).
#include "block_scan.cuh"
#include "common.cuh"
#include "internal.h"

namespace hsa {

namespace {

constexpr int kThreads = 256;
constexpr int kNB1 = 2048;
constexpr unsigned long long kSpinLimit = 1ull << 24;
constexpr int kStages = 3;  // 48 KiB of copies in flight per CTA
constexpr int kStageBytes = 16384;
constexpr int kMaxCpt = 4;  // chunks per thread in the last phase: at most 4 * kThreads chunks per row
// The row's verdict word: a launch number (upper bits) and the verdict (lower
// kVerdictBits): b1, or kVerdictFast.
constexpr int kVerdictBits = 12;
constexpr unsigned kVerdictMask = (1u << kVerdictBits) - 1u;
constexpr int kVerdictFast = (int)kVerdictMask;
constexpr int kB1Cap = 64;  // keys of b1 listed for the threshold (more: level-2 histogram)

__device__ __forceinline__ unsigned ld_relaxed(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(unsigned *p, unsigned v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
// Stores taken under a predicate without a branch around them.
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

// Thread 0 waits (bounded) until *ctr reaches `target`; the block learns whether
// it did.  Returns false (and raises the device flag) if the wait gave up.
__device__ __forceinline__ bool wait_count(const unsigned *ctr, unsigned target, int *s_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
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

// (one thread) Waits (bounded) until *p differs from `old`; false if it gave up.
__device__ __forceinline__ bool wait_change(const unsigned *p, unsigned old) {
    unsigned long long it = 0;
    while (ld_acquire(p) == old) {
        if (++it > kSpinLimit) {
            raise_flag(FLAG_INDEX_RANGE | 0x100u);
            return false;
        }
        __nanosleep(64);
    }
    return true;
}

// Staged candidate list: 16-entry groups with their entries rotated by the group
// number, so that threads reading 16 consecutive entries each hit distinct banks.
__device__ __forceinline__ int swz(int L) { return (L & ~15) | ((L + (L >> 4)) & 15); }

__device__ __forceinline__ int dot16(const int4 &x, const int4 &y) {
    int s = __dp4a(x.x, y.x, 0);
    s = __dp4a(x.y, y.y, s);
    s = __dp4a(x.z, y.z, s);
    return __dp4a(x.w, y.w, s);
}

struct Ws {
    unsigned *hist1;  // [rows][kNB1]
    unsigned *bar;    // [rows][4]: arrivals, verdict generation, verdict, arrivals of the rewrite
    int *rec;         // [rows][C] candidates per chunk
    int *cut;         // [rows][C] the lowest bin of each chunk's first candidates
    unsigned *verd;   // the row's verdict word (a 128-byte line of its own)
    uint2 *cand;      // [rows][C * chunk] (key, index) in bins >= b1, chunk c at c * chunk
};
__device__ __forceinline__ Ws carve(void *ws, const FusedIndexPlan &p, int r) {
    char *b = static_cast<char *>(ws);
    Ws w;
    w.hist1 = reinterpret_cast<unsigned *>(b + p.off_hist1) + (size_t)r * kNB1;
    w.bar = reinterpret_cast<unsigned *>(b + p.off_bar) + (size_t)r * 4;
    w.rec = reinterpret_cast<int *>(b + p.off_rec) + (size_t)r * p.ctas_per_row;
    w.cut = reinterpret_cast<int *>(b + p.off_cut) + (size_t)r * p.ctas_per_row;
    w.verd = reinterpret_cast<unsigned *>(b + p.off_verd) + (size_t)r * 32;
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

// This chunk's keys in bins >= bin, as (key, index) in index order, to the chunk's
// region of the row's candidate list; returns how many (to every thread).  Thread
// t takes keys [t * per, (t + 1) * per): one pass counts, a block scan gives its
// first slot, a second pass stores under a predicate (no branches per key).
__device__ __forceinline__ int write_candidates(const uint32_t *s_keys, int n, int per, int shift1, int bin,
                                                uint2 *cand, int64_t c0, int *s_scan) {
    const int my0 = threadIdx.x * per, my1 = min(n, my0 + per);
    int nc = 0;
    for (int e = my0; e < my1; ++e) nc += (int)(s_keys[e] >> shift1) >= bin;
    int tot;
    int o = block_exclusive_sum(nc, s_scan, tot);
    for (int e = my0; e < my1; ++e) {
        const uint32_t u = s_keys[e];
        const bool take = (int)(u >> shift1) >= bin;
        st_if(cand + o, make_uint2(u, (uint32_t)(c0 + e)), take);
        o += take;
    }
    return tot;
}

template <int LPE>
__global__ void __launch_bounds__(kThreads, 2) index_fused_kernel(IndexArgs a, FusedIndexPlan p, void *ws) {
    // a kernel launched after this one with programmatic stream serialization (the
    // decode attention) may be scheduled now; it waits for this grid's completion
    // before it reads anything
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t *s_keys = reinterpret_cast<uint32_t *>(smem);          // [chunk], kept over all phases
    unsigned *s_h = reinterpret_cast<unsigned *>(smem + (size_t)p.chunk * 4);  // [max(kNB1, nb2)]
    __shared__ int s_scan[33];
    __shared__ int s_misc[8];
    __shared__ uint32_t s_kmax;

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
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the verdict word before this chunk arrives (chunk 0 replaces it only after
    // every chunk has arrived)
    unsigned verd0 = 0;
    if (threadIdx.x == 0) {
        verd0 = ld_relaxed(w.verd);
        s_kmax = 0;
    }

    // ---------------------------------------------------------------- phase 1
    for (int i = threadIdx.x; i < kNB1; i += kThreads) s_h[i] = 0;
    uint32_t kmax = 0;  // this thread's largest key
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
            kmax = max(kmax, key);
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
    if (kmax) atomicMax(&s_kmax, kmax);
    __syncthreads();

    // ---------------------------------------------------------------- phase 2
    // Before anything global is known: this chunk's histogram goes into the row's,
    // and its candidates -- its keys in bins >= bc, bc the highest bin with at least
    // G of its keys at or above it, G a few times the chunk's even share of the
    // top-k -- go to its region of the row's candidate list, with their count and
    // bc.  Then the chunk arrives at the row counter.
    for (int i = threadIdx.x; i < kNB1; i += kThreads)
        if (s_h[i]) atomicAdd(&w.hist1[i], s_h[i]);
    if (warp == 0) {
        // walk the bins down from the chunk's largest key, 32 at a time
        const int G = min(n, 2 * ((kE + nch - 1) / nch) + 16);
        int cum = 0, bc = 0;
        for (int b0 = (int)(s_kmax >> p.shift1); b0 >= 0; b0 -= 32) {
            const int bin = b0 - lane;
            const int inc = warp_inclusive_sum(bin >= 0 ? (int)s_h[bin] : 0);
            const unsigned hit = __ballot_sync(0xffffffffu, cum + inc >= G);
            if (hit) {
                bc = b0 - (__ffs(hit) - 1);
                break;
            }
            cum += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) s_misc[0] = bc;
    }
    __syncthreads();
    const int bc = s_misc[0];
    const int per_key = (p.chunk + kThreads - 1) / kThreads;  // keys per thread in write_candidates
    {
        const int tot = write_candidates(s_keys, n, per_key, p.shift1, bc, w.cand + c0, c0, s_scan);
        if (threadIdx.x == 0) {
            w.rec[c] = tot;
            w.cut[c] = bc;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(&w.bar[0], 1u);
    }

    // the row's finisher: chunk row % nch, so that the rows' finishers are far apart
    // in launch order (and so on different SMs)
    const int fin = row % nch;
    if (c != fin) {
        // Wait for the finisher's verdict.  Fast: every chunk's candidates hold all its
        // keys in bins >= b1, nothing more to do.  Otherwise the verdict is b1 and
        // every chunk rewrites its candidates as its keys in bins >= b1.
        if (threadIdx.x == 0) {
            int v = -1;
            unsigned long long it = 0;
            for (;;) {
                const unsigned now = ld_relaxed(w.verd);
                if ((now >> kVerdictBits) != (verd0 >> kVerdictBits)) {
                    v = (int)(now & kVerdictMask);
                    break;
                }
                if (++it > kSpinLimit) {
                    raise_flag(FLAG_INDEX_RANGE | 0x100u);
                    break;
                }
                __nanosleep(128);
            }
            s_misc[7] = v;
        }
        __syncthreads();
        const int v = s_misc[7];
        if (v < 0 || v == kVerdictFast) return;
        const int tot = write_candidates(s_keys, n, per_key, p.shift1, v, w.cand + c0, c0, s_scan);
        if (threadIdx.x == 0) w.rec[c] = tot;
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(&w.bar[3], 1u);
        }
        return;
    }

    // ---------------------------------------------------------------- phase 3
    // (the finisher, once every chunk has arrived) One round trip to L2 brings every
    // chunk's count and bc, the row histogram and the first `spec` slots of every
    // chunk's region.  The histogram gives b1, the bin of the k-th largest key; if
    // no bc is above b1 the candidates hold every key in bins >= b1 (fast
    // verdict), else every chunk rewrites its region with exactly those keys and
    // the finisher waits for them.  The regions, one after another, list the candidates
    // in index order.  When every region fits its first `spec` slots the selection
    // runs on the slots held in registers: slot order is index order, the
    // threshold key T comes from the keys in b1, and one scan of per-warp counts
    // places the keys above T and the first ties at T.  Longer regions take the
    // general pass: the list is staged in shared memory while a level-2 histogram
    // of the low bits of the keys in b1 gives T, and an ordered pass writes the
    // winners.
    if (!wait_count(&w.bar[0], (unsigned)nch, &s_misc[7])) return;
    constexpr int kSpecPer = 20;  // candidate slots per thread: slot t * kSpecPer + q (even, loaded in pairs)
    static_assert(8192 + kThreads * kSpecPer * 8 <= kStages * kStageBytes, "slot staging outside the stage region");
    int lg_spec = 6;
    while (lg_spec > 1 && (nch << lg_spec) > kThreads * kSpecPer) --lg_spec;
    const int spec = (nch << lg_spec) <= kThreads * kSpecPer ? 1 << lg_spec : 0;
    const int cpt = (nch + kThreads - 1) / kThreads;  // chunks per thread (<= kMaxCpt)
    const int i0 = threadIdx.x * cpt;
    uint2 sv[kSpecPer];
    int rv[kMaxCpt];
    auto load_counts = [&]() {
#pragma unroll
        for (int q = 0; q < kMaxCpt; ++q) rv[q] = q < cpt && i0 + q < nch ? __ldcg(&w.rec[i0 + q]) : 0;
    };
    // The slots travel L2 -> shared memory as coalesced 16-byte copies (slot pairs
    // 2j, 2j + 1 with j = q * kThreads + t; slots of chunks >= nch are zero-filled)
    // and are then read back by each thread as its kSpecPer consecutive slots.
    uint2 *s_slots = reinterpret_cast<uint2 *>(smem + p.off_stage_smem + 8192);  // [kThreads * kSpecPer]
    auto load_slots = [&]() {
#pragma unroll
        for (int q = 0; q < kSpecPer / 2; ++q) {
            const int sp = 2 * (q * kThreads + threadIdx.x);
            const int cc = spec ? sp >> lg_spec : nch;
            const uint2 *src = cc < nch ? w.cand + (int64_t)cc * p.chunk + (sp & (spec - 1)) : w.cand;
            cp_async_16(smem_u32(s_slots + sp), src, cc < nch ? 16 : 0);
        }
        cp_async_commit();
    };
    auto land_slots = [&]() {
        cp_async_wait<0>();
        __syncthreads();
        const uint4 *src = reinterpret_cast<const uint4 *>(s_slots + threadIdx.x * kSpecPer);
#pragma unroll
        for (int q = 0; q < kSpecPer; q += 2) {
            const uint4 x = src[q / 2];
            sv[q] = make_uint2(x.x, x.y);
            sv[q + 1] = make_uint2(x.z, x.w);
        }
    };
    // every load of this round trip is issued before any is used
    constexpr int PB = kNB1 / kThreads;  // bins per thread, descending
    const int top = kNB1 - 1 - threadIdx.x * PB;
    int hv[PB];
#pragma unroll
    for (int q = 0; q < PB; ++q) hv[q] = (int)__ldcg(&w.hist1[top - q]);
    load_counts();
    int cut[kMaxCpt];  // the bc of this thread's chunks
#pragma unroll
    for (int q = 0; q < kMaxCpt; ++q) cut[q] = q < cpt && i0 + q < nch ? __ldcg(&w.cut[i0 + q]) : 0;
    load_slots();
    if (threadIdx.x == 0) {
        w.bar[0] = 0;  // every chunk has arrived: the counter is free for the next launch
        s_misc[0] = s_misc[1] = s_misc[2] = s_misc[3] = s_misc[4] = s_misc[5] = 0;
    }
    {
        int local = 0;
#pragma unroll
        for (int q = 0; q < PB; ++q) local += hv[q];
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
        // the row histogram returns to zero for the next launch (its loads are done)
#pragma unroll
        for (int q = 0; q < PB; ++q)
            if (hv[q]) w.hist1[top - q] = 0;
        __syncthreads();
    }
    const int b1 = s_misc[0], count_above = s_misc[1], n_in = s_misc[2];
    int cv = 0;  // the highest bc of this thread's chunks
#pragma unroll
    for (int q = 0; q < kMaxCpt; ++q) cv = max(cv, cut[q]);
    const bool fast = !__syncthreads_or(cv > b1);
    if (fast) land_slots();
    if (threadIdx.x == 0)
        st_relaxed(w.verd, (((verd0 >> kVerdictBits) + 1u) << kVerdictBits) | (fast ? (unsigned)kVerdictFast : (unsigned)b1));
    if (!fast) {
        const int tot = write_candidates(s_keys, n, per_key, p.shift1, b1, w.cand + c0, c0, s_scan);
        if (threadIdx.x == 0) w.rec[c] = tot;
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(&w.bar[3], 1u);
        }
        if (!wait_count(&w.bar[3], (unsigned)nch, &s_misc[7])) return;
        if (threadIdx.x == 0) w.bar[3] = 0;
        cp_async_wait<0>();  // the first copies have landed before the buffer is reused
        __syncthreads();
        load_counts();
        load_slots();
        land_slots();
    }
    const int need = kE - count_above;  // >= 1
    int *s_off = reinterpret_cast<int *>(smem + p.off_stage_smem);  // [nch + 1]
    int rmax = 0;
#pragma unroll
    for (int q = 0; q < kMaxCpt; ++q) rmax = max(rmax, rv[q]);
    if (spec > 0 && !__syncthreads_or(rmax > spec)) {
        // ---- every region fits its first spec slots: selection on the registers
        uint32_t *s_b1 = reinterpret_cast<uint32_t *>(s_off + ((nch + 4) & ~3));  // [kB1Cap] keys in b1
        unsigned *s_h2 = s_h;
#pragma unroll
        for (int q = 0; q < kMaxCpt; ++q)
            if (q < cpt && i0 + q < nch) s_off[i0 + q] = rv[q];  // here: the count of each region
        if (threadIdx.x == 0) s_off[nch] = 0;
        if (n_in > kB1Cap)
            for (int i = threadIdx.x; i < p.nb2; i += kThreads) s_h2[i] = 0;
        __syncthreads();
        unsigned vbits = 0;  // bit q: slot q of this thread holds a candidate
#pragma unroll
        for (int q = 0; q < kSpecPer; ++q) {
            const int sp = threadIdx.x * kSpecPer + q;
            vbits |= (unsigned)((sp & (spec - 1)) < s_off[min(sp >> lg_spec, nch)]) << q;
        }
        // the keys of b1: listed (few) or counted by their low bits (many)
#pragma unroll
        for (int q = 0; q < kSpecPer; ++q) {
            if (((vbits >> q) & 1u) && (int)(sv[q].x >> p.shift1) == b1) {
                if (n_in <= kB1Cap) {
                    const int j = atomicAdd(&s_misc[3], 1);
                    if (j < kB1Cap) s_b1[j] = sv[q].x;
                } else {
                    atomicAdd(&s_misc[3], 1);
                    atomicAdd(&s_h2[sv[q].x & ((uint32_t)p.nb2 - 1u)], 1u);
                }
            }
        }
        __syncthreads();
        if (threadIdx.x == 0 && s_misc[3] != n_in) raise_flag(FLAG_INDEX_RANGE | 0x400u);
        uint32_t T;
        int n_gt_in;  // keys of b1 above T
        if (n_in <= kB1Cap) {
            // T: the key of b1 with fewer than `need` keys above it and at least `need`
            // at or above it (every thread holding that key writes the same values)
            if (threadIdx.x < n_in) {
                const uint32_t k = s_b1[threadIdx.x];
                int gt = 0, ge = 0;
                for (int j = 0; j < n_in; ++j) {
                    const uint32_t u = s_b1[j];
                    gt += u > k;
                    ge += u >= k;
                }
                if (gt < need && need <= ge) {
                    s_misc[4] = (int)k;
                    s_misc[5] = gt;
                }
            }
            __syncthreads();
            T = (uint32_t)s_misc[4];
            n_gt_in = s_misc[5];
        } else {
            find_threshold(s_h2, p.nb2, need, s_scan, &s_misc[4]);
            T = ((uint32_t)b1 << p.shift1) | (uint32_t)s_misc[4];
            n_gt_in = s_misc[5];
        }
        const int n_eq_need = need - n_gt_in;  // ties at T to take, the first in index order
        // slot order is index order: count the keys above T and the ties, one block
        // scan of the packed counts (above T in the high half) places every winner
        int cg = 0, ce = 0;
#pragma unroll
        for (int q = 0; q < kSpecPer; ++q) {
            const bool v = (vbits >> q) & 1u;
            cg += v && sv[q].x > T;
            ce += v && sv[q].x == T;
        }
        int all;
        const int pre = block_exclusive_sum((cg << 16) | ce, s_scan, all);
        if (threadIdx.x == 0 && (all >> 16) + min(all & 0xffff, n_eq_need) != kE) raise_flag(FLAG_INDEX_RANGE | 0x400u);
        int a_ = pre >> 16, e_ = pre & 0xffff;
        bool bad = false;
#pragma unroll
        for (int q = 0; q < kSpecPer; ++q) {
            const bool v = (vbits >> q) & 1u;
            const bool gt = v && sv[q].x > T, eq = v && sv[q].x == T;
            const int o = gt ? a_ + min(e_, n_eq_need) : a_ + e_;
            const bool take = gt || (eq && e_ < n_eq_need);
            st_if(idx_out + (o < kE ? o : 0), (int32_t)sv[q].y, take && o < kE);
            bad |= take && o >= kE;
            a_ += gt;
            e_ += eq;
        }
        if (bad) raise_flag(FLAG_INDEX_RANGE | 0x400u);
        return;
    }

    // ---- general pass: regions longer than spec slots
    int *s_roff = s_off + (nch + 1);  // [nch + 1] offsets past the first spec slots
    const int l_off = (2 * (nch + 1) * 4 + 15) & ~15;
    uint2 *s_l = reinterpret_cast<uint2 *>(smem + p.off_stage_smem + l_off);
    const int l_cap = ((kStages * kStageBytes - l_off) / 8) & ~15;
    unsigned *s_h2 = s_h;
    const uint32_t mask2 = (uint32_t)p.nb2 - 1u;
    for (int i = threadIdx.x; i < p.nb2; i += kThreads) s_h2[i] = 0;
    if (threadIdx.x == 0) s_misc[3] = s_misc[4] = s_misc[5] = 0;
    {
        int loc = 0, rest = 0;
#pragma unroll
        for (int q = 0; q < kMaxCpt; ++q) {
            loc += rv[q];
            rest += rv[q] > spec ? rv[q] - spec : 0;
        }
        int tot, rtot;
        int o = block_exclusive_sum(loc, s_scan, tot);
        int ro = block_exclusive_sum(rest, s_scan, rtot);
#pragma unroll
        for (int q = 0; q < kMaxCpt; ++q)
            if (q < cpt && i0 + q < nch) {
                s_off[i0 + q] = o;
                s_roff[i0 + q] = ro;
                o += rv[q];
                ro += rv[q] > spec ? rv[q] - spec : 0;
            }
        if (threadIdx.x == 0) {
            s_off[nch] = tot;
            s_roff[nch] = rtot;
        }
        __syncthreads();
    }
    const int total = s_off[nch], n_rest = s_roff[nch];
    const bool staged = total <= l_cap;
    int n_hi = 0;  // candidates in bins >= b1
    auto take_in = [&](const uint2 &v, int L) {
        if (staged) s_l[swz(L)] = v;
        const int bin = (int)(v.x >> p.shift1);
        if (bin == b1) atomicAdd(&s_h2[v.x & mask2], 1u);
        n_hi += bin >= b1;
    };
#pragma unroll
    for (int q = 0; q < kSpecPer; ++q) {
        const int sp = threadIdx.x * kSpecPer + q;
        const int cc = spec ? sp >> lg_spec : nch;
        if (cc < nch) {
            const int i = sp & (spec - 1);
            if (i < s_off[cc + 1] - s_off[cc]) take_in(sv[q], s_off[cc] + i);
        }
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
    {
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
    }
    if (n_hi) atomicAdd(&s_misc[3], n_hi);
    __syncthreads();
    if (threadIdx.x == 0 && s_misc[3] != count_above + n_in) raise_flag(FLAG_INDEX_RANGE | 0x400u);
    find_threshold(s_h2, p.nb2, need, s_scan, &s_misc[4]);
    const uint32_t T = ((uint32_t)b1 << p.shift1) | (uint32_t)s_misc[4];
    const int n_eq_need = need - s_misc[5];
    const bool all_eq = n_eq_need == (int)s_h2[s_misc[4]];  // every key equal to T is taken
    int eq_base = 0, pos_base = 0;
    constexpr int PER = 8;
    for (int t0 = 0; t0 < total; t0 += kThreads * PER) {
        const int m0 = t0 + threadIdx.x * PER;
        uint2 v[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int L = m0 + q;
            if (L >= total) v[q] = make_uint2(0u, 0u);
            else if (staged) v[q] = s_l[swz(L)];
            else {
                const int cc = find_chunk(s_off, L);
                v[q] = __ldcg(w.cand + (int64_t)cc * p.chunk + (L - s_off[cc]));
            }
        }
        bool take[PER];
        int nsel = 0;
        if (all_eq) {
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                take[q] = m0 + q < total && v[q].x >= T;
                nsel += take[q];
            }
        } else {
            int eq = 0;
#pragma unroll
            for (int q = 0; q < PER; ++q) eq += m0 + q < total && v[q].x == T;
            int tot_eq;
            int er = eq_base + block_exclusive_sum(eq, s_scan, tot_eq);
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                take[q] = m0 + q < total && v[q].x > T;
                if (m0 + q < total && v[q].x == T) {
                    take[q] = er < n_eq_need;
                    ++er;
                }
                nsel += take[q];
            }
            eq_base += tot_eq;
        }
        int tot_sel;
        int o = pos_base + block_exclusive_sum(nsel, s_scan, tot_sel);
#pragma unroll
        for (int q = 0; q < PER; ++q)
            if (take[q]) {
                if (o < kE) idx_out[o] = (int32_t)v[q].y;
                else raise_flag(FLAG_INDEX_RANGE | 0x400u);
                ++o;
            }
        pos_base += tot_sel;
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
    // Chunks are multiples of 64 entries; pick the smallest chunk whose launch
    // (ceil(E/chunk) CTAs per row) is resident all at once, so every SM streams
    // an equal share.
    for (int chunk = 256; chunk <= 16384; chunk += 64) {
        const int64_t C = (E_cap + chunk - 1) / chunk;
        if (C > (int64_t)kMaxCpt * kThreads) continue;
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
    p.off_verd = off;
    off = align256(off + sizeof(unsigned) * 32 * (size_t)rows);
    p.off_rec = off;
    p.zero_bytes = off;
    off = align256(off + sizeof(int) * (size_t)p.ctas_per_row * rows);
    p.off_cut = off;
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
