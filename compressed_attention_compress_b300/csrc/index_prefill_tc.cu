// Lightning indexer + exact top-k for many query rows (prefill), scored on the
// 5th-generation tensor cores.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制, CSA step 2: every query token
// scores every visible compressed entry with a light indexer and keeps the top-k.
// Scores are exact int32 dot products of int8 vectors.  int8 values are exact in
// bf16, their products are at most 2^14 and, for DI <= 128, every partial sum is
// an integer below 2^22, so bf16 tcgen05 MMAs with fp32 accumulation give the
// exact integer scores.
//
//   convert   int8 -> bf16 copies of the query and entry vectors (workspace).
//   sample    per 128-query tile, score every 16th 128-entry tile, keep a
//             per-row 128-bin histogram over the row's score bound and set the
//             row's candidate threshold tau so that about 1.6*k entries of the
//             whole row are expected at or above it.
//   collect   per (128-query tile, entry segment), score every entry; a row's
//             thread appends (score, index) of the entries at or above tau, in
//             index order, to the row's list for that segment.
//   select    per row: exact top-k over the concatenated lists (two radix
//             levels, ties by index), written in ascending index order.  A row
//             whose lists hold fewer than k candidates or overflowed falls back
//             to an exact three-pass dp4a scan of its keys (rare: only for
//             heavily tied or adversarial scores).
// The result is the same bit for bit as the decode-shaped kernels give.
#include <math.h>

#include <cudaTypedefs.h>

#include "block_scan.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace hsa {

namespace {

constexpr int kRows = 128;    // query rows per tile
constexpr int kN = 128;       // entries per score tile
constexpr int kSampleEvery = 16;
constexpr int kBins = 128;
constexpr int kThreads = 192;  // 4 epilogue warps, MMA warp, TMA warp
constexpr unsigned long long kWaitLimit = 1ull << 24;

struct PfArgs {
    int B, T, DI, m, topk;
    int64_t E_cap;
    const int64_t *q_pos0;
    const int8_t *q8;      // original int8 queries (for bounds / fallback)
    int64_t q_sb, q_st;
    const int8_t *k8;      // original int8 entry vectors (fallback)
    int64_t k_sb, k_se;
    float *tau;            // [B*T]
    int2 *lists;           // [B*T][S][cap_seg]
    int *counts;           // [B*T][S]
    int n_seg, cap_seg, seg_tiles;
    int32_t *idx_out, *cnt_out;
};

__device__ __forceinline__ bool wait_bar(uint64_t *bar, unsigned parity, volatile int *abort) {
    for (unsigned long long i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    raise_flag(FLAG_INDEX_RANGE | 0x800u);
    *abort = 1;
    return false;
}
__device__ __forceinline__ void arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------------ convert
__global__ void __launch_bounds__(256) int8_to_bf16_kernel(const int8_t *src, int64_t rows, int DI, int64_t sb,
                                                          int64_t s_row, int64_t rows_per_b,
                                                          __nv_bfloat16 *dst) {
    // dst is dense [rows, DI]; src row r = b*rows_per_b + i at src + b*sb + i*s_row
    const int per = DI / 16;
    const int64_t total = rows * per;
    for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < total; w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = w / per;
        const int c = (int)(w - r * per);
        const int64_t b = r / rows_per_b, i = r - b * rows_per_b;
        const int4 v = *reinterpret_cast<const int4 *>(src + b * sb + i * s_row + c * 16);
        const int8_t *x = reinterpret_cast<const int8_t *>(&v);
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = pack_bf16x2((float)x[2 * e], (float)x[2 * e + 1]);
        uint4 *d = reinterpret_cast<uint4 *>(dst + r * DI + c * 16);
        d[0] = make_uint4(o[0], o[1], o[2], o[3]);
        d[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// ------------------------------------------------------- score tile engine
// Shared by the sample and collect kernels: a TMA warp streams entry tiles,
// one thread issues S = Q K^T (M = 128 queries, N = 128 entries) into one of
// two TMEM buffers, and four epilogue warps consume S (one query row per thread).
template <int DI>
struct Layout {
    static constexpr int kKB = DI / 64;                 // 128-byte K blocks
    static constexpr int kQ = kRows * 128 * kKB;        // Q tile bytes
    static constexpr int kK = kN * 128 * kKB;           // entry tile bytes
    static constexpr int kStages = 4;
    static constexpr int kSmemTiles = kQ + kStages * kK;
};

struct __align__(8) Bars {
    uint64_t q_full, k_full[4], k_empty[4], s_full[2], s_free[2], fin;
};

template <int DI, bool SAMPLE>
__global__ void __launch_bounds__(kThreads, SAMPLE ? 1 : 2)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, PfArgs a) {
    using Lay = Layout<DI>;
    extern __shared__ __align__(16) unsigned char smem_raw[];  // rounded up to 1024 at run time
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *sQ = smem;
    unsigned char *sK = smem + Lay::kQ;
    uint32_t *sHist = reinterpret_cast<uint32_t *>(smem + Lay::kSmemTiles);  // [kBins][kRows] (sample only)
    __shared__ Bars bars;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    // work item: query tile of one sequence, entry segment
    const int tiles_per_b = (a.T + kRows - 1) / kRows;
    const int item = blockIdx.x;
    const int seg = SAMPLE ? 0 : item % a.n_seg;
    const int qtile = SAMPLE ? item : item / a.n_seg;
    const int b = qtile / tiles_per_b;
    const int t0 = (qtile - b * tiles_per_b) * kRows;
    const int64_t p_last = a.q_pos0[b] + (t0 + kRows - 1 < a.T ? t0 + kRows - 1 : a.T - 1);
    int64_t E_last = num_entries(p_last, a.m);
    if (E_last > a.E_cap) E_last = a.E_cap;
    const int n_tiles_row = (int)((E_last + kN - 1) / kN);
    // tiles this CTA scores: every kSampleEvery-th (sample) or its segment's range
    int tile_begin, tile_step, n_my;
    if (SAMPLE) {
        tile_begin = 0;
        tile_step = kSampleEvery;
        n_my = (n_tiles_row + kSampleEvery - 1) / kSampleEvery;
    } else {
        tile_begin = seg * a.seg_tiles;
        tile_step = 1;
        const int end = min(n_tiles_row, tile_begin + a.seg_tiles);
        n_my = end > tile_begin ? end - tile_begin : 0;
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bars.q_full, 1);
        for (int i = 0; i < Lay::kStages; ++i) {
            mbar_init(&bars.k_full[i], 1);
            mbar_init(&bars.k_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.s_free[i], kRows);
        }
        mbar_init(&bars.fin, 1);
        fence_mbar_init();
        s_abort = 0;
    }
    if (SAMPLE)
        for (int i = threadIdx.x; i < kBins * kRows; i += kThreads) sHist[i] = 0;
    if (warp == 0) tc::tmem_alloc(&s_tmem, 256);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 5) {
        if (lane == 0 && n_my > 0) {
            bool ok = true;
            mbar_expect_tx(&bars.q_full, Lay::kQ);
#pragma unroll
            for (int kb = 0; kb < Lay::kKB; ++kb)
                tc::tma_load_2d(sQ + kb * kRows * 128, &tm_q, kb * 64, b * a.T + t0, &bars.q_full);
            int last[Lay::kStages];
            for (int i = 0; i < Lay::kStages; ++i) last[i] = -1;
            for (int it = 0; it < n_my && ok; ++it) {
                const int st = it % Lay::kStages;
                if (it >= Lay::kStages) ok = wait_bar(&bars.k_empty[st], (unsigned)(((it / Lay::kStages) - 1) & 1), &s_abort);
                if (!ok) break;
                const int tile = tile_begin + it * tile_step;
                mbar_expect_tx(&bars.k_full[st], Lay::kK);
                last[st] = it / Lay::kStages;
#pragma unroll
                for (int kb = 0; kb < Lay::kKB; ++kb)
                    tc::tma_load_3d(sK + st * Lay::kK + kb * kN * 128, &tm_k, kb * 64, tile * kN, b, &bars.k_full[st]);
            }
            if (!ok) s_abort = 1;
            volatile int never = 0;
            wait_bar(&bars.q_full, 0u, &never);
            for (int st = 0; st < Lay::kStages; ++st)
                if (last[st] >= 0) wait_bar(&bars.k_full[st], (unsigned)(last[st] & 1), &never);
        }
    } else if (warp == 4) {
        if (lane == 0 && n_my > 0) {
            constexpr uint32_t idS = tc::idesc_bf16(kRows, kN, false, false);
            bool ok = wait_bar(&bars.q_full, 0u, &s_abort);
            tc::fence_after();
            const uint32_t aQ = smem_u32(sQ);
            for (int it = 0; it < n_my && ok; ++it) {
                const int st = it % Lay::kStages, sb = it & 1;
                ok = wait_bar(&bars.k_full[st], (unsigned)((it / Lay::kStages) & 1), &s_abort);
                if (ok && it >= 2) ok = wait_bar(&bars.s_free[sb], (unsigned)(((it >> 1) - 1) & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                const uint32_t aK = smem_u32(sK + st * Lay::kK);
#pragma unroll
                for (int kk = 0; kk < DI / 16; ++kk) {
                    const uint64_t da = tc::desc_sw128(aQ + (kk >> 2) * kRows * 128 + (kk & 3) * 32, 16, 1024);
                    const uint64_t db = tc::desc_sw128(aK + (kk >> 2) * kN * 128 + (kk & 3) * 32, 16, 1024);
                    tc::mma_bf16(tmem + sb * kN, da, db, idS, kk > 0 ? 1u : 0u);
                }
                tc::commit(&bars.s_full[sb]);
                tc::commit(&bars.k_empty[st]);
            }
            if (!ok) s_abort = 1;
            tc::commit(&bars.fin);
            volatile int never = 0;
            wait_bar(&bars.fin, 0u, &never);
        }
    } else {
        // epilogue: thread r owns query row t0 + r of sequence b
        const int r = threadIdx.x;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const int t = t0 + r;
        const bool live = t < a.T;
        const int64_t row = (int64_t)b * a.T + (live ? t : 0);
        const int64_t p = a.q_pos0[b] + t;
        int64_t E = num_entries(p, a.m);
        if (E > a.E_cap) E = a.E_cap;
        if (!live) E = 0;
        // per-row bound on |score| for the sample histogram
        float lo = 0.f, inv_w = 0.f;
        float tau = 0.f;
        int cnt = 0;
        int2 *my_list = nullptr;
        if (SAMPLE) {
            int sabs = 0;
            if (live)
                for (int c = 0; c < a.DI; ++c) {
                    const int v = a.q8[b * a.q_sb + (int64_t)t * a.q_st + c];
                    sabs += v < 0 ? -v : v;
                }
            const float R = 128.f * (float)sabs + 1.f;
            lo = -R;
            inv_w = (float)kBins / (2.f * R);
        } else {
            tau = live ? a.tau[row] : INFINITY;
            my_list = a.lists + (row * a.n_seg + seg) * (int64_t)a.cap_seg;
        }
        bool ok = true;
        for (int it = 0; it < n_my && ok; ++it) {
            const int sb = it & 1;
            ok = wait_bar(&bars.s_full[sb], (unsigned)((it >> 1) & 1), &s_abort);
            if (!ok) break;
            tc::fence_after();
            const int64_t j0 = (int64_t)(tile_begin + it * tile_step) * kN;
#pragma unroll
            for (int c = 0; c < kN / 32; ++c) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + sb * kN + lane_off + c * 32, v);
                tc::tmem_wait_ld();
                if (SAMPLE) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int64_t j = j0 + c * 32 + e;
                        if (j < E) {
                            int bin = (int)((__uint_as_float(v[e]) - lo) * inv_w);
                            bin = bin < 0 ? 0 : (bin >= kBins ? kBins - 1 : bin);
                            sHist[bin * kRows + r] += 1u;
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float sc = __uint_as_float(v[e]);
                        const int64_t j = j0 + c * 32 + e;
                        if (sc >= tau && j < E) {
                            if (cnt < a.cap_seg) my_list[cnt] = make_int2((int)sc, (int)j);
                            ++cnt;
                        }
                    }
                }
            }
            tc::fence_before();
            arrive(&bars.s_free[sb]);
        }
        if (!ok) s_abort = 1;
        if (live) {
            if (SAMPLE) {
                // threshold: expect ~1.6*k of the row's E entries at or above it
                const int kE = (int)(E < a.topk ? E : a.topk);
                int n_samp = 0;
                for (int i = 0; i < kBins; ++i) n_samp += (int)sHist[i * kRows + r];
                float th = -INFINITY;
                if (E > 4 * kE && n_samp > 0) {
                    const float want = 1.6f * (float)kE * (float)n_samp / (float)E;
                    float cum = 0.f;
                    for (int i = kBins - 1; i >= 0; --i) {
                        cum += (float)sHist[i * kRows + r];
                        if (cum >= want) {
                            th = floorf(lo + (float)i / inv_w);
                            break;
                        }
                    }
                }
                a.tau[row] = th;
            } else {
                a.counts[row * a.n_seg + seg] = cnt;
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// --------------------------------------------------------------- selection
constexpr int kSelThreads = 256;
constexpr int kSelCap = 8192;  // candidates held in shared memory

__device__ __forceinline__ int dot16(const int4 &x, const int4 &y) {
    int s = __dp4a(x.x, y.x, 0);
    s = __dp4a(x.y, y.y, s);
    s = __dp4a(x.z, y.z, s);
    return __dp4a(x.w, y.w, s);
}

// Exact selection over candidates held in shared memory in ascending index order.
// Keys are biased scores (>= 0).  Writes min(kE, n) indices (n >= kE required).
__device__ void select_sorted(const uint32_t *s_u, const int32_t *s_j, int n, int kE, int key_bits, unsigned *hist,
                              int *s_scan, int *s_misc, int32_t *out) {
    const int shift = key_bits - 11;
    // level 1: 2048 bins of the top bits
    for (int i = threadIdx.x; i < 2048; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kSelThreads) atomicAdd(&hist[s_u[i] >> shift], 1u);
    __syncthreads();
    {
        const int per = 2048 / kSelThreads, top = 2047 - threadIdx.x * per;
        int local = 0;
        for (int q = 0; q < per; ++q) local += (int)hist[top - q];
        int tot;
        const int before = block_exclusive_sum(local, s_scan, tot);
        if (before < kE && before + local >= kE) {
            int cum = before;
            for (int q = 0; q < per; ++q) {
                const int hv = (int)hist[top - q];
                if (cum + hv >= kE) {
                    s_misc[0] = top - q;
                    s_misc[1] = cum;
                    break;
                }
                cum += hv;
            }
        }
        __syncthreads();
    }
    const uint32_t b1 = (uint32_t)s_misc[0];
    const int above = s_misc[1];
    const int need = kE - above;
    // level 2: low bits inside b1 (at most 2^11 bins for DI <= 128)
    const int nb2 = 1 << shift;
    for (int i = threadIdx.x; i < nb2; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kSelThreads)
        if ((s_u[i] >> shift) == b1) atomicAdd(&hist[s_u[i] & (uint32_t)(nb2 - 1)], 1u);
    __syncthreads();
    {
        const int per = nb2 / kSelThreads, top = nb2 - 1 - threadIdx.x * per;
        int local = 0;
        for (int q = 0; q < per; ++q) local += (int)hist[top - q];
        int tot;
        const int before = block_exclusive_sum(local, s_scan, tot);
        if (before < need && before + local >= need) {
            int cum = before;
            for (int q = 0; q < per; ++q) {
                const int hv = (int)hist[top - q];
                if (cum + hv >= need) {
                    s_misc[2] = top - q;
                    s_misc[3] = cum;
                    break;
                }
                cum += hv;
            }
        }
        __syncthreads();
    }
    const uint32_t T = (b1 << shift) | (uint32_t)s_misc[2];
    const int n_eq_need = need - s_misc[3];
    // ordered compaction (candidates are in index order)
    const int per = (n + kSelThreads - 1) / kSelThreads, my0 = threadIdx.x * per;
    int eq = 0;
    for (int q = 0; q < per; ++q) {
        const int i = my0 + q;
        if (i < n && s_u[i] == T) ++eq;
    }
    int tot;
    int er = block_exclusive_sum(eq, s_scan, tot);
    int nsel = 0;
    {
        int e2 = er;
        for (int q = 0; q < per; ++q) {
            const int i = my0 + q;
            if (i >= n) break;
            if (s_u[i] > T) ++nsel;
            else if (s_u[i] == T) { nsel += e2 < n_eq_need; ++e2; }
        }
    }
    int o = block_exclusive_sum(nsel, s_scan, tot);
    for (int q = 0; q < per; ++q) {
        const int i = my0 + q;
        if (i >= n) break;
        bool take = s_u[i] > T;
        if (s_u[i] == T) { take = er < n_eq_need; ++er; }
        if (take) out[o++] = s_j[i];
    }
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(PfArgs a, int key_bits) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t *s_u = reinterpret_cast<uint32_t *>(smem);         // [kSelCap]
    int32_t *s_j = reinterpret_cast<int32_t *>(s_u + kSelCap);  // [kSelCap]
    unsigned *hist = reinterpret_cast<unsigned *>(s_j + kSelCap);  // [2048]
    __shared__ int s_scan[33];
    __shared__ int s_misc[8];
    __shared__ int s_off[16];

    const int64_t row = blockIdx.x;
    const int b = (int)(row / a.T), t = (int)(row - (int64_t)b * a.T);
    const int64_t p = a.q_pos0[b] + t;
    int64_t E = num_entries(p, a.m);
    if (E > a.E_cap) {
        if (threadIdx.x == 0) raise_flag(FLAG_INDEX_RANGE);
        E = a.E_cap;
    }
    const int kE = (int)(E < a.topk ? E : a.topk);
    int32_t *out = a.idx_out + row * a.topk;
    for (int i = kE + threadIdx.x; i < a.topk; i += kSelThreads) out[i] = -1;
    if (threadIdx.x == 0) a.cnt_out[row] = kE;
    if (kE == 0) return;
    const int bias = a.DI * 16256;

    // gather the segment lists (each in index order, segments in order)
    if (threadIdx.x == 0) {
        int off = 0;
        bool fits = true;
        for (int s = 0; s < a.n_seg; ++s) {
            const int c = a.counts[row * a.n_seg + s];
            if (c > a.cap_seg) fits = false;
            s_off[s] = off;
            off += c;
        }
        s_misc[4] = off;
        s_misc[5] = fits && off <= kSelCap && off >= kE;
    }
    __syncthreads();
    const int n = s_misc[4];
    if (s_misc[5]) {
        for (int s = 0; s < a.n_seg; ++s) {
            const int c = a.counts[row * a.n_seg + s];
            const int2 *lst = a.lists + (row * a.n_seg + s) * (int64_t)a.cap_seg;
            for (int i = threadIdx.x; i < c; i += kSelThreads) {
                const int2 v = lst[i];
                s_u[s_off[s] + i] = (uint32_t)(v.x + bias);
                s_j[s_off[s] + i] = v.y;
            }
        }
        __syncthreads();
        select_sorted(s_u, s_j, n, kE, key_bits, hist, s_scan, s_misc, out);
        return;
    }
    // ---- exact fallback: three dp4a passes over the row's keys
    const int lpe = a.DI / 16;
    const int lane_e = threadIdx.x % lpe, grp = threadIdx.x / lpe, groups = kSelThreads / lpe;
    const int4 qv = *reinterpret_cast<const int4 *>(a.q8 + b * a.q_sb + (int64_t)t * a.q_st + lane_e * 16);
    const char *kbase = reinterpret_cast<const char *>(a.k8 + b * a.k_sb) + lane_e * 16;
    const int shift = key_bits - 11;
    auto key_of = [&](int64_t j, bool valid) {
        const int4 kv = valid ? *reinterpret_cast<const int4 *>(kbase + j * a.k_se) : make_int4(0, 0, 0, 0);
        int s = dot16(qv, kv);
        for (int o = 1; o < lpe; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        return (uint32_t)(s + bias);
    };
    // pass 1: level-1 histogram
    for (int i = threadIdx.x; i < 2048; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int64_t j0 = 0; j0 < E; j0 += groups) {
        const int64_t j = j0 + grp;
        const uint32_t u = key_of(j, j < E);
        if (lane_e == 0 && j < E) atomicAdd(&hist[u >> shift], 1u);
    }
    __syncthreads();
    {
        const int per = 2048 / kSelThreads, top = 2047 - threadIdx.x * per;
        int local = 0;
        for (int q = 0; q < per; ++q) local += (int)hist[top - q];
        int tot;
        const int before = block_exclusive_sum(local, s_scan, tot);
        if (before < kE && before + local >= kE) {
            int cum = before;
            for (int q = 0; q < per; ++q) {
                const int hv = (int)hist[top - q];
                if (cum + hv >= kE) { s_misc[0] = top - q; s_misc[1] = cum; break; }
                cum += hv;
            }
        }
        __syncthreads();
    }
    const uint32_t b1 = (uint32_t)s_misc[0];
    const int need = kE - s_misc[1];
    const int nb2 = 1 << shift;
    // pass 2: low bits inside b1
    for (int i = threadIdx.x; i < nb2; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int64_t j0 = 0; j0 < E; j0 += groups) {
        const int64_t j = j0 + grp;
        const uint32_t u = key_of(j, j < E);
        if (lane_e == 0 && j < E && (u >> shift) == b1) atomicAdd(&hist[u & (uint32_t)(nb2 - 1)], 1u);
    }
    __syncthreads();
    {
        const int per = nb2 / kSelThreads, top = nb2 - 1 - threadIdx.x * per;
        int local = 0;
        for (int q = 0; q < per; ++q) local += (int)hist[top - q];
        int tot;
        const int before = block_exclusive_sum(local, s_scan, tot);
        if (before < need && before + local >= need) {
            int cum = before;
            for (int q = 0; q < per; ++q) {
                const int hv = (int)hist[top - q];
                if (cum + hv >= need) { s_misc[2] = top - q; s_misc[3] = cum; break; }
                cum += hv;
            }
        }
        __syncthreads();
    }
    const uint32_t T = (b1 << shift) | (uint32_t)s_misc[2];
    const int n_eq_need = need - s_misc[3];
    // pass 3: ordered compaction, one group-tile of entries at a time
    int eq_base = 0, pos_base = 0;
    for (int64_t j0 = 0; j0 < E; j0 += groups) {
        const int64_t j = j0 + grp;
        const uint32_t u = key_of(j, j < E);
        const bool valid = lane_e == 0 && j < E;
        const int is_eq = valid && u == T, is_gt = valid && u > T;
        int tot_eq;
        const int er = eq_base + block_exclusive_sum(is_eq, s_scan, tot_eq);
        const int take = is_gt || (is_eq && er < n_eq_need);
        int tot_sel;
        const int o = pos_base + block_exclusive_sum(take, s_scan, tot_sel);
        if (take) out[o] = (int32_t)j;
        eq_base += tot_eq;
        pos_base += tot_sel;
    }
}

template <int DI>
cudaError_t launch_score(const CUtensorMap &tq, const CUtensorMap &tk, const PfArgs &p, int grid, bool sample,
                         cudaStream_t s) {
    using Lay = Layout<DI>;
    const size_t smem = 1024 + (size_t)Lay::kSmemTiles + (sample ? (size_t)kBins * kRows * 4 : 0);
    if (sample) {
        static unsigned long long done = 0;
        cudaError_t e = smem_limit_once(score_kernel<DI, true>, (int)smem, done);
        if (e != cudaSuccess) return e;
        score_kernel<DI, true><<<grid, kThreads, smem, s>>>(tq, tk, p);
    } else {
        static unsigned long long done = 0;
        cudaError_t e = smem_limit_once(score_kernel<DI, false>, (int)smem, done);
        if (e != cudaSuccess) return e;
        score_kernel<DI, false><<<grid, kThreads, smem, s>>>(tq, tk, p);
    }
    return cudaGetLastError();
}

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

PrefillIndexPlan plan_index_prefill(int B, int T, int DI, int64_t E_cap, int topk, int num_sms) {
    PrefillIndexPlan p{};
    p.ok = (DI == 64 || DI == 128) && T >= kRows && E_cap >= 4 * kN && topk <= 2048;
    if (!p.ok) return p;
    const int tiles_per_b = (T + kRows - 1) / kRows;
    p.n_qtiles = B * tiles_per_b;
    const int n_tiles_row = (int)((E_cap + kN - 1) / kN);
    // entry segments so that (query tiles x segments) is about one wave at two CTAs per SM
    int seg = 2 * num_sms / p.n_qtiles;
    if (seg < 1) seg = 1;
    if (seg > 16) seg = 16;
    p.seg_tiles = (n_tiles_row + seg - 1) / seg;
    p.n_seg = (n_tiles_row + p.seg_tiles - 1) / p.seg_tiles;
    p.cap_seg = 4096;
    const int64_t rows = (int64_t)B * T;
    size_t off = 0;
    p.off_q16 = off;
    off = al256(off + (size_t)rows * DI * 2);
    p.off_k16 = off;
    off = al256(off + (size_t)B * E_cap * DI * 2);
    p.off_tau = off;
    off = al256(off + (size_t)rows * 4);
    p.off_counts = off;
    off = al256(off + (size_t)rows * p.n_seg * 4);
    p.off_lists = off;
    off = al256(off + (size_t)rows * p.n_seg * p.cap_seg * 8);
    p.total = off;
    return p;
}

cudaError_t launch_index_prefill(const IndexArgs &a, const PrefillIndexPlan &p, void *ws, int num_sms,
                                 cudaStream_t s) {
    (void)num_sms;
    char *w = static_cast<char *>(ws);
    __nv_bfloat16 *q16 = reinterpret_cast<__nv_bfloat16 *>(w + p.off_q16);
    __nv_bfloat16 *k16 = reinterpret_cast<__nv_bfloat16 *>(w + p.off_k16);
    const int64_t rows = (int64_t)a.B * a.T;
    int8_to_bf16_kernel<<<1184, 256, 0, s>>>(a.q, rows, a.DI, a.q_sb, a.q_st, a.T, q16);
    int8_to_bf16_kernel<<<2368, 256, 0, s>>>(a.k, (int64_t)a.B * a.E_cap, a.DI, a.k_sb, a.k_se, a.E_cap, k16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tk;
    {
        const uint64_t dims[2] = {(uint64_t)a.DI, (uint64_t)rows};
        const uint64_t str[1] = {(uint64_t)a.DI};
        if (!make_tmap_bf16(&tq, q16, 2, dims, str, kRows)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)a.DI, (uint64_t)a.E_cap, (uint64_t)a.B};
        const uint64_t str[2] = {(uint64_t)a.DI, (uint64_t)a.E_cap * a.DI};
        if (!make_tmap_bf16(&tk, k16, 3, dims, str, kN)) return cudaErrorInvalidValue;
    }
    PfArgs pa;
    pa.B = a.B;
    pa.T = a.T;
    pa.DI = a.DI;
    pa.m = a.m;
    pa.topk = a.topk;
    pa.E_cap = a.E_cap;
    pa.q_pos0 = a.q_pos0;
    pa.q8 = a.q;
    pa.q_sb = a.q_sb;
    pa.q_st = a.q_st;
    pa.k8 = a.k;
    pa.k_sb = a.k_sb;
    pa.k_se = a.k_se;
    pa.tau = reinterpret_cast<float *>(w + p.off_tau);
    pa.lists = reinterpret_cast<int2 *>(w + p.off_lists);
    pa.counts = reinterpret_cast<int *>(w + p.off_counts);
    pa.n_seg = p.n_seg;
    pa.cap_seg = p.cap_seg;
    pa.seg_tiles = p.seg_tiles;
    pa.idx_out = a.idx_out;
    pa.cnt_out = a.cnt_out;
    if (a.DI == 64) {
        if ((e = launch_score<64>(tq, tk, pa, p.n_qtiles, true, s)) != cudaSuccess) return e;
        if ((e = launch_score<64>(tq, tk, pa, p.n_qtiles * p.n_seg, false, s)) != cudaSuccess) return e;
    } else {
        if ((e = launch_score<128>(tq, tk, pa, p.n_qtiles, true, s)) != cudaSuccess) return e;
        if ((e = launch_score<128>(tq, tk, pa, p.n_qtiles * p.n_seg, false, s)) != cudaSuccess) return e;
    }
    int key_bits = 0;
    while ((1ll << key_bits) <= (long long)a.DI * 32640) ++key_bits;
    const size_t smem = (size_t)kSelCap * 8 + 2048 * 4;
    static unsigned long long done = 0;
    if ((e = smem_limit_once(select_kernel, (int)smem, done)) != cudaSuccess) return e;
    select_kernel<<<(unsigned)rows, kSelThreads, smem, s>>>(pa, key_bits);
    return cudaGetLastError();
}

}  // namespace hsa
