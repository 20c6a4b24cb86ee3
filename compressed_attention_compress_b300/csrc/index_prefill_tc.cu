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
//   sample    per 128-query tile (split over a few CTAs), score every 16th
//             128-entry tile and add to a per-row 128-bin histogram over the
//             row's score bound.
//   collect   per (128-query tile, entry segment): each row's thread first sets
//             the row's candidate threshold tau from the histogram so that about
//             2*k entries of the whole row are expected at or above it, then
//             scores every entry and appends the indices of those at or above
//             tau, in index order, to the row's list for that segment.
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
constexpr int kHalf = kN / 2;  // entries per column half of an S tile
constexpr int kEpiWarps = 8;   // two per TMEM lane quadrant, one per column half
constexpr int kThreads = (kEpiWarps + 2) * 32;  // epilogue warps, MMA warp, TMA warp
constexpr unsigned long long kWaitLimit = 1ull << 24;

struct PfArgs {
    int B, T, DI, m, topk;
    int64_t E_cap;
    const int64_t *q_pos0;
    const int8_t *q8;      // original int8 queries (for bounds / fallback)
    int64_t q_sb, q_st;
    const int8_t *k8;      // original int8 entry vectors (fallback)
    int64_t k_sb, k_se;
    uint32_t *hist;        // [B*T][kBins] sampled score histogram per row (zero between calls)
    int sample_split;      // CTAs sharing one query tile's sampled entry tiles
    int32_t *lists;        // [B*T][S][list_stride] entry indices (scores are recomputed exactly later)
    int *counts;           // [B*T][S]
    int n_seg, cap_seg, seg_tiles;
    int n_lists;      // 2 * n_seg: lists of a row, in index order when concatenated
    int list_stride;  // entries between consecutive lists: cap_seg padded off a power of two, so the
                      // lists of neighbouring rows do not all map to the same memory partition
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
constexpr uint64_t kTwo2 = 0x4000000040000000ull;   // (2.0f, 2.0f)
constexpr uint64_t kBias2 = 0x4B0000004B000000ull;  // (2^23, 2^23)
// Two fp32 fused multiply-adds in one packed instruction.
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t x, uint64_t y, uint64_t z) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(x), "l"(y), "l"(z));
    return d;
}
// Two fp32 additions in one packed instruction (lanes: low and high 32 bits).
__device__ __forceinline__ uint64_t add_f32x2(uint64_t x, uint64_t y) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(x), "l"(y));
    return d;
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

// Histogram range of one query row: every score lies within +-(128 * sum|q| + 1).
__device__ __forceinline__ void row_bins(const int8_t *q, int DI, float &lo, float &inv_w) {
    int sabs = 0;
    const int4 *qp = reinterpret_cast<const int4 *>(q);
    for (int c = 0; c < DI / 16; ++c) {
        const int4 w4 = qp[c];
        const int wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
            for (int by = 0; by < 4; ++by) {
                const int x = (int)(int8_t)(wv[h] >> (8 * by));
                sabs += x < 0 ? -x : x;
            }
    }
    const float R = 128.f * (float)sabs + 1.f;
    lo = -R;
    inv_w = (float)kBins / (2.f * R);
}

// Candidate threshold of a row from its sampled histogram: about 2*k of the row's E
// entries are expected at or above it (the sample count above it is ~2*k/16, so the
// row falling short of k candidates is a > 5 sigma event; select still handles it).
// -inf (every entry a candidate) when the row has at most 4*k entries.
__device__ float row_threshold(const uint32_t *hist, int64_t E, int topk, float lo, float inv_w) {
    const int kE = (int)(E < topk ? E : topk);
    if (E <= 4 * (int64_t)kE) return -INFINITY;
    const uint4 *h4 = reinterpret_cast<const uint4 *>(hist);
    int n_samp = 0;
#pragma unroll 4
    for (int i = 0; i < kBins / 4; ++i) {
        const uint4 x = h4[i];
        n_samp += (int)(x.x + x.y + x.z + x.w);
    }
    if (n_samp == 0) return -INFINITY;
    const float want = 2.0f * (float)kE * (float)n_samp / (float)E;
    float cum = 0.f;
#pragma unroll 1
    for (int i = kBins - 1; i >= 0; --i) {
        const float c = (float)hist[i];
        if (cum + c >= want) {
            // the samples still wanted, taken as spread evenly over bin i
            const float f = (want - cum) / c;
            return floorf(lo + ((float)(i + 1) - f) / inv_w);
        }
        cum += c;
    }
    return -INFINITY;
}

// Column half h of an S tile (entries [64h, 64h + 64)) is fed from its own run of
// 64-entry blocks.  collect: the CTA's segment is cut into two halves of whole
// blocks and step `it` scores block `it` of each half, so each half's list comes out
// in index order and the half-0 list precedes the half-1 list.  sample: the two
// halves of one 128-entry tile.
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

    // work item: query tile of one sequence, entry segment (sample: share of the sampled tiles)
    const int tiles_per_b = (a.T + kRows - 1) / kRows;
    const int item = blockIdx.x;
    const int seg = SAMPLE ? item % a.sample_split : item % a.n_seg;
    const int qtile = SAMPLE ? item / a.sample_split : item / a.n_seg;
    const int b = qtile / tiles_per_b;
    const int t0 = (qtile - b * tiles_per_b) * kRows;
    const int64_t p_last = a.q_pos0[b] + (t0 + kRows - 1 < a.T ? t0 + kRows - 1 : a.T - 1);
    int64_t E_last = num_entries(p_last, a.m);
    if (E_last > a.E_cap) E_last = a.E_cap;
    int n_my;                        // steps (S tiles) of this CTA
    int64_t tile_begin = 0, tile_step = 0;  // sample: 128-entry tiles scored
    int64_t seg_begin = 0, mid = 0, seg_end = 0;  // collect: entry ranges of the halves
    if (SAMPLE) {
        const int64_t n_tiles_row = (E_last + kN - 1) / kN;
        tile_begin = (int64_t)seg * kSampleEvery;
        tile_step = (int64_t)kSampleEvery * a.sample_split;
        n_my = n_tiles_row > tile_begin ? (int)((n_tiles_row - tile_begin + tile_step - 1) / tile_step) : 0;
    } else {
        seg_begin = (int64_t)seg * a.seg_tiles * kN;
        seg_end = seg_begin + (int64_t)a.seg_tiles * kN;
        const int64_t used = (E_last < seg_end ? E_last : seg_end) - seg_begin;
        const int nblk = used > 0 ? (int)((used + kHalf - 1) / kHalf) : 0;
        n_my = (nblk + 1) / 2;
        mid = seg_begin + (int64_t)n_my * kHalf;
    }
    // first entry of column half h at step it
    auto half_start = [&](int h, int it) -> int64_t {
        if (SAMPLE) return (tile_begin + it * tile_step) * kN + h * kHalf;
        return (h ? mid : seg_begin) + (int64_t)it * kHalf;
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bars.q_full, 1);
        for (int i = 0; i < Lay::kStages; ++i) {
            mbar_init(&bars.k_full[i], 1);
            mbar_init(&bars.k_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.s_free[i], kEpiWarps * 32);
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

    if (warp == kEpiWarps + 1) {
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
                mbar_expect_tx(&bars.k_full[st], Lay::kK);
                last[st] = it / Lay::kStages;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // rows past the tensor's end are zero-filled; past the segment they are masked
                    const int row0 = (int)half_start(h, it);
#pragma unroll
                    for (int kb = 0; kb < Lay::kKB; ++kb)
                        tc::tma_load_3d(sK + st * Lay::kK + kb * kN * 128 + h * kHalf * 128, &tm_k, kb * 64, row0, b,
                                        &bars.k_full[st]);
                }
            }
            if (!ok) s_abort = 1;
            volatile int never = 0;
            wait_bar(&bars.q_full, 0u, &never);
            for (int st = 0; st < Lay::kStages; ++st)
                if (last[st] >= 0) wait_bar(&bars.k_full[st], (unsigned)(last[st] & 1), &never);
        }
    } else if (warp == kEpiWarps) {
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
        // epilogue: warp (quadrant q, half h); thread owns query row t0 + r, columns [64h, 64h + 64)
        const int q = warp & 3, h = warp >> 2;
        const int r = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int t = t0 + r;
        const bool live = t < a.T;
        const int64_t row = (int64_t)b * a.T + (live ? t : 0);
        const int64_t p = a.q_pos0[b] + t;
        int64_t E = num_entries(p, a.m);
        if (E > a.E_cap) E = a.E_cap;
        if (!live) E = 0;
        // entries of this half that count: below E, and (collect) inside the half's range
        const int64_t limit = SAMPLE ? E : ((h ? seg_end : mid) < E ? (h ? seg_end : mid) : E);
        float lo = 0.f, inv_w = 0.f;
        if (live) row_bins(a.q8 + b * a.q_sb + (int64_t)t * a.q_st, DI, lo, inv_w);
        uint64_t ntau2 = 0;  // (-tau, -tau) as a packed f32 pair
        float c1 = 0.f;      // 1 - tau
        int cnt = 0;
        const int list_id = seg * 2 + h;
        int32_t *my_list = nullptr;
        if (!SAMPLE) {
            const float tau = live ? row_threshold(a.hist + row * kBins, E, a.topk, lo, inv_w) : INFINITY;
            ntau2 = ((uint64_t)__float_as_uint(-tau) << 32) | __float_as_uint(-tau);
            c1 = 1.f - tau;
            my_list = a.lists + (row * a.n_lists + list_id) * (int64_t)a.list_stride;
        }
        bool ok = true;
        for (int it = 0; it < n_my && ok; ++it) {
            const int sb = it & 1;
            ok = wait_bar(&bars.s_full[sb], (unsigned)((it >> 1) & 1), &s_abort);
            if (!ok) break;
            tc::fence_after();
            const int64_t j0 = half_start(h, it);
            const int64_t rem = limit - j0;
            const int n_valid = rem <= 0 ? 0 : (rem >= kHalf ? kHalf : (int)rem);
            if (SAMPLE) {
                uint32_t v[kHalf];
#pragma unroll
                for (int c = 0; c < kHalf / 32; ++c)
                    tc::tmem_ld32(tmem + sb * kN + lane_off + h * kHalf + c * 32, v + c * 32);
                tc::tmem_wait_ld();
                tc::fence_before();
                arrive(&bars.s_free[sb]);  // S has been copied to registers
#pragma unroll
                for (int e = 0; e < kHalf; ++e) {
                    int bin = __float2int_rz((__uint_as_float(v[e]) - lo) * inv_w);
                    bin = bin < 0 ? 0 : (bin >= kBins ? kBins - 1 : bin);
                    atomicAdd(&sHist[bin * kRows + r], e < n_valid ? 1u : 0u);  // no branch per element
                }
            } else {
                // hit masks of the two 32-column chunks (bit e: column 32c + e scored at or
                // above tau; scores and tau are integers below 2^24, so every step below is
                // exact).  The chunks take different routes to balance the integer and the
                // floating-point pipes:
                //   chunk 0: sign bits of S - tau (packed add), gathered by funnel shifts;
                //   chunk 1: h = sat(S + 1 - tau) is 1.0 or 0.0, gathered by a packed
                //            Horner sum m = 2m + h over columns (e, e + 16), then the two
                //            16-bit integers are taken from the float bits (m + 2^23).
                uint32_t v[32];
                tc::tmem_ld32(tmem + sb * kN + lane_off + h * kHalf, v);
                tc::tmem_wait_ld();
                uint32_t below0 = 0;
#pragma unroll
                for (int e = 30; e >= 0; e -= 2) {
                    const uint64_t d = add_f32x2(((uint64_t)v[e + 1] << 32) | v[e], ntau2);
                    below0 = __funnelshift_l((uint32_t)(d >> 32), below0, 1);
                    below0 = __funnelshift_l((uint32_t)d, below0, 1);
                }
                tc::tmem_ld32(tmem + sb * kN + lane_off + h * kHalf + 32, v);
                tc::tmem_wait_ld();
                tc::fence_before();
                arrive(&bars.s_free[sb]);  // S has been copied to registers
                uint64_t m2 = 0;
#pragma unroll
                for (int e = 15; e >= 0; --e) {
                    const float h_lo = __saturatef(__uint_as_float(v[e]) + c1);
                    const float h_hi = __saturatef(__uint_as_float(v[e + 16]) + c1);
                    m2 = fma_f32x2(m2, kTwo2, ((uint64_t)__float_as_uint(h_hi) << 32) | __float_as_uint(h_lo));
                }
                m2 = add_f32x2(m2, kBias2);
                const uint32_t hits1 = __byte_perm((uint32_t)m2, (uint32_t)(m2 >> 32), 0x5410);
                uint64_t hits = ((uint64_t)hits1 << 32) | ~below0;
                if (n_valid < kHalf) hits &= (1ull << n_valid) - 1ull;
                while (hits) {  // usually 0-3 per 64 columns
                    const int e = __ffsll((long long)hits) - 1;
                    hits &= hits - 1ull;
                    if (cnt < a.cap_seg) my_list[cnt] = (int32_t)(j0 + e);
                    ++cnt;
                }
            }
        }
        if (!ok) s_abort = 1;
        if (SAMPLE) {
            // both halves have added to the row's bins (every epilogue warp reaches this
            // barrier: the loop above is bounded), then each flushes half of the bins
            asm volatile("bar.sync 1, %0;\n" ::"r"(kEpiWarps * 32) : "memory");
            if (live) {
                uint32_t *gh = a.hist + row * kBins;
                for (int i = h * (kBins / 2); i < (h + 1) * (kBins / 2); ++i) {
                    const uint32_t c = sHist[i * kRows + r];
                    if (c) atomicAdd(gh + i, c);
                }
            }
        } else if (live) {
            a.counts[row * a.n_lists + list_id] = cnt;
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// --------------------------------------------------------------- selection
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCap = 4096;  // candidates held in shared memory (2-3k are expected)

__device__ __forceinline__ int dot16(const int4 &x, const int4 &y) {
    int s = __dp4a(x.x, y.x, 0);
    s = __dp4a(x.y, y.y, s);
    s = __dp4a(x.z, y.z, s);
    return __dp4a(x.w, y.w, s);
}

// The bin of hist[0 .. nb) (bin index grows with the key) where the count taken from
// the top first reaches `want`: s_misc[slot] = bin, s_misc[slot + 1] = count above it.
__device__ void find_bin(const unsigned *hist, int nb, int want, int *s_scan, int *s_misc, int slot) {
    const int per = nb / kSelThreads, top = nb - 1 - threadIdx.x * per;
    int local = 0;
    for (int q = 0; q < per; ++q) local += (int)hist[top - q];
    int tot;
    const int before = block_exclusive_sum(local, s_scan, tot);
    if (before < want && before + local >= want) {
        int cum = before;
        for (int q = 0; q < per; ++q) {
            const int hv = (int)hist[top - q];
            if (cum + hv >= want) {
                s_misc[slot] = top - q;
                s_misc[slot + 1] = cum;
                break;
            }
            cum += hv;
        }
    }
    __syncthreads();
}

// Exact k-th largest key over items 0 .. n-1 (n >= kE): two radix levels of 11 and
// key_bits - 11 bits.  Returns the threshold key T and how many items equal to T
// belong to the top kE (the rest of the top kE are the items above T).
template <class KeyF>
__device__ void kth_key(int64_t n, int kE, int key_bits, KeyF key, unsigned *hist, int *s_scan, int *s_misc,
                        uint32_t &T, int &n_eq_need) {
    const int shift = key_bits - 11;
    for (int i = threadIdx.x; i < 2048; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += kSelThreads) atomicAdd(&hist[key(i) >> shift], 1u);
    __syncthreads();
    find_bin(hist, 2048, kE, s_scan, s_misc, 0);
    const uint32_t b1 = (uint32_t)s_misc[0];
    const int need = kE - s_misc[1];
    const int nb2 = 1 << shift;
    for (int i = threadIdx.x; i < nb2; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += kSelThreads) {
        const uint32_t u = key(i);
        if ((u >> shift) == b1) atomicAdd(&hist[u & (uint32_t)(nb2 - 1)], 1u);
    }
    __syncthreads();
    find_bin(hist, nb2, need, s_scan, s_misc, 2);
    T = (b1 << shift) | (uint32_t)s_misc[2];
    n_eq_need = need - s_misc[3];
}

// Ordered compaction of items 0 .. n-1 (ascending entry index): keeps every item whose
// key is above T and the first n_eq_need items whose key equals T, and writes their
// entry indices to out in item order.  Each warp owns one contiguous run of items;
// output slots come from per-warp counts and lane ballots.
template <class KeyF, class IdxF>
__device__ void ordered_take(int64_t n, uint32_t T, int n_eq_need, KeyF key, IdxF idx, int *s_w, int32_t *out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t run = ((n + kSelWarps - 1) / kSelWarps + 31) & ~(int64_t)31;
    const int64_t w0 = warp * run < n ? warp * run : n;
    const int64_t w1 = w0 + run < n ? w0 + run : n;
    int gt = 0, eq = 0;
    for (int64_t i = w0 + lane; i < w1; i += 32) {
        const uint32_t u = key(i);
        gt += u > T;
        eq += u == T;
    }
    gt = __reduce_add_sync(~0u, gt);
    eq = __reduce_add_sync(~0u, eq);
    if (lane == 0) {
        s_w[warp] = gt;
        s_w[kSelWarps + warp] = eq;
    }
    __syncthreads();
    int eq_run = 0, sel_run = 0;
    for (int v = 0; v < warp; ++v) {
        const int ev = s_w[kSelWarps + v];
        int tk = n_eq_need - eq_run;
        tk = tk < 0 ? 0 : (tk > ev ? ev : tk);
        sel_run += s_w[v] + tk;
        eq_run += ev;
    }
    const uint32_t lt = (1u << lane) - 1u;
    for (int64_t base = w0; base < w1; base += 32) {  // warp-uniform trip count
        const int64_t i = base + lane;
        const bool valid = i < w1;
        const uint32_t u = valid ? key(i) : 0u;
        const bool is_eq = valid && u == T;
        const uint32_t em = __ballot_sync(~0u, is_eq);
        const bool take = (valid && u > T) || (is_eq && eq_run + __popc(em & lt) < n_eq_need);
        const uint32_t tm = __ballot_sync(~0u, take);
        if (take) out[sel_run + __popc(tm & lt)] = idx(i);
        eq_run += __popc(em);
        sel_run += __popc(tm);
    }
    __syncthreads();
}

template <int DI>
__global__ void __launch_bounds__(kSelThreads, 4) select_kernel(PfArgs a) {
    constexpr int kKeyBits = DI == 64 ? 21 : 22;  // biased keys lie in [0, 2 * DI * 127^2]
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t *s_u = reinterpret_cast<uint32_t *>(smem);            // [kSelCap]
    int32_t *s_j = reinterpret_cast<int32_t *>(s_u + kSelCap);     // [kSelCap]
    unsigned *hist = reinterpret_cast<unsigned *>(s_j + kSelCap);  // [2048]
    __shared__ int s_scan[33];
    __shared__ int s_misc[8];
    __shared__ int s_off[33];
    __shared__ int s_w[2 * kSelWarps];

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
    for (int i = threadIdx.x; i < kBins; i += kSelThreads) a.hist[row * kBins + i] = 0;  // left zero
    int4 qv[DI / 16];
    {
        const int4 *qp = reinterpret_cast<const int4 *>(a.q8 + b * a.q_sb + (int64_t)t * a.q_st);
#pragma unroll
        for (int q = 0; q < DI / 16; ++q) qv[q] = qp[q];
    }
    for (int i = kE + threadIdx.x; i < a.topk; i += kSelThreads) out[i] = -1;
    if (threadIdx.x == 0) a.cnt_out[row] = kE;
    if (kE == 0) return;
    const int bias = DI * 16256;

    // the segment lists, each in index order, concatenated in segment order
    if (threadIdx.x == 0) {
        int off = 0;
        bool fits = true;
        for (int sg = 0; sg < a.n_lists; ++sg) {
            const int c = a.counts[row * a.n_lists + sg];
            if (c > a.cap_seg) fits = false;
            s_off[sg] = off;
            off += c;
        }
        s_off[a.n_lists] = off;
        s_misc[4] = off;
        s_misc[5] = fits && off >= kE;  // the lists hold the whole top-k
    }
    __syncthreads();
    const int n = s_misc[4];
    const bool from_lists = s_misc[5];
    const int32_t *lists_row = a.lists + row * a.n_lists * (int64_t)a.list_stride;
    const char *kbase = reinterpret_cast<const char *>(a.k8 + b * a.k_sb);
    auto key_of = [&](int64_t j) {
        const int4 *kr = reinterpret_cast<const int4 *>(kbase + j * a.k_se);
        int sc = 0;
#pragma unroll
        for (int q = 0; q < DI / 16; ++q) sc += dot16(qv[q], __ldg(kr + q));  // one 16-byte load each
        return (uint32_t)(sc + bias);
    };
    uint32_t T;
    int n_eq_need;
    if (from_lists && n <= kSelCap) {
        // common case: stage (key, index) in shared memory -- indices first (coalesced),
        // then the keys with several independent row reads in flight per thread
        for (int sg = 0; sg < a.n_lists; ++sg) {
            const int c = s_off[sg + 1] - s_off[sg];
            const int32_t *lst = lists_row + sg * (int64_t)a.list_stride;
            for (int i = threadIdx.x; i < c; i += kSelThreads) s_j[s_off[sg] + i] = lst[i];
        }
        __syncthreads();
#pragma unroll 4
        for (int i = threadIdx.x; i < n; i += kSelThreads) s_u[i] = key_of(s_j[i]);
        __syncthreads();
        auto key_s = [&](int64_t i) { return s_u[i]; };
        auto idx_s = [&](int64_t i) { return s_j[i]; };
        kth_key(n, kE, kKeyBits, key_s, hist, s_scan, s_misc, T, n_eq_need);
        ordered_take(n, T, n_eq_need, key_s, idx_s, s_w, out);
        return;
    }
    // Streaming exact selection over items 0 .. n_items-1 (index order), keys
    // recomputed on every pass: the concatenated lists when they hold the top-k but
    // not in shared memory, otherwise every entry of the row (a sampled threshold that
    // came out too high, or a list overflow).
    const int64_t n_items = from_lists ? (int64_t)n : E;
    auto index_of = [&](int64_t i) -> int32_t {
        if (!from_lists) return (int32_t)i;
        int sg = 0;
        while (sg + 1 < a.n_lists && i >= s_off[sg + 1]) ++sg;
        return lists_row[sg * (int64_t)a.list_stride + (i - s_off[sg])];
    };
    auto key_g = [&](int64_t i) { return key_of(index_of(i)); };
    kth_key(n_items, kE, kKeyBits, key_g, hist, s_scan, s_misc, T, n_eq_need);
    ordered_take(n_items, T, n_eq_need, key_g, index_of, s_w, out);
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
    p.ok = (DI == 64 || DI == 128) && T >= kRows && E_cap >= 4 * kN && topk <= 1024;
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
    // sampled tiles of one query tile shared by several CTAs so the sample pass fills the GPU
    p.sample_split = num_sms / p.n_qtiles;
    if (p.sample_split < 1) p.sample_split = 1;
    if (p.sample_split > 8) p.sample_split = 8;
    const int64_t rows = (int64_t)B * T;
    size_t off = 0;
    p.off_q16 = off;
    off = al256(off + (size_t)rows * DI * 2);
    p.off_k16 = off;
    off = al256(off + (size_t)B * E_cap * DI * 2);
    p.off_hist = off;
    off = al256(off + (size_t)rows * kBins * 4);
    p.off_counts = off;
    off = al256(off + (size_t)rows * 2 * p.n_seg * 4);
    p.off_lists = off;
    off = al256(off + (size_t)rows * 2 * p.n_seg * (p.cap_seg + 40) * 4);
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
        if (!make_tmap_bf16(&tk, k16, 3, dims, str, kHalf)) return cudaErrorInvalidValue;
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
    pa.hist = reinterpret_cast<uint32_t *>(w + p.off_hist);
    pa.sample_split = p.sample_split;
    pa.lists = reinterpret_cast<int32_t *>(w + p.off_lists);
    pa.counts = reinterpret_cast<int *>(w + p.off_counts);
    pa.n_seg = p.n_seg;
    pa.n_lists = 2 * p.n_seg;
    pa.cap_seg = p.cap_seg;
    pa.list_stride = p.cap_seg + 40;
    pa.seg_tiles = p.seg_tiles;
    pa.idx_out = a.idx_out;
    pa.cnt_out = a.cnt_out;
    if (a.DI == 64) {
        if ((e = launch_score<64>(tq, tk, pa, p.n_qtiles * p.sample_split, true, s)) != cudaSuccess) return e;
        if ((e = launch_score<64>(tq, tk, pa, p.n_qtiles * p.n_seg, false, s)) != cudaSuccess) return e;
    } else {
        if ((e = launch_score<128>(tq, tk, pa, p.n_qtiles * p.sample_split, true, s)) != cudaSuccess) return e;
        if ((e = launch_score<128>(tq, tk, pa, p.n_qtiles * p.n_seg, false, s)) != cudaSuccess) return e;
    }
    const size_t smem = (size_t)kSelCap * 8 + 2048 * 4;
    if (a.DI == 64) {
        static unsigned long long done = 0;
        if ((e = smem_limit_once(select_kernel<64>, (int)smem, done)) != cudaSuccess) return e;
        select_kernel<64><<<(unsigned)rows, kSelThreads, smem, s>>>(pa);
    } else {
        static unsigned long long done = 0;
        if ((e = smem_limit_once(select_kernel<128>, (int)smem, done)) != cudaSuccess) return e;
        select_kernel<128><<<(unsigned)rows, kSelThreads, smem, s>>>(pa);
    }
    return cudaGetLastError();
}

}  // namespace hsa
