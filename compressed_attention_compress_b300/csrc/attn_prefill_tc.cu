// Prefill attention over all compressed entries plus the window (HCA layer) on
// the 5th-generation tensor cores: tcgen05 MMAs with TMEM accumulators, operands
// brought in by TMA.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制: HCA runs dense attention over
// every heavily compressed entry; the sliding-window paragraph adds the most
// recent raw tokens to the same softmax; strict causality limits query p to the
// E(p) = floor((p+1)/m) complete blocks.
//
// Queries are the rows of q viewed as [B*T*H, d] (d = 128); a tile is 128 rows,
// i.e. 128/H consecutive tokens with all their heads (one KV head).  For a tile
// the KV sequence is ceil(E(p_last)/128) entry tiles of Kc/Vc, then the raw
// window tokens [p_first - W + 1, p_last] in 128-token tiles; per-row masks
// apply E(p_row) and the row's own window.  One persistent CTA per SM walks
// query tiles; its warps specialise:
//   warps 0-3  softmax: one query row per thread.  S comes from TMEM, P (bf16)
//              goes to shared memory for the second MMA, O is rescaled in TMEM
//              only when a row's running max grows by more than 2^8 (until then
//              the stale max keeps P <= 256), and the final O / l is written out.
//   warp 4     MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//              buffers, then O += P_{j-1} V_{j-1}; completion via tcgen05.commit.
//   warp 5     TMA producer (one thread): Q tile, then K_j / V_j into a 2-stage
//              ring.
// All waits are bounded; a wait that gives up raises the device flag and the
// CTA stops issuing work.
#include <math.h>
#include <stdio.h>

#include <cudaTypedefs.h>

#include "internal.h"
#include "tc_common.cuh"

namespace hsa {

namespace {

constexpr int kRows = 128;   // query rows per tile
constexpr int kCols = 128;   // KV items per tile
constexpr int kD = 128;      // head dim
constexpr int kTileBytes = kRows * kD * 2;     // 32 KiB (two 128-byte-wide K blocks)
constexpr int kBlk = kRows * 128;              // 16 KiB per 64-element block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;  // log2 units
constexpr unsigned long long kWaitLimit = 1ull << 24;

struct PrefillTcArgs {
    int B, T, H, m, window;
    int64_t E_cap, N_cap;
    const int64_t *q_pos0;
    float scale_log2;
    __nv_bfloat16 *out;
    float *lse;
    int n_qtiles;
};

struct __align__(8) Bars {
    uint64_t q_full, q_empty;
    uint64_t kv_full[2], kv_empty[2];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, o_done, o_free;
    uint64_t mma_fin;
};

struct TileInfo {
    int b;
    int64_t p_first, p_last;
    int n_ent, n_win;  // entry tiles, window tiles
    int64_t w0;        // first raw token of the window range
};

__device__ __forceinline__ TileInfo tile_info(const PrefillTcArgs &a, int qt) {
    TileInfo ti;
    const int64_t rows_b = (int64_t)a.T * a.H;
    const int64_t r0 = (int64_t)qt * kRows;
    ti.b = (int)(r0 / rows_b);
    const int64_t rin = r0 - ti.b * rows_b;
    const int64_t tok_first = rin / a.H, tok_last = (rin + kRows - 1) / a.H;
    const int64_t p0 = a.q_pos0[ti.b];
    ti.p_first = p0 + tok_first;
    ti.p_last = p0 + tok_last;
    int64_t E = num_entries(ti.p_last, a.m);
    if (E > a.E_cap) E = a.E_cap;
    ti.n_ent = (int)((E + kCols - 1) / kCols);
    ti.w0 = ti.p_first - a.window + 1;
    const int64_t span = a.window > 0 ? ti.p_last - ti.w0 + 1 : 0;
    ti.n_win = (int)((span + kCols - 1) / kCols);
    return ti;
}

// Bounded wait; gives up (and raises the device flag) after kWaitLimit polls or as
// soon as another role of the CTA has given up.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, unsigned parity, volatile int *abort) {
    for (unsigned long long i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    raise_flag(FLAG_ATTN_RANGE | 0x400u);
    *abort = 1;
    return false;
}
__device__ __forceinline__ void arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(192, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                           const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kr,
                           const __grid_constant__ CUtensorMap tm_vr, PrefillTcArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];  // rounded up to 1024 below, at run time
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *sQ = smem;                       // 32 KiB
    unsigned char *sKV = smem + kTileBytes;         // 2 stages x (K 32 KiB + V 32 KiB)
    unsigned char *sP = sKV + 4 * kTileBytes;       // 32 KiB
    __shared__ Bars bars;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.kv_full[i], 1);
            mbar_init(&bars.kv_empty[i], 1);
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.s_free[i], kRows);
        }
        mbar_init(&bars.p_full, kRows);
        mbar_init(&bars.o_done, 1);
        mbar_init(&bars.o_free, kRows);
        mbar_init(&bars.mma_fin, 1);
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t tS[2] = {tmem, tmem + 128};
    const uint32_t tO = tmem + 256;

    if (warp == 5) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int g = 0, it = 0;
            int q_issued = 0, last_use[2] = {-1, -1};
            bool ok = true;
            for (int qt = blockIdx.x; qt < a.n_qtiles && ok; qt += gridDim.x, ++it) {
                const TileInfo ti = tile_info(a, qt);
                if (it > 0) ok = wait_bar(&bars.q_empty, (unsigned)((it - 1) & 1), &s_abort);
                if (!ok) break;
                mbar_expect_tx(&bars.q_full, kTileBytes);
                tc::tma_load_2d(sQ, &tm_q, 0, qt * kRows, &bars.q_full);
                tc::tma_load_2d(sQ + kBlk, &tm_q, 64, qt * kRows, &bars.q_full);
                ++q_issued;
                const int n_kv = ti.n_ent + ti.n_win;
                for (int j = 0; j < n_kv && ok; ++j, ++g) {
                    const int s = g & 1;
                    if (g >= 2) ok = wait_bar(&bars.kv_empty[s], (unsigned)(((g - 2) >> 1) & 1), &s_abort);
                    if (!ok) break;
                    unsigned char *dk = sKV + s * 2 * kTileBytes;
                    unsigned char *dv = dk + kTileBytes;
                    mbar_expect_tx(&bars.kv_full[s], 2 * kTileBytes);
                    last_use[s] = g >> 1;
                    if (j < ti.n_ent) {
                        const int y = j * kCols;
                        tc::tma_load_3d(dk, &tm_kc, 0, y, ti.b, &bars.kv_full[s]);
                        tc::tma_load_3d(dk + kBlk, &tm_kc, 64, y, ti.b, &bars.kv_full[s]);
                        tc::tma_load_3d(dv, &tm_vc, 0, y, ti.b, &bars.kv_full[s]);
                        tc::tma_load_3d(dv + kBlk, &tm_vc, 64, y, ti.b, &bars.kv_full[s]);
                    } else {
                        const int y = (int)(ti.w0 + (int64_t)(j - ti.n_ent) * kCols);
                        tc::tma_load_3d(dk, &tm_kr, 0, y, ti.b, &bars.kv_full[s]);
                        tc::tma_load_3d(dk + kBlk, &tm_kr, 64, y, ti.b, &bars.kv_full[s]);
                        tc::tma_load_3d(dv, &tm_vr, 0, y, ti.b, &bars.kv_full[s]);
                        tc::tma_load_3d(dv + kBlk, &tm_vr, 64, y, ti.b, &bars.kv_full[s]);
                    }
                }
            }
            if (!ok) s_abort = 1;
            // let every copy this thread issued land before the CTA can exit
            volatile int never = 0;
            if (q_issued > 0) wait_bar(&bars.q_full, (unsigned)((q_issued - 1) & 1), &never);
            for (int st = 0; st < 2; ++st)
                if (last_use[st] >= 0) wait_bar(&bars.kv_full[st], (unsigned)(last_use[st] & 1), &never);
        }
    } else if (warp == 4) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_bf16(kRows, kCols, false, false);
            constexpr uint32_t idO = tc::idesc_bf16(kRows, kD, false, true);
            const uint32_t aQ = smem_u32(sQ), aP = smem_u32(sP);
            int g = 0, it = 0;
            bool ok = true;
            auto issue_pv = [&](int gg, bool first) {
                // O (+)= P V_gg : P K-major [rows x items], V MN-major [items x d]
                const int s = gg & 1;
                const uint32_t aV = smem_u32(sKV + s * 2 * kTileBytes + kTileBytes);
#pragma unroll
                for (int kk = 0; kk < kCols / 16; ++kk) {
                    const uint64_t da = tc::desc_sw128(aP + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
                    const uint64_t db = tc::desc_sw128(aV + kk * 16 * 128, kBlk, 1024);
                    tc::mma_bf16(tO, da, db, idO, (first && kk == 0) ? 0u : 1u);
                }
                tc::commit(&bars.o_done);
                tc::commit(&bars.kv_empty[s]);
            };
            for (int qt = blockIdx.x; qt < a.n_qtiles && ok; qt += gridDim.x, ++it) {
                const TileInfo ti = tile_info(a, qt);
                const int n_kv = ti.n_ent + ti.n_win;
                ok = wait_bar(&bars.q_full, (unsigned)(it & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                if (n_kv == 0) tc::commit(&bars.q_empty);
                const int g0 = g;
                for (int j = 0; j < n_kv && ok; ++j, ++g) {
                    const int s = g & 1;
                    ok = wait_bar(&bars.kv_full[s], (unsigned)((g >> 1) & 1), &s_abort);
                    if (ok && g >= 2) ok = wait_bar(&bars.s_free[s], (unsigned)(((g - 2) >> 1) & 1), &s_abort);
                    if (!ok) break;
                    tc::fence_after();
                    const uint32_t aK = smem_u32(sKV + s * 2 * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint64_t da = tc::desc_sw128(aQ + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
                        const uint64_t db = tc::desc_sw128(aK + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
                        tc::mma_bf16(tS[s], da, db, idS, kk > 0 ? 1u : 0u);
                    }
                    tc::commit(&bars.s_full[s]);
                    if (j == n_kv - 1) tc::commit(&bars.q_empty);
                    if (j > 0) {
                        // PV for the previous item tile of this query tile
                        ok = wait_bar(&bars.p_full, (unsigned)((g - 1) & 1), &s_abort);
                        if (!ok) break;
                        if (j == 1 && it > 0) ok = wait_bar(&bars.o_free, (unsigned)((it - 1) & 1), &s_abort);
                        if (!ok) break;
                        tc::fence_after();
                        issue_pv(g - 1, j == 1);
                    }
                }
                if (ok && n_kv > 0) {
                    ok = wait_bar(&bars.p_full, (unsigned)((g - 1) & 1), &s_abort);
                    if (ok && n_kv == 1 && it > 0) ok = wait_bar(&bars.o_free, (unsigned)((it - 1) & 1), &s_abort);
                    if (ok) {
                        tc::fence_after();
                        issue_pv(g - 1, n_kv == 1);
                    }
                }
                (void)g0;
            }
            if (!ok) s_abort = 1;
            // every MMA this thread issued completes before TMEM is released
            tc::commit(&bars.mma_fin);
            volatile int never = 0;
            wait_bar(&bars.mma_fin, 0u, &never);
        }
    } else {
        // ---------------------------------------------------------- softmax rows
        const int r = threadIdx.x;  // 0..127 == TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        int g = 0, it = 0;
        bool ok = true;
        for (int qt = blockIdx.x; qt < a.n_qtiles && ok; qt += gridDim.x, ++it) {
            const TileInfo ti = tile_info(a, qt);
            const int n_kv = ti.n_ent + ti.n_win;
            const int64_t qrow = (int64_t)qt * kRows + r;
            const int64_t rin = qrow - (int64_t)ti.b * a.T * a.H;
            const int64_t p = a.q_pos0[ti.b] + rin / a.H;
            int64_t E = num_entries(p, a.m);
            if (E > a.E_cap) E = a.E_cap;
            const int64_t wlo = (p - a.window + 1) < 0 ? 0 : p - a.window + 1;
            const int64_t whi = p < a.N_cap ? p : a.N_cap - 1;  // the raw cache must hold the query
            if (p >= a.N_cap && a.window > 0) raise_flag(FLAG_ATTN_RANGE);
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < n_kv && ok; ++j, ++g) {
                const int s = g & 1;
                ok = wait_bar(&bars.s_full[s], (unsigned)((g >> 1) & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                float x[kCols];
#pragma unroll
                for (int c = 0; c < kCols / 32; ++c) {
                    uint32_t v[32];
                    tc::tmem_ld32(tS[s] + lane_off + c * 32, v);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(v[e]);
                }
                tc::fence_before();
                arrive(&bars.s_free[s]);
                // mask and scale (log2 domain)
                float mx = -INFINITY;
                if (j < ti.n_ent) {
                    const int64_t base = (int64_t)j * kCols;
#pragma unroll
                    for (int c = 0; c < kCols; ++c) {
                        x[c] = (base + c < E) ? x[c] * a.scale_log2 : -INFINITY;
                        mx = fmaxf(mx, x[c]);
                    }
                } else {
                    const int64_t base = ti.w0 + (int64_t)(j - ti.n_ent) * kCols;
#pragma unroll
                    for (int c = 0; c < kCols; ++c) {
                        const int64_t t = base + c;
                        x[c] = (t >= wlo && t <= whi) ? x[c] * a.scale_log2 : -INFINITY;
                        mx = fmaxf(mx, x[c]);
                    }
                }
                // the P buffer and O are free once the previous PV has completed
                if (g > 0) ok = wait_bar(&bars.o_done, (unsigned)((g - 1) & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                bool rescale = false;
                float alpha = 1.f;
                if (mx > m_used + kRescale) {
                    if (m_used != -INFINITY) {
                        alpha = tc::ex2(m_used - mx);
                        rescale = j > 0;
                    }
                    l *= (m_used == -INFINITY) ? 0.f : alpha;
                    m_used = mx;
                }
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int c = 0; c < kD / 32; ++c) {
                        uint32_t v[32];
                        tc::tmem_ld32(tO + lane_off + c * 32, v);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tc::tmem_st32(tO + lane_off + c * 32, v);
                    }
                    tc::tmem_wait_st();
                }
                // P = 2^(x - m_used) in bf16, 128-byte-swizzled K-major rows
                float sum = 0.f;
                const float mu = m_used == -INFINITY ? 0.f : m_used;
#pragma unroll
                for (int cc = 0; cc < kCols / 8; ++cc) {
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p0 = tc::ex2(x[cc * 8 + 2 * e] - mu);
                        const float p1 = tc::ex2(x[cc * 8 + 2 * e + 1] - mu);
                        sum += p0 + p1;
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                    const int blk = cc >> 3, ch = cc & 7;
                    uint4 *dst = reinterpret_cast<uint4 *>(sP + blk * kBlk + r * 128 + ((ch ^ (r & 7)) << 4));
                    *dst = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                l += sum;
                tc::fence_proxy_async();
                tc::fence_before();
                arrive(&bars.p_full);
            }
            if (!ok) break;
            // epilogue: O / l once the last PV of this tile is done
            __nv_bfloat16 *orow = a.out + qrow * kD;
            if (n_kv > 0) {
                ok = wait_bar(&bars.o_done, (unsigned)((g - 1) & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t v[32];
                    tc::tmem_ld32(tO + lane_off + c * 32, v);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 pk;
                        pk.x = pack_bf16x2(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
                        pk.y = pack_bf16x2(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv);
                        pk.z = pack_bf16x2(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv);
                        pk.w = pack_bf16x2(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + c * 32 + e) = pk;
                    }
                }
                tc::fence_before();
                arrive(&bars.o_free);
            } else {
                for (int c = 0; c < kD; c += 8) *reinterpret_cast<uint4 *>(orow + c) = make_uint4(0, 0, 0, 0);
                arrive(&bars.o_free);  // keeps the per-tile phases of o_free aligned
            }
            if (a.lse) a.lse[qrow] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
        }
        if (!ok) s_abort = 1;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

constexpr size_t kSmemBytes = 1024 + 6 * (size_t)kTileBytes;

}  // namespace

bool make_tmap_bf16(CUtensorMap *tm, const void *base, int rank, const uint64_t *dims, const uint64_t *strides_elems,
                    uint32_t box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    cuuint64_t gdim[3], gstride[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) gdim[i] = dims[i];
    for (int i = 0; i + 1 < rank; ++i) gstride[i] = strides_elems[i] * 2;  // bytes, dims 1..rank-1
    box[0] = 64;
    box[1] = box_rows;
    box[2] = 1;
    const CUresult r = encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), gdim,
                              gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool prefill_tc_supported(const AttnArgs &a) {
    return a.d == kD && !a.idx && ((int64_t)a.T * a.H) % kRows == 0 && a.rows > 0;
}

cudaError_t launch_attn_prefill_tc(const AttnArgs &a, int num_sms, cudaStream_t s) {
    const int B = a.rows / a.T;
    CUtensorMap tq, tkc, tvc, tkr, tvr;
    {
        const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)a.rows * a.H};
        const uint64_t str[1] = {(uint64_t)kD};
        if (!make_tmap_bf16(&tq, a.q, 2, dims, str, kRows)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.E_cap, (uint64_t)B};
        const uint64_t str[2] = {(uint64_t)a.c_se, (uint64_t)a.c_sb};
        if (!make_tmap_bf16(&tkc, a.kc, 3, dims, str, kCols)) return cudaErrorInvalidValue;
        if (!make_tmap_bf16(&tvc, a.vc, 3, dims, str, kCols)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.N_cap, (uint64_t)B};
        const uint64_t str[2] = {(uint64_t)a.r_st, (uint64_t)a.r_sb};
        if (!make_tmap_bf16(&tkr, a.k_raw, 3, dims, str, kCols)) return cudaErrorInvalidValue;
        if (!make_tmap_bf16(&tvr, a.v_raw, 3, dims, str, kCols)) return cudaErrorInvalidValue;
    }
    PrefillTcArgs p;
    p.B = B;
    p.T = a.T;
    p.H = a.H;
    p.m = a.m;
    p.window = a.window;
    p.E_cap = a.E_cap;
    p.N_cap = a.N_cap;
    p.q_pos0 = a.pos;
    p.scale_log2 = a.scale * kLog2e;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.lse = a.lse;
    p.n_qtiles = (int)(((int64_t)a.rows * a.H) / kRows);
    static unsigned long long done = 0;
    cudaError_t e = smem_limit_once(attn_prefill_tc_kernel, (int)kSmemBytes, done);
    if (e != cudaSuccess) return e;
    const int grid = p.n_qtiles < num_sms ? p.n_qtiles : num_sms;
    attn_prefill_tc_kernel<<<grid, 192, kSmemBytes, s>>>(tq, tkc, tvc, tkr, tvr, p);
    return cudaGetLastError();
}

}  // namespace hsa
