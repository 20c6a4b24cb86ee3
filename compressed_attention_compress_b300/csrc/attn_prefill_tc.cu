// Prefill attention over all compressed entries plus the window (HCA layer) on
// the 5th-generation tensor cores: tcgen05 MMAs with TMEM accumulators, operands
// brought in by TMA.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制: HCA runs dense attention over
// every heavily compressed entry; the sliding-window paragraph adds the most
// recent raw tokens to the same softmax; strict causality limits query p to the
// E(p) = floor((p+1)/m) complete blocks.
//
// Queries are the rows of q viewed as [B*T*H, d] (d = 128); a query tile is 128
// rows, i.e. 128/H consecutive tokens with all their heads (one KV head).  A CTA
// takes a pair of consecutive query tiles (A, B) of one sequence and walks one
// KV sequence for both: ceil(E(p_last)/128) entry tiles of Kc/Vc, then the raw
// window tokens [p_first - W + 1, p_last] in 128-token tiles; per-row masks
// apply each row's E(p) and window.  One persistent CTA per SM; its warps
// specialise:
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: one query row
//              per thread.  S comes from TMEM; P (bf16) goes back into the
//              first 64 columns of the same TMEM buffer and is the A operand of
//              the PV MMA; O is rescaled in TMEM only when a row's running max
//              grows by more than 2^8 (until then the stale max keeps P <= 256).
//   warp 8     MMA issuer (one thread), in the order
//                S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//              so that while one tile's softmax runs the tensor core works on
//              the other tile; completion via tcgen05.commit.
//   warp 9     TMA producer (one thread): both Q tiles, then K_0, V_0, K_1, V_1,
//              ... through a 4-slot ring of 32 KiB shared-memory tiles (only K_j
//              when one buffer is both K and V, V4's shared key/value entry).
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
constexpr int kTileBytes = kRows * kD * 2;     // 32 KiB (two 128-byte-wide column blocks)
constexpr int kBlk = kRows * 128;              // 16 KiB per 64-element block
constexpr int kRing = 4;                       // K/V tile slots
constexpr int kSoftWarps = 8;
constexpr int kThreadsTc = (kSoftWarps + 2) * 32;
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
    int tiles_per_seq, pairs_per_seq, n_pairs;
    int shared_kv;  // one buffer is both K and V: each item tile is loaded once
};

struct __align__(8) Bars {
    uint64_t q_full, q_empty;
    uint64_t kv_full[kRing], kv_empty[kRing];
    uint64_t s_full[2], p_full[2], o_done[2], o_free[2];  // per query tile (A, B)
    uint64_t mma_fin;
};

struct PairInfo {
    int b;
    int64_t tile0;     // global index of tile A
    bool has_b;        // tile B exists (a sequence may have an odd number of tiles)
    int n_ent, n_win;  // entry tiles, window tiles
    int64_t w0;        // first raw token of the window range
};

__device__ __forceinline__ PairInfo pair_info(const PrefillTcArgs &a, int pr) {
    PairInfo pi;
    pi.b = pr / a.pairs_per_seq;
    const int lp = pr - pi.b * a.pairs_per_seq;
    const int t_in = 2 * lp;  // tile index within the sequence
    pi.tile0 = (int64_t)pi.b * a.tiles_per_seq + t_in;
    pi.has_b = t_in + 1 < a.tiles_per_seq;
    const int64_t r0 = (int64_t)t_in * kRows;                        // first row within the sequence
    const int64_t r1 = r0 + (pi.has_b ? 2 : 1) * (int64_t)kRows - 1;  // last row
    const int64_t p0 = a.q_pos0[pi.b];
    const int64_t p_first = p0 + r0 / a.H, p_last = p0 + r1 / a.H;
    int64_t E = num_entries(p_last, a.m);
    if (E > a.E_cap) E = a.E_cap;
    pi.n_ent = (int)((E + kCols - 1) / kCols);
    pi.w0 = p_first - a.window + 1;
    const int64_t span = a.window > 0 ? p_last - pi.w0 + 1 : 0;
    pi.n_win = (int)((span + kCols - 1) / kCols);
    return pi;
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

// D (+)= A B with A [128 x 16] in TMEM (lane = row, bf16 pairs along the columns)
// and B described in shared memory.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Two fp32 operations in one packed instruction (lanes: low and high 32 bits).
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t x, uint64_t y, uint64_t z) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(x), "l"(y), "l"(z));
    return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t x, uint64_t y) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(x), "l"(y));
    return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo_of(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_of(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

__global__ void __launch_bounds__(kThreadsTc, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                           const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kr,
                           const __grid_constant__ CUtensorMap tm_vr, PrefillTcArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];  // rounded up to 1024 below, at run time
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *sQ = smem;                        // tiles A, B: 2 x 32 KiB
    unsigned char *sKV = smem + 2 * kTileBytes;      // kRing x 32 KiB (K_0, V_0, K_1, V_1, ...)
    __shared__ Bars bars;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bars.kv_full[i], 1);
            mbar_init(&bars.kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.p_full[i], kRows);
            mbar_init(&bars.o_done[i], 1);
            mbar_init(&bars.o_free[i], kRows);
        }
        mbar_init(&bars.mma_fin, 1);
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    // per tile X: S_X (fp32, 128 columns; P_X bf16 pairs overwrite its first 64) and O_X
    const uint32_t tS[2] = {tmem, tmem + 256};
    const uint32_t tO[2] = {tmem + 128, tmem + 384};

    if (warp == kSoftWarps + 1) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int it = 0, q_issued = 0;
            int64_t u = 0;  // K/V loads issued
            bool ok = true;
            for (int pr = blockIdx.x; pr < a.n_pairs && ok; pr += gridDim.x, ++it) {
                const PairInfo pi = pair_info(a, pr);
                if (it > 0) ok = wait_bar(&bars.q_empty, (unsigned)((it - 1) & 1), &s_abort);
                if (!ok) break;
                mbar_expect_tx(&bars.q_full, (pi.has_b ? 2 : 1) * kTileBytes);
                for (int x = 0; x < (pi.has_b ? 2 : 1); ++x) {
                    const int y = (int)((pi.tile0 + x) * kRows);
                    tc::tma_load_2d(sQ + x * kTileBytes, &tm_q, 0, y, &bars.q_full);
                    tc::tma_load_2d(sQ + x * kTileBytes + kBlk, &tm_q, 64, y, &bars.q_full);
                }
                ++q_issued;
                const int n_kv = pi.n_ent + pi.n_win;
                for (int j = 0; j < n_kv && ok; ++j) {
                    for (int kv = 0; kv < (a.shared_kv ? 1 : 2) && ok; ++kv, ++u) {
                        const int slot = (int)(u % kRing);
                        if (u >= kRing) ok = wait_bar(&bars.kv_empty[slot], (unsigned)(((u / kRing) - 1) & 1), &s_abort);
                        if (!ok) break;
                        unsigned char *dst = sKV + slot * kTileBytes;
                        mbar_expect_tx(&bars.kv_full[slot], kTileBytes);
                        const CUtensorMap *tm;
                        int y;
                        if (j < pi.n_ent) {
                            tm = kv ? &tm_vc : &tm_kc;
                            y = j * kCols;
                        } else {
                            tm = kv ? &tm_vr : &tm_kr;
                            y = (int)(pi.w0 + (int64_t)(j - pi.n_ent) * kCols);
                        }
                        tc::tma_load_3d(dst, tm, 0, y, pi.b, &bars.kv_full[slot]);
                        tc::tma_load_3d(dst + kBlk, tm, 64, y, pi.b, &bars.kv_full[slot]);
                    }
                }
            }
            if (!ok) s_abort = 1;
            // let every copy this thread issued land before the CTA can exit
            volatile int never = 0;
            if (q_issued > 0) wait_bar(&bars.q_full, (unsigned)((q_issued - 1) & 1), &never);
            for (int64_t v = (u > kRing ? u - kRing : 0); v < u; ++v)
                wait_bar(&bars.kv_full[v % kRing], (unsigned)((v / kRing) & 1), &never);
        }
    } else if (warp == kSoftWarps) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_bf16(kRows, kCols, false, false);
            constexpr uint32_t idO = tc::idesc_bf16(kRows, kD, false, true);
            int it = 0;
            int g[2] = {0, 0};        // steps done per tile (s_full / p_full / o_done uses)
            int pairs_x[2] = {0, 0};  // non-empty pairs per tile (o_free uses)
            int64_t u = 0;            // K/V tiles consumed
            bool ok = true;
            auto wait_kv = [&](int64_t uu) -> uint32_t {
                const int slot = (int)(uu % kRing);
                ok = ok && wait_bar(&bars.kv_full[slot], (unsigned)((uu / kRing) & 1), &s_abort);
                return smem_u32(sKV + slot * kTileBytes);
            };
            auto issue_s = [&](int x, uint32_t aK) {
                const uint32_t aQ = smem_u32(sQ + x * kTileBytes);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t da = tc::desc_sw128(aQ + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
                    const uint64_t db = tc::desc_sw128(aK + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
                    tc::mma_bf16(tS[x], da, db, idS, kk > 0 ? 1u : 0u);
                }
                tc::commit(&bars.s_full[x]);
            };
            auto issue_pv = [&](int x, uint32_t aV, bool first) {
                // O_X (+)= P_X V : P_X from TMEM (64 columns of bf16 pairs), V MN-major in smem
#pragma unroll
                for (int kk = 0; kk < kCols / 16; ++kk) {
                    const uint64_t db = tc::desc_sw128(aV + kk * 16 * 128, kBlk, 1024);
                    mma_bf16_tmem_a(tO[x], tS[x] + kk * 8, db, idO, (first && kk == 0) ? 0u : 1u);
                }
                tc::commit(&bars.o_done[x]);
            };
            for (int pr = blockIdx.x; pr < a.n_pairs && ok; pr += gridDim.x, ++it) {
                const PairInfo pi = pair_info(a, pr);
                const int nx = pi.has_b ? 2 : 1;
                const int n_kv = pi.n_ent + pi.n_win;
                ok = wait_bar(&bars.q_full, (unsigned)(it & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                if (n_kv == 0) {
                    tc::commit(&bars.q_empty);
                    continue;
                }
                // S_X(0) for both tiles
                uint32_t aK = wait_kv(u);
                int64_t uk = u++;
                if (!ok) break;
                tc::fence_after();
                for (int x = 0; x < nx; ++x) issue_s(x, aK);
                if (!a.shared_kv) tc::commit(&bars.kv_empty[uk % kRing]);  // shared: K_0 is also V_0
                for (int j = 0; j < n_kv && ok; ++j) {
                    // V_j: its own tile, or K_j itself when one buffer is both
                    uint32_t aV = aK;
                    int64_t uv = uk;
                    if (!a.shared_kv) {
                        aV = wait_kv(u);
                        uv = u++;
                    }
                    for (int x = 0; x < nx && ok; ++x) {
                        ok = wait_bar(&bars.p_full[x], (unsigned)(g[x] & 1), &s_abort);
                        if (ok && j == 0 && pairs_x[x] > 0)
                            ok = wait_bar(&bars.o_free[x], (unsigned)((pairs_x[x] - 1) & 1), &s_abort);
                        if (!ok) break;
                        tc::fence_after();
                        issue_pv(x, aV, j == 0);
                        ++g[x];
                        if (x == nx - 1) tc::commit(&bars.kv_empty[uv % kRing]);
                        if (j + 1 < n_kv) {
                            if (x == 0) {
                                aK = wait_kv(u);
                                uk = u++;
                                if (!ok) break;
                                tc::fence_after();
                            }
                            issue_s(x, aK);
                            if (x == nx - 1 && !a.shared_kv) tc::commit(&bars.kv_empty[uk % kRing]);
                        }
                    }
                }
                tc::commit(&bars.q_empty);
                for (int x = 0; x < nx; ++x) ++pairs_x[x];
            }
            if (!ok) s_abort = 1;
            // every MMA this thread issued completes before TMEM is released
            tc::commit(&bars.mma_fin);
            volatile int never = 0;
            wait_bar(&bars.mma_fin, 0u, &never);
        }
    } else {
        // ---------------------------------------------------------- softmax rows
        const int x = warp >> 2;                    // query tile of this warpgroup
        const int r = (warp & 3) * 32 + lane;       // row in the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint64_t sc2 = pack2(a.scale_log2, a.scale_log2);
        int g = 0, pairs_done = 0;
        bool ok = true;
        for (int pr = blockIdx.x; pr < a.n_pairs && ok; pr += gridDim.x) {
            const PairInfo pi = pair_info(a, pr);
            if (x == 1 && !pi.has_b) continue;
            const int n_kv = pi.n_ent + pi.n_win;
            const int64_t qrow = (pi.tile0 + x) * kRows + r;                  // global query row
            const int64_t rin = qrow - (int64_t)pi.b * a.tiles_per_seq * kRows;  // row within the sequence
            const int64_t p = a.q_pos0[pi.b] + rin / a.H;
            int64_t E = num_entries(p, a.m);
            if (E > a.E_cap) E = a.E_cap;
            const int64_t wlo = (p - a.window + 1) < 0 ? 0 : p - a.window + 1;
            const int64_t whi = p < a.N_cap ? p : a.N_cap - 1;  // the raw cache must hold the query
            if (p >= a.N_cap && a.window > 0) raise_flag(FLAG_ATTN_RANGE);
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < n_kv && ok; ++j, ++g) {
                ok = wait_bar(&bars.s_full[x], (unsigned)(g & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                // pass 1 over S_X: masked raw maximum (eight independent chains), 64
                // columns at a time; the scale (> 0) goes into the exponent in pass 2.
                // Only tiles reaching past some row's visible range need the mask.
                const bool ent = j < pi.n_ent;
                const int64_t base = ent ? (int64_t)j * kCols : pi.w0 + (int64_t)(j - pi.n_ent) * kCols;
                const bool masked = !ent || !__all_sync(0xffffffffu, base + kCols <= E);
                auto visible = [&](int c) {
                    const int64_t t = base + c;
                    return ent ? t < E : (t >= wlo && t <= whi);
                };
                float mx8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) mx8[q] = -INFINITY;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t v[64];
                    tc::tmem_ld32(tS[x] + lane_off + hf * 64, v);
                    tc::tmem_ld32(tS[x] + lane_off + hf * 64 + 32, v + 32);
                    tc::tmem_wait_ld();
                    if (masked) {
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            mx8[c & 7] = fmaxf(mx8[c & 7], visible(hf * 64 + c) ? __uint_as_float(v[c]) : -INFINITY);
                    } else {
#pragma unroll
                        for (int c = 0; c < 64; c += 2)
                            mx8[(c >> 1) & 7] =
                                tc::fmax3(mx8[(c >> 1) & 7], __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
                    }
                }
                const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) *
                                 a.scale_log2;
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
                    // O_X changes only once the previous PV has completed (the next one
                    // needs this step's P, not written yet)
                    ok = wait_bar(&bars.o_done[x], (unsigned)((g - 1) & 1), &s_abort);
                    if (!ok) break;
                    tc::fence_after();
#pragma unroll
                    for (int c = 0; c < kD / 32; ++c) {
                        uint32_t v[32];
                        tc::tmem_ld32(tO[x] + lane_off + c * 32, v);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tc::tmem_st32(tO[x] + lane_off + c * 32, v);
                    }
                }
                // pass 2: P = 2^(x * scale_log2 - m_used) as bf16 pairs into the first 64
                // columns of S_X; columns 64h..64h+63 are read before P words 32h..32h+31
                // are written over columns already read
                const float nmu = m_used == -INFINITY ? 0.f : -m_used;
                const uint64_t nmu2 = pack2(nmu, nmu);
                uint64_t acc2[4] = {0, 0, 0, 0};
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t v[64];
                    tc::tmem_ld32(tS[x] + lane_off + hf * 64, v);
                    tc::tmem_ld32(tS[x] + lane_off + hf * 64 + 32, v + 32);
                    tc::tmem_wait_ld();
                    if (masked) {
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (!visible(hf * 64 + c)) v[c] = __float_as_uint(-INFINITY);
                    }
                    uint32_t pw[32];
#pragma unroll
                    for (int w = 0; w < 32; ++w) {
                        const uint64_t arg = fma_f32x2(((uint64_t)v[2 * w + 1] << 32) | v[2 * w], sc2, nmu2);
                        const float p0 = tc::ex2(lo_of(arg)), p1 = tc::ex2(hi_of(arg));
                        acc2[w & 3] = add_f32x2(acc2[w & 3], pack2(p0, p1));
                        pw[w] = pack_bf16x2(p0, p1);
                    }
                    tc::tmem_st32(tS[x] + lane_off + hf * 32, pw);
                }
                const uint64_t s01 = add_f32x2(acc2[0], acc2[1]), s23 = add_f32x2(acc2[2], acc2[3]);
                const uint64_t s4 = add_f32x2(s01, s23);
                l += lo_of(s4) + hi_of(s4);
                tc::tmem_wait_st();
                tc::fence_before();
                arrive(&bars.p_full[x]);
            }
            if (!ok) break;
            // epilogue: O / l once the last PV of this tile is done
            __nv_bfloat16 *orow = a.out + qrow * kD;
            if (n_kv > 0) {
                ok = wait_bar(&bars.o_done[x], (unsigned)((g - 1) & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t v[32];
                    tc::tmem_ld32(tO[x] + lane_off + c * 32, v);
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
                arrive(&bars.o_free[x]);
                ++pairs_done;
            } else {
                for (int c = 0; c < kD; c += 8) *reinterpret_cast<uint4 *>(orow + c) = make_uint4(0, 0, 0, 0);
            }
            if (a.lse) a.lse[qrow] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
        }
        (void)pairs_done;
        if (!ok) s_abort = 1;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

constexpr size_t kSmemBytes = 1024 + (2 + kRing) * (size_t)kTileBytes;  // Q_A, Q_B, K/V ring

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
    p.tiles_per_seq = (int)(((int64_t)a.T * a.H) / kRows);
    p.pairs_per_seq = (p.tiles_per_seq + 1) / 2;
    p.n_pairs = B * p.pairs_per_seq;
    p.shared_kv = a.shared_kv;
    static unsigned long long done = 0;
    cudaError_t e = smem_limit_once(attn_prefill_tc_kernel, (int)kSmemBytes, done);
    if (e != cudaSuccess) return e;
    const int grid = p.n_pairs < num_sms ? p.n_pairs : num_sms;
    attn_prefill_tc_kernel<<<grid, kThreadsTc, kSmemBytes, s>>>(tq, tkc, tvc, tkr, tvr, p);
    return cudaGetLastError();
}

}  // namespace hsa
