// Prefill attention over each query token's own selected entries plus its window
// (CSA layer) on the 5th-generation tensor cores.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制: CSA step 3 runs
// Multi-Query Attention over the top-k compressed entries the indexer selected for
// the query token; the sliding-window paragraph adds the most recent raw tokens to
// the same softmax.
//
// Every query token has its own item set, shared by its H = 64 heads, so a token is
// an M = 64 (heads) problem: S = Q K_j^T (N = 128 items per tile, K = d = 128) and
// O += P V_j, with S and O in TMEM (row h of an M = 64 accumulator lives in TMEM
// lane (h / 16) * 32 + h % 16).  One persistent CTA per SM walks tokens:
//   warps 0-3  softmax, two lanes per head (lane l < 16 and l + 16 of warp w take
//              halves of head 16w + l's row): S from TMEM into registers, masked
//              maximum, exponents, P (bf16) into shared memory for the second MMA,
//              O rescaled in TMEM only when the maximum grows by > 2^8.
//   gather     resolve each item row of tile j (selected entry of Kc/Vc or window
//              token of the raw cache; invalid rows are zero) and copy it into a
//              5-slot ring of 32 KiB 128-byte-swizzled tiles; a 128-bit validity
//              mask per tile goes to a small ring of its own.  Where the caches can
//              be viewed as 2-D tensors of rows, warps 4-7 copy K rows by the
//              tensor-memory-access unit, four rows per `cp.async.bulk.tensor`
//              `tile::gather4` instruction (one per 64-column half, tensor maps one
//              row high), and warps 8-10 copy V rows by 16-byte `cp.async`, so the
//              two engines work in parallel; otherwise warps 4-7 copy both by
//              `cp.async`.  The first gather thread also loads each token's Q by TMA.
//   last warp  MMA issuer (one thread): S(g) into one of two TMEM buffers, then
//              O += P(g-1) V(g-1) (g counted over all the CTA's tokens); completion via
//              tcgen05.commit.
// All waits are bounded; a wait that gives up raises the device flag and the CTA
// stops issuing work.
#include <math.h>

#include <cudaTypedefs.h>

#include "internal.h"
#include "tc_common.cuh"

namespace hsa {

namespace {

constexpr int kH = 64;        // heads = MMA M
constexpr int kD = 128;       // head dim
constexpr int kN = 128;       // items per tile
constexpr int kQBytes = kH * kD * 2;       // 16 KiB
constexpr int kQBlk = kH * 128;            // 8 KiB per 64-column block of Q or P
constexpr int kTile = kN * kD * 2;         // 32 KiB K or V tile
constexpr int kTBlk = kN * 128;            // 16 KiB per 64-column block of a tile
constexpr int kRing = 5;
constexpr int kMaskRing = 8;
constexpr int kSoftWarps = 4, kGatherWarps = 4;
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kKWarps = 4, kVWarps = 3;  // tile::gather4 variant: K-copy and V-copy warps
// warps: softmax, gather (4, or 4 K + 3 V), MMA issuer
template <bool kTma>
constexpr int kThreadsOf = (kSoftWarps + (kTma ? kKWarps + kVWarps : kGatherWarps) + 1) * 32;
template <bool kTma>
constexpr int kMmaWarpOf = kSoftWarps + (kTma ? kKWarps + kVWarps : kGatherWarps);
constexpr int kLag = 3;       // cp.async groups a gather thread keeps in flight: the MMA takes
                              // K_{g+1} before releasing V_g, so kLag <= kRing - 2 keeps the ring live
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;
constexpr unsigned long long kWaitLimit = 1ull << 24;

struct __align__(8) Bars {
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[kRing], kv_empty[kRing];
    uint64_t m_full[kMaskRing], m_empty[kMaskRing];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, o_done, o_free, mma_fin;
};

struct GatherArgs {
    int rows, T, topk, window, m, n_tiles;
    int64_t E_cap, N_cap, c_sb, c_se, r_sb, r_st;
    int64_t c_rows_b, r_rows_b;  // row-coordinate step per sequence of the 2-D cache views (c_sb / c_se, r_sb / r_st)
    const int64_t *q_pos0;
    const int32_t *idx, *cnt;
    const __nv_bfloat16 *kc, *vc, *k_raw, *v_raw;
    float scale_log2;
    __nv_bfloat16 *out;
    float *lse;
};

__device__ __forceinline__ bool wait_bar(uint64_t *bar, unsigned parity, volatile int *abort) {
    for (unsigned long long i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    raise_flag(FLAG_ATTN_RANGE | 0x800u);
    *abort = 1;
    return false;
}
__device__ __forceinline__ void arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void arrive2(uint64_t *bar) {  // two arrivals at once
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], 2;\n" ::"r"(smem_u32(bar)) : "memory");
}
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
// Four rows (r0..r3) of a 2-D tensor, columns [x, x + box width), into 4 consecutive
// box rows at dst, counted in bytes on bar.
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *tm, int x, int r0, int r1, int r2, int r3,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], "
        "[%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(smem_u32(dst)),
        "l"(tm), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
        : "memory");
}
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// kTma: rows by tile::gather4 (tm_kc, tm_vc, tm_kr, tm_vr: the caches as 2-D tensors of
// d-wide rows, boxes of 64 columns x 1 row); otherwise by cp.async (those maps unused).
template <bool kTma>
__global__ void __launch_bounds__(kThreadsOf<kTma>, 1)
    attn_gather_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                          const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kr,
                          const __grid_constant__ CUtensorMap tm_vr, GatherArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];  // rounded up to 1024 at run time
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *sQ = smem;                          // 2 x 16 KiB
    unsigned char *sRing = smem + 2 * kQBytes;         // kRing x 32 KiB
    unsigned char *sP = sRing + kRing * kTile;         // 16 KiB
    __shared__ Bars bars;
    __shared__ uint32_t s_mask[kMaskRing][4];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.q_full[i], 1);
            mbar_init(&bars.q_empty[i], 1);
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.s_free[i], kSoftWarps * 32);
        }
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bars.kv_full[i], kGatherThreads);
            mbar_init(&bars.kv_empty[i], 1);
        }
        for (int i = 0; i < kMaskRing; ++i) {
            mbar_init(&bars.m_full[i], kTma ? kKWarps : kGatherWarps);
            mbar_init(&bars.m_empty[i], kSoftWarps * 32);
        }
        mbar_init(&bars.p_full, kSoftWarps * 32);
        mbar_init(&bars.o_done, 1);
        mbar_init(&bars.o_free, kSoftWarps * 32);
        mbar_init(&bars.mma_fin, 1);
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    auto tS = [tmem](int64_t gg) -> uint32_t { return tmem + (uint32_t)(gg & 1) * 128u; };  // S double buffer
    const uint32_t tO = tmem + 256;
    const int nt = a.n_tiles;

    if (kTma && warp >= kSoftWarps && warp < kMmaWarpOf<kTma>) {
        // ------------------------------------------------------ gather (two engines)
        // Warps 4-7 copy K tiles with tile::gather4 (the tensor-memory-access unit; a warp's
        // gather4 lanes issue one after another, so four warps share the K rows), warps 8-10
        // copy V tiles with cp.async (the load/store unit), so the two engines work in
        // parallel.  Each group resolves the rows it copies itself, so the groups only meet
        // at the ring's barriers: K warp w takes row 32w + t (and publishes the tile's
        // validity word w); V warp w takes the row pairs (2i, 2i + 1) with i ≡ w (mod 3), lane t
        // resolving the t-th and (32 + t)-th row of its list.  Groups of 4 rows go to one
        // gather4: an invalid row copies a valid row of its group (its logits are masked, so
        // it adds nothing), a group with no valid row is zeroed instead; valid rows of one
        // group share a cache because topk is a multiple of 4.
        const int gw = warp - kSoftWarps;
        const bool k_role = gw < kKWarps;
        const int w2 = k_role ? gw : gw - kKWarps;
        const int n_pairs = (64 - w2 + kVWarps - 1) / kVWarps;  // V warp: row pairs it copies
        auto v_row = [&](int q) {  // q-th row of a V warp's list (127 past its end: never copied)
            return (q >> 1) < n_pairs ? 2 * (w2 + kVWarps * (q >> 1)) + (q & 1) : 127;
        };
        const int R1 = k_role ? 32 * w2 + lane : v_row(lane), R2 = k_role ? 0 : v_row(32 + lane);
        int it = 0;
        int64_t g = 0;  // item tiles
        bool ok = true;
        // slot i of the row's list: the selected entry or window token, its address (V), its row
        // coordinate in the 2-D view of its cache and which cache (K); false when invalid
        auto resolve = [&](int b, int64_t p, int64_t E, int slot_i, int32_t e, const __nv_bfloat16 *&vp, int &crd,
                           int &raw) -> bool {
            vp = nullptr;
            crd = 0;
            raw = 0;
            if (slot_i < a.topk) {
                if (e >= E) raise_flag(FLAG_ATTN_INDEX);
                if (e >= 0 && e < E) {
                    vp = a.vc + b * a.c_sb + (int64_t)e * a.c_se;
                    crd = (int)(b * a.c_rows_b + e);
                    return true;
                }
            } else if (slot_i < a.topk + a.window) {
                const int64_t tr = p - a.window + 1 + (slot_i - a.topk);
                if (tr >= 0 && tr <= p) {
                    if (tr >= a.N_cap) {
                        raise_flag(FLAG_ATTN_RANGE);
                    } else {
                        vp = a.v_raw + b * a.r_sb + tr * a.r_st;
                        crd = (int)(b * a.r_rows_b + tr);
                        raw = 1;
                        return true;
                    }
                }
            }
            return false;
        };
        // the four row coordinates of this lane's group (lanes 4q..4q+3), invalid rows replaced
        auto group = [&](bool v, int crd, int raw, int (&c4)[4], int &graw) -> uint32_t {
            const uint32_t bits = __ballot_sync(0xffffffffu, v);
            const uint32_t gb = (bits >> (lane & ~3)) & 0xFu;
            const int src = (lane & ~3) + (gb ? __ffs(gb) - 1 : 0);
            const int sc = __shfl_sync(0xffffffffu, crd, src);
            graw = __shfl_sync(0xffffffffu, raw, src);
            const int mine = v ? crd : sc;
#pragma unroll
            for (int i = 0; i < 4; ++i) c4[i] = __shfl_sync(0xffffffffu, mine, (lane & ~3) + i);
            return gb;
        };
        for (int row = blockIdx.x; row < a.rows && ok; row += gridDim.x, ++it) {
            const int b = row / a.T, t = row - (row / a.T) * a.T;
            const int64_t p = a.q_pos0[b] + t;
            int64_t E = num_entries(p, a.m);
            if (E > a.E_cap) E = a.E_cap;
            const int cntr = a.cnt ? min(max(a.cnt[row], 0), a.topk) : a.topk;
            if (gw == 0 && lane == 0) {
                if (it >= 2) ok = wait_bar(&bars.q_empty[it & 1], (unsigned)(((it >> 1) - 1) & 1), &s_abort);
                if (ok) {
                    mbar_expect_tx(&bars.q_full[it & 1], kQBytes);
                    tc::tma_load_2d(sQ + (it & 1) * kQBytes, &tm_q, 0, row * kH, &bars.q_full[it & 1]);
                    tc::tma_load_2d(sQ + (it & 1) * kQBytes + kQBlk, &tm_q, 64, row * kH, &bars.q_full[it & 1]);
                }
            }
            ok = __all_sync(0xffffffffu, ok);
            auto sel = [&](int slot_i) -> int32_t {
                return (slot_i < a.topk && slot_i < cntr) ? a.idx[(int64_t)row * a.topk + slot_i] : -1;
            };
            // selected indices one tile ahead, so each load's round trip overlaps the copies
            int32_t n1 = sel(R1), n2 = k_role ? -1 : sel(R2);
            for (int j = 0; j < nt && ok; ++j, ++g) {
                const int s1 = j * kN + R1, s2 = j * kN + R2;
                const int32_t e1 = n1, e2 = n2;
                n1 = sel(s1 + kN);
                if (!k_role) n2 = sel(s2 + kN);
                const __nv_bfloat16 *vp1, *vp2 = nullptr;
                int crd1, raw1, crd2 = 0, raw2 = 0;
                const bool v1 = resolve(b, p, E, s1, e1, vp1, crd1, raw1);
                const bool v2 = k_role ? false : resolve(b, p, E, s2, e2, vp2, crd2, raw2);
                if (k_role) {
                    int c4a[4], graw1;
                    const uint32_t gb1 = group(v1, crd1, raw1, c4a, graw1);
                    // validity word w of the tile (rows 32w..32w + 31)
                    const uint32_t bits = __ballot_sync(0xffffffffu, v1);
                    const int ms = (int)(g % kMaskRing);
                    if (g >= kMaskRing)
                        ok = wait_bar(&bars.m_empty[ms], (unsigned)(((g / kMaskRing) - 1) & 1), &s_abort);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    if (lane == 0) {
                        s_mask[ms][w2] = bits;
                        arrive(&bars.m_full[ms]);
                    }
                    const int64_t uk = 2 * g;
                    const int sk = (int)(uk % kRing);
                    if (uk >= kRing) ok = wait_bar(&bars.kv_empty[sk], (unsigned)(((uk / kRing) - 1) & 1), &s_abort);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    unsigned char *dK = sRing + sk * kTile;
                    if (gb1 == 0) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            *reinterpret_cast<uint4 *>(dK + R1 * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4 *>(dK + kTBlk + R1 * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                        }
                        tc::fence_proxy_async();  // generic zeros before the MMA reads the tile
                    }
                    const uint32_t l1 = __ballot_sync(0xffffffffu, (lane & 3) == 0 && gb1 != 0);
                    __syncwarp();
                    // one arrival per K thread; lane 0 of each warp brings that warp's bytes
                    // before the warp's copies issue
                    if (lane == 0) mbar_expect_tx(&bars.kv_full[sk], (unsigned)__popc(l1) * 1024u);
                    else arrive(&bars.kv_full[sk]);
                    __syncwarp();
                    if ((l1 >> lane) & 1u) {
                        const CUtensorMap *tm = graw1 ? &tm_kr : &tm_kc;
                        tma_gather4(dK + R1 * 128, tm, 0, c4a[0], c4a[1], c4a[2], c4a[3], &bars.kv_full[sk]);
                        tma_gather4(dK + kTBlk + R1 * 128, tm, 64, c4a[0], c4a[1], c4a[2], c4a[3], &bars.kv_full[sk]);
                    }
                } else {
                    (void)v1;
                    (void)v2;
                    const int64_t uv = 2 * g + 1;
                    const int sv = (int)(uv % kRing);
                    if (uv >= kRing) ok = wait_bar(&bars.kv_empty[sv], (unsigned)(((uv / kRing) - 1) & 1), &s_abort);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    // a half-warp copies one 256-byte row (lane l: 16-byte chunk l % 16), two
                    // rows per instruction; row pointers come by shuffle from the resolving lane
                    unsigned char *dV = sRing + sv * kTile;
                    const unsigned long long a1 = reinterpret_cast<unsigned long long>(vp1);
                    const unsigned long long a2 = reinterpret_cast<unsigned long long>(vp2);
                    const int c = lane & 15;
#pragma unroll 4
                    for (int k = 0; k < n_pairs; ++k) {
                        const int q = 2 * k + (lane >> 4);  // position in this warp's row list
                        const unsigned long long rs = __shfl_sync(0xffffffffu, 2 * k < 32 ? a1 : a2, q & 31);
                        const int rr = 2 * (w2 + kVWarps * k) + (lane >> 4);  // row within the tile
                        const uint32_t off = (uint32_t)((c >> 3) * kTBlk + rr * 128 + (((c & 7) ^ (rr & 7)) << 4));
                        const __nv_bfloat16 *rp = reinterpret_cast<const __nv_bfloat16 *>(rs);
                        cp_async_16(smem_u32(dV + off), rp ? (const void *)(rp + c * 8) : (const void *)a.vc,
                                    rp ? 16 : 0);  // zero-fill invalid rows
                    }
                    cp_async_commit();
                    // the previous tile's V has landed once at most this tile's copies are pending
                    // (the barrier counts 128 arrivals: one per thread of V warps 0-1, two per
                    // thread of V warp 2)
                    if (g > 0) {
                        cp_wait<1>();
                        tc::fence_proxy_async();
                        if (w2 == 2) arrive2(&bars.kv_full[(uv - 2) % kRing]);
                        else arrive(&bars.kv_full[(uv - 2) % kRing]);
                    }
                }
            }
        }
        if (!ok) s_abort = 1;
        if (k_role) {
            // the last two K tiles' slots are not reused: their copies land before the CTA exits
            // (normally the MMA has already consumed them)
            if (lane == 0) {
                volatile int never = 0;
                for (int64_t h = (g > 2 ? g - 2 : 0); h < g; ++h)
                    wait_bar(&bars.kv_full[(2 * h) % kRing], (unsigned)(((2 * h) / kRing) & 1), &never);
            }
            if (gw == 0 && lane == 0 && it > 0) {
                volatile int never = 0;
                wait_bar(&bars.q_full[(it - 1) & 1], (unsigned)(((it - 1) >> 1) & 1), &never);
            }
        } else {
            // publish the last V tile
            cp_wait<0>();
            tc::fence_proxy_async();
            if (g > 0) {
                if (w2 == 2) arrive2(&bars.kv_full[(2 * (g - 1) + 1) % kRing]);
                else arrive(&bars.kv_full[(2 * (g - 1) + 1) % kRing]);
            }
        }
    } else if (!kTma && warp >= kSoftWarps && warp < kMmaWarpOf<kTma>) {
        // ------------------------------------------------------- gather (cp.async)
        const int gt = threadIdx.x - kSoftWarps * 32;  // 0..127: the item row this thread copies
        const int gw = gt >> 5;
        int it = 0;
        int64_t u = 0;  // tiles (K or V) issued
        int64_t g = 0;  // item tiles (mask ring uses)
        bool ok = true;
        for (int row = blockIdx.x; row < a.rows && ok; row += gridDim.x, ++it) {
            const int b = row / a.T, t = row - (row / a.T) * a.T;
            const int64_t p = a.q_pos0[b] + t;
            int64_t E = num_entries(p, a.m);
            if (E > a.E_cap) E = a.E_cap;
            const int cntr = a.cnt ? min(max(a.cnt[row], 0), a.topk) : a.topk;
            if (gt == 0) {
                if (it >= 2) ok = wait_bar(&bars.q_empty[it & 1], (unsigned)(((it >> 1) - 1) & 1), &s_abort);
                if (ok) {
                    mbar_expect_tx(&bars.q_full[it & 1], kQBytes);
                    tc::tma_load_2d(sQ + (it & 1) * kQBytes, &tm_q, 0, row * kH, &bars.q_full[it & 1]);
                    tc::tma_load_2d(sQ + (it & 1) * kQBytes + kQBlk, &tm_q, 64, row * kH, &bars.q_full[it & 1]);
                }
            }
            ok = __all_sync(0xffffffffu, ok);  // the warp's lanes leave together (ballots below)
            // selected indices are loaded one tile ahead, so each load's round trip overlaps
            // the copies of the tile before
            int32_t e_next = (gt < a.topk && gt < cntr) ? a.idx[(int64_t)row * a.topk + gt] : -1;
            for (int j = 0; j < nt && ok; ++j, ++g) {
                // the item this thread copies, and whether it is valid
                const int slot_i = j * kN + gt;
                const int32_t e = e_next;
                {
                    const int slot_n = slot_i + kN;
                    e_next = (slot_n < a.topk && slot_n < cntr) ? a.idx[(int64_t)row * a.topk + slot_n] : -1;
                }
                const __nv_bfloat16 *ksrc = nullptr, *vsrc = nullptr;
                if (slot_i < a.topk) {
                    if (e >= E) raise_flag(FLAG_ATTN_INDEX);
                    if (e >= 0 && e < E) {
                        ksrc = a.kc + b * a.c_sb + (int64_t)e * a.c_se;
                        vsrc = a.vc + b * a.c_sb + (int64_t)e * a.c_se;
                    }
                } else if (slot_i < a.topk + a.window) {
                    const int64_t tr = p - a.window + 1 + (slot_i - a.topk);
                    if (tr >= 0 && tr <= p) {
                        if (tr >= a.N_cap) raise_flag(FLAG_ATTN_RANGE);
                        else {
                            ksrc = a.k_raw + b * a.r_sb + tr * a.r_st;
                            vsrc = a.v_raw + b * a.r_sb + tr * a.r_st;
                        }
                    }
                }
                // validity mask of the tile (one word per gather warp)
                const uint32_t bits = __ballot_sync(0xffffffffu, ksrc != nullptr);
                const int ms = (int)(g % kMaskRing);
                if (g >= kMaskRing)
                    ok = wait_bar(&bars.m_empty[ms], (unsigned)(((g / kMaskRing) - 1) & 1), &s_abort);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (lane == 0) {
                    s_mask[ms][gw] = bits;
                    arrive(&bars.m_full[ms]);
                }
                for (int kv = 0; kv < 2 && ok; ++kv, ++u) {
                    const int slot = (int)(u % kRing);
                    if (u >= kRing) ok = wait_bar(&bars.kv_empty[slot], (unsigned)(((u / kRing) - 1) & 1), &s_abort);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    // a half-warp copies one 256-byte row (lane l: 16-byte chunk l % 16), so
                    // each instruction moves two whole rows; row pointers come by shuffle
                    // from the lane that resolved the row
                    const __nv_bfloat16 *src = kv ? vsrc : ksrc;
                    const unsigned long long sv = reinterpret_cast<unsigned long long>(src);
                    unsigned char *dst = sRing + slot * kTile;
                    const int c = lane & 15;
#pragma unroll 4
                    for (int i = 0; i < 16; ++i) {
                        const int rl = 2 * i + (lane >> 4);            // row within this warp's 32
                        const unsigned long long rs = __shfl_sync(0xffffffffu, sv, rl);
                        const int r = gw * 32 + rl;                     // row within the tile
                        const uint32_t off = (uint32_t)((c >> 3) * kTBlk + r * 128 + (((c & 7) ^ (r & 7)) << 4));
                        const __nv_bfloat16 *rp = reinterpret_cast<const __nv_bfloat16 *>(rs);
                        cp_async_16(smem_u32(dst + off), rp ? (const void *)(rp + c * 8) : (const void *)a.kc,
                                    rp ? 16 : 0);  // zero-fill invalid rows
                    }
                    cp_async_commit();
                    // the tile issued kLag groups ago has landed: publish it to the MMA
                    if (u >= kLag) {
                        cp_wait<kLag>();
                        tc::fence_proxy_async();
                        arrive(&bars.kv_full[(u - kLag) % kRing]);
                    }
                }
            }
        }
        // publish the last tiles (and let every copy land before the CTA exits)
        cp_wait<0>();
        tc::fence_proxy_async();
        for (int64_t v = (u > kLag ? u - kLag : 0); v < u; ++v) arrive(&bars.kv_full[v % kRing]);
        if (!ok) s_abort = 1;
        if (gt == 0 && it > 0) {
            volatile int never = 0;
            wait_bar(&bars.q_full[(it - 1) & 1], (unsigned)(((it - 1) >> 1) & 1), &never);
        }
    } else if (warp == kMmaWarpOf<kTma>) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_bf16(kH, kN, false, false);
            constexpr uint32_t idO = tc::idesc_bf16(kH, kD, false, true);
            const uint32_t aP = smem_u32(sP);
            int it = 0;
            int64_t g = 0, u = 0;
            bool ok = true;
            auto wait_tile = [&](int64_t uu) -> uint32_t {
                const int slot = (int)(uu % kRing);
                ok = ok && wait_bar(&bars.kv_full[slot], (unsigned)((uu / kRing) & 1), &s_abort);
                return smem_u32(sRing + slot * kTile);
            };
            // PV of item tile gg (ring use uv); the first of token tok waits until the softmax
            // has read the previous token's O
            auto issue_pv = [&](int64_t gg, int64_t uv, bool first, int tok) {
                ok = ok && wait_bar(&bars.p_full, (unsigned)(gg & 1), &s_abort);
                if (ok && first && tok > 0) ok = wait_bar(&bars.o_free, (unsigned)((tok - 1) & 1), &s_abort);
                const uint32_t aV = wait_tile(uv);
                if (!ok) return;
                tc::fence_after();
#pragma unroll
                for (int kk = 0; kk < kN / 16; ++kk) {
                    const uint64_t da = tc::desc_sw128(aP + (kk >> 2) * kQBlk + (kk & 3) * 32, 16, 1024);
                    const uint64_t db = tc::desc_sw128(aV + kk * 16 * 128, kTBlk, 1024);
                    tc::mma_bf16(tO, da, db, idO, (first && kk == 0) ? 0u : 1u);
                }
                tc::commit(&bars.o_done);
                tc::commit(&bars.kv_empty[uv % kRing]);
            };
            // S(g) goes out before PV(g-1), across token boundaries too, so the softmax finds the
            // next token's first S ready when it finishes a token
            int64_t pv_g = -1, pv_u = -1;  // the PV still to issue
            bool pv_first = false;
            int pv_tok = 0;
            for (int row = blockIdx.x; row < a.rows && ok; row += gridDim.x, ++it) {
                ok = wait_bar(&bars.q_full[it & 1], (unsigned)((it >> 1) & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                const uint32_t aQ = smem_u32(sQ + (it & 1) * kQBytes);
                for (int j = 0; j < nt && ok; ++j, ++g) {
                    const int64_t uk = u, uv = u + 1;
                    u += 2;
                    const uint32_t aK = wait_tile(uk);
                    if (ok && g >= 2) ok = wait_bar(&bars.s_free[g & 1], (unsigned)(((g >> 1) - 1) & 1), &s_abort);
                    if (!ok) break;
                    tc::fence_after();
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint64_t da = tc::desc_sw128(aQ + (kk >> 2) * kQBlk + (kk & 3) * 32, 16, 1024);
                        const uint64_t db = tc::desc_sw128(aK + (kk >> 2) * kTBlk + (kk & 3) * 32, 16, 1024);
                        tc::mma_bf16(tS(g), da, db, idS, kk > 0 ? 1u : 0u);
                    }
                    tc::commit(&bars.s_full[g & 1]);
                    tc::commit(&bars.kv_empty[uk % kRing]);
                    if (j == nt - 1) tc::commit(&bars.q_empty[it & 1]);
                    if (pv_g >= 0) issue_pv(pv_g, pv_u, pv_first, pv_tok);
                    pv_g = g;
                    pv_u = uv;
                    pv_first = j == 0;
                    pv_tok = it;
                }
            }
            if (ok && pv_g >= 0) issue_pv(pv_g, pv_u, pv_first, pv_tok);
            if (!ok) s_abort = 1;
            tc::commit(&bars.mma_fin);
            volatile int never = 0;
            wait_bar(&bars.mma_fin, 0u, &never);
        }
    } else if (warp < kSoftWarps) {
        // ---------------------------------------------------------------- softmax
        const bool active = lane < 16;
        const int h = warp * 16 + lane;  // head of this thread (active lanes)
        const bool upper = lane >= 16;
        const int hr = warp * 16 + (lane & 15);  // the head whose row this lane works on
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        int64_t g = 0;
        int it = 0;
        bool ok = true;
        for (int row = blockIdx.x; row < a.rows && ok; row += gridDim.x, ++it) {
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < nt && ok; ++j, ++g) {
                ok = wait_bar(&bars.s_full[g & 1], (unsigned)((g >> 1) & 1), &s_abort);
                const int ms = (int)(g % kMaskRing);
                if (ok) ok = wait_bar(&bars.m_full[ms], (unsigned)((g / kMaskRing) & 1), &s_abort);
                ok = __all_sync(0xffffffffu, ok);  // warp-collective TMEM loads below
                if (!ok) break;
                tc::fence_after();
                uint32_t mw[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) mw[q] = s_mask[ms][q];
                arrive(&bars.m_empty[ms]);
                // S of this tile into registers, two lanes per head: lane l < 16 takes
                // columns 0-63 of head h's row (TMEM lane 32w + l), lane l + 16 columns
                // 64-127 of the same row, passed over by a shuffle; 32 columns per load.
                // The S buffer is free for the next tile's MMA as soon as it is read.
                uint32_t v[64];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t w[32];
                    tc::tmem_ld32(tS(g) + lane_off + 64 + q * 32, w);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) v[q * 32 + c] = __shfl_xor_sync(0xffffffffu, w[c], 16);
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t w[32];
                    tc::tmem_ld32(tS(g) + lane_off + q * 32, w);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) v[q * 32 + c] = upper ? v[q * 32 + c] : w[c];
                }
                tc::fence_before();
                arrive(&bars.s_free[g & 1]);  // S has been read in full
                // tiles with every item valid (the common case) skip the mask
                if ((mw[0] & mw[1] & mw[2] & mw[3]) != 0xffffffffu) {
                    const uint32_t m0 = upper ? mw[2] : mw[0], m1 = upper ? mw[3] : mw[1];
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (!(((c < 32 ? m0 : m1) >> (c & 31)) & 1u)) v[c] = __float_as_uint(-INFINITY);
                }
                float mx8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) mx8[q] = -INFINITY;
#pragma unroll
                for (int c = 0; c < 64; c += 2)
                    mx8[(c >> 1) & 7] = tc::fmax3(mx8[(c >> 1) & 7], __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
                float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16)) * a.scale_log2;
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
                // P = 2^(x * scale_log2 - m_used) in bf16 (each lane its 64 columns), computed
                // in registers while the previous PV still reads P; invalid items read as -inf
                // (exponent 0), the scale goes into a packed FMA
                const float nmu = m_used == -INFINITY ? 0.f : -m_used;
                const uint64_t nmu2 = pack2(nmu, nmu), sc2 = pack2(a.scale_log2, a.scale_log2);
                uint64_t acc2[4] = {0, 0, 0, 0};
                uint32_t pk[32];
#pragma unroll
                for (int c2 = 0; c2 < 32; ++c2) {
                    const uint64_t arg = fma_f32x2(((uint64_t)v[2 * c2 + 1] << 32) | v[2 * c2], sc2, nmu2);
                    const float p0 = tc::ex2(lo_of(arg)), p1 = tc::ex2(hi_of(arg));
                    acc2[c2 & 3] = add_f32x2(acc2[c2 & 3], pack2(p0, p1));
                    pk[c2] = pack_bf16x2(p0, p1);
                }
                // P and O are free once the previous PV has completed
                if (g > 0) ok = wait_bar(&bars.o_done, (unsigned)((g - 1) & 1), &s_abort);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc::fence_after();
                if (__any_sync(0xffffffffu, rescale && active)) {
#pragma unroll
                    for (int c = 0; c < kD / 32; ++c) {
                        uint32_t o[32];
                        tc::tmem_ld32(tO + lane_off + c * 32, o);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::tmem_st32(tO + lane_off + c * 32, o);
                    }
                    tc::tmem_wait_st();
                }
                // P into 128-byte-swizzled K-major rows
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4 *>(sP + (upper ? kQBlk : 0) + hr * 128 + ((cc ^ (hr & 7)) << 4)) =
                        make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                const uint64_t s4 = add_f32x2(add_f32x2(acc2[0], acc2[1]), add_f32x2(acc2[2], acc2[3]));
                float sum = lo_of(s4) + hi_of(s4);
                sum += __shfl_xor_sync(0xffffffffu, sum, 16);
                l += sum;
                tc::fence_proxy_async();
                tc::fence_before();
                arrive(&bars.p_full);
            }
            if (!ok) break;
            // epilogue: O / l once the token's last PV is done
            ok = wait_bar(&bars.o_done, (unsigned)((g - 1) & 1), &s_abort);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc::fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *orow = a.out + ((int64_t)row * kH + h) * kD;
#pragma unroll
            for (int c = 0; c < kD / 32; ++c) {
                uint32_t o[32];
                tc::tmem_ld32(tO + lane_off + c * 32, o);
                tc::tmem_wait_ld();
                if (active) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 pk;
                        pk.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                        pk.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        pk.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        pk.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + c * 32 + e) = pk;
                    }
                }
            }
            tc::fence_before();
            arrive(&bars.o_free);
            if (active && a.lse) a.lse[(int64_t)row * kH + h] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
        }
        if (!ok) s_abort = 1;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

constexpr size_t kSmemBytes = 1024 + 2 * (size_t)kQBytes + kRing * (size_t)kTile + kQBytes;

}  // namespace

bool gather_tc_supported(const AttnArgs &a) {
    return a.d == kD && a.H == kH && a.idx != nullptr && a.topk > 0 && a.rows > 0;
}

cudaError_t launch_attn_gather_tc(const AttnArgs &a, int num_sms, cudaStream_t s) {
    CUtensorMap tq;
    {
        const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)a.rows * kH};
        const uint64_t str[1] = {(uint64_t)kD};
        if (!make_tmap_bf16(&tq, a.q, 2, dims, str, kH)) return cudaErrorInvalidValue;
    }
    GatherArgs g;
    g.rows = a.rows;
    g.T = a.T;
    g.topk = a.topk;
    g.window = a.window;
    g.m = a.m;
    g.n_tiles = (a.topk + a.window + kN - 1) / kN;
    g.E_cap = a.E_cap;
    g.N_cap = a.N_cap;
    g.c_sb = a.c_sb;
    g.c_se = a.c_se;
    g.r_sb = a.r_sb;
    g.r_st = a.r_st;
    g.q_pos0 = a.pos;
    g.idx = a.idx;
    g.cnt = a.cnt;
    g.kc = static_cast<const __nv_bfloat16 *>(a.kc);
    g.vc = static_cast<const __nv_bfloat16 *>(a.vc);
    g.k_raw = static_cast<const __nv_bfloat16 *>(a.k_raw);
    g.v_raw = static_cast<const __nv_bfloat16 *>(a.v_raw);
    g.scale_log2 = a.scale * kLog2e;
    g.out = static_cast<__nv_bfloat16 *>(a.out);
    g.lse = a.lse;
    // Rows by tile::gather4 when each cache is a 2-D tensor of rows (a sequence's first row
    // a whole number of rows after the previous one's), every row coordinate fits 31 bits,
    // and a gather group of 4 slots never spans the selected entries and the window.
    const int B = a.rows / a.T;
    const bool strides_ok = a.c_se > 0 && a.c_sb % a.c_se == 0 && a.r_st > 0 && a.r_sb % a.r_st == 0;
    CUtensorMap tkc = tq, tvc = tq, tkr = tq, tvr = tq;
    bool tma = a.topk % 4 == 0 && strides_ok;
    if (tma) {
        g.c_rows_b = a.c_sb / a.c_se;
        g.r_rows_b = a.r_sb / a.r_st;
        const int64_t c_rows = (int64_t)(B - 1) * g.c_rows_b + a.E_cap;
        const int64_t r_rows = (int64_t)(B - 1) * g.r_rows_b + a.N_cap;
        tma = c_rows > 0 && r_rows > 0 && c_rows < (int64_t)INT32_MAX && r_rows < (int64_t)INT32_MAX;
        if (tma) {
            const uint64_t cd[2] = {(uint64_t)kD, (uint64_t)c_rows}, rd[2] = {(uint64_t)kD, (uint64_t)r_rows};
            const uint64_t cs[1] = {(uint64_t)a.c_se}, rs[1] = {(uint64_t)a.r_st};
            tma = make_tmap_bf16(&tkc, a.kc, 2, cd, cs, 1) && make_tmap_bf16(&tvc, a.vc, 2, cd, cs, 1) &&
                  make_tmap_bf16(&tkr, a.k_raw, 2, rd, rs, 1) && make_tmap_bf16(&tvr, a.v_raw, 2, rd, rs, 1);
        }
    }
    if (!tma) g.c_rows_b = g.r_rows_b = 0;
    const int grid = a.rows < num_sms ? a.rows : num_sms;
    if (tma) {
        static unsigned long long done = 0;
        cudaError_t e = smem_limit_once(attn_gather_tc_kernel<true>, (int)kSmemBytes, done);
        if (e != cudaSuccess) return e;
        attn_gather_tc_kernel<true><<<grid, kThreadsOf<true>, kSmemBytes, s>>>(tq, tkc, tvc, tkr, tvr, g);
    } else {
        static unsigned long long done = 0;
        cudaError_t e = smem_limit_once(attn_gather_tc_kernel<false>, (int)kSmemBytes, done);
        if (e != cudaSuccess) return e;
        attn_gather_tc_kernel<false><<<grid, kThreadsOf<false>, kSmemBytes, s>>>(tq, tkc, tvc, tkr, tvr, g);
    }
    return cudaGetLastError();
}

}  // namespace hsa
