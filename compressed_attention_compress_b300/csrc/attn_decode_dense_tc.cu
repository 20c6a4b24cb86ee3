// Decode attention of an HCA layer (one query token per sequence, dense over all
// visible compressed entries plus the raw window), bf16, d = 128, H a multiple
// of 64, on the 5th-generation tensor cores with TMA-fed operands.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制: HCA runs dense
// attention over every heavily compressed entry (m' = 128); the sliding-window
// paragraph adds the most recent raw tokens to the same softmax; strict causality
// limits the query at p to the E(p) = floor((p+1)/m) complete blocks.
//
// The items of a (sequence, 64-head group) -- its E entries, then its window
// tokens -- form a run of 128-item tiles (entry tiles, then window tiles); the
// runs of the batch, one after another, form one list of T tiles.  CTA c of the
// persistent grid (one per SM, G CTAs) takes the contiguous range
// [floor(c T / G), floor((c+1) T / G)) of that list, so every SM streams the same
// number of tiles whatever the sequences' lengths.  Inside its range a CTA
// accumulates each run's tiles in TMEM with an online softmax and writes
// partials (unnormalised O, maximum, sum) for the runs it touches;
// attn_decode_dense_merge_kernel combines the pieces of every run in list order.
// The split depends on the whole batch: results are deterministic for a given
// batch, not bit-identical across batches.
// The kernel is launched with programmatic stream serialization: its barrier set-up,
// TMEM allocation and tensor-map prefetch overlap the preceding kernel, and every CTA
// waits for that kernel's completion (griddepcontrol.wait) before it reads any input.
//
// Warp roles:
//   warp 0      TMA producer (one thread): Q of the run (64 heads x 128), then
//               the K and V tiles (two 64-column boxes of 128 rows, 128-byte
//               swizzle) through a 2-slot K ring and a 3-slot V ring of 32 KiB,
//               V one tile behind K.
//   warp 1      S issuer (one thread): S(j) = Q K_j^T (M = 64 heads, N = 128
//               items) into TMEM buffer j % 2.
//   warp 2      PV issuer (one thread): O_g += P(j) V_j (N = d) for softmax group
//               g = j % 2; the two issuers wait only on their own inputs.
//   warps 4-11  two softmax warpgroups, group g taking tiles j = g, g + 2, ...
//               with its own P buffer and O accumulator (online softmax, O
//               rescaled in TMEM only when a head's maximum grows by more than
//               2^8); four threads per head (TMEM reads of shape 16x256b); at the
//               end of its tiles of a run the group writes one piece (O, maximum,
//               sum), so a run has up to two pieces per CTA.
// V rows a tile loads past its visible items (entries at or beyond E, raw tokens
// after p) are zeroed in shared memory before the PV MMA: those cache rows may
// hold any bits, their P is 0, and 0 times a NaN would still poison the sum.
// Every wait is bounded; a wait that gives up raises the device flag and the CTA
// stops issuing work, lets its copies and MMAs land and frees its TMEM.
#include <math.h>

#include <cudaTypedefs.h>

#include "internal.h"
#include "tc_common.cuh"

namespace hsa {

namespace {

constexpr int kH = 64;                  // heads per run = MMA M
constexpr int kD = 128;                 // head dim
constexpr int kN = 128;                 // items per tile = MMA N of S, K of PV
constexpr int kQBlk = kH * 128;         // 8 KiB: one 64-column block of Q or P
constexpr int kQBytes = 2 * kQBlk;      // 16 KiB
constexpr int kTBlk = kN * 128;         // 16 KiB: one 64-column block of a K or V tile
constexpr int kTile = 2 * kTBlk;        // 32 KiB
constexpr int kKRing = 2;               // K tile slots (freed by S)
constexpr int kVRing = 3;               // V tile slots (freed by PV)
constexpr int kRing = kKRing + kVRing;
constexpr int kThreads = 12 * 32;       // producer, S issuer, PV issuer, idle, 2 softmax warpgroups
constexpr int kMaxB = 1024;             // sequences per call (per-sequence data kept in shared memory)
constexpr int kMaxGrid = 256;           // CTAs of the main kernel (one per SM)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;        // log2 units
constexpr unsigned long long kWaitLimit = 1ull << 24;
// 1 KiB alignment | Q | K/V ring | P (2)
constexpr size_t kSmemBytes = 1024 + (size_t)kQBytes + kRing * (size_t)kTile + 2 * (size_t)kQBytes;

struct DenseArgs {
    int B, H, HG, m, window, n_win_tiles, t_max;
    int64_t E_cap, N_cap;
    const int64_t *ctx;  // [B]: the query sits at p = ctx - 1
    float scale_log2;
    __nv_bfloat16 *part_o;  // [B * HG * t_max][64][128]: unnormalised O of a piece (bf16), at the piece's first tile
    float *part_ml;      // [B * HG * t_max][2][64]: maximum (log2 units), sum
    int *cum;            // [B + 1]: the tile prefix, for the merge
    __nv_bfloat16 *out;  // [B, H, d]
    float *lse;          // [B, H] or null
};

struct __align__(8) Bars {
    uint64_t q_full, q_empty;
    uint64_t k_full[kKRing], k_empty[kKRing], v_full[kVRing], v_empty[kVRing];
    uint64_t s_full[2], p_full[2], p_empty[2], o_full[2], o_empty[2];  // per softmax group
    uint64_t mma_fin[2];
};

struct Sched {
    const int *cum;     // [B + 1]: tiles before sequence b (all its head groups)
    const int *E;       // [B]: visible entries (clamped to E_cap)
    const int64_t *p;   // [B]: query position
    int total;          // T
};

// Per-sequence position, visible entries and tiles, and the prefix of the tiles
// over the batch, into shared memory (all threads of the block take part).
__device__ void build_sched(const DenseArgs &a, int *s_cum, int *s_E, int64_t *s_p, bool flag) {
    const int lane = threadIdx.x & 31;
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
        const int64_t p = a.ctx[b] - 1;
        int64_t E = num_entries(p, a.m);
        if (E > a.E_cap) {
            if (flag) raise_flag(FLAG_ATTN_RANGE);
            E = a.E_cap;
        }
        if (p >= a.N_cap && a.window > 0 && flag) raise_flag(FLAG_ATTN_RANGE);
        if (s_p) s_p[b] = p;
        if (s_E) s_E[b] = (int)E;
        const int tiles = p < 0 ? 0 : (int)((E + kN - 1) / kN) + a.n_win_tiles;
        s_cum[b + 1] = tiles * a.HG;
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // inclusive scan of s_cum[1..B], 32 sequences at a time
        int carry = 0;
        for (int b0 = 0; b0 < a.B; b0 += 32) {
            int v = b0 + lane < a.B ? s_cum[b0 + lane + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            if (b0 + lane < a.B) s_cum[b0 + lane + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) s_cum[0] = 0;
    }
    __syncthreads();
}

// Tile U of the list: sequence b, head group hg, tile t of the run.
struct Tile {
    int b, hg, t, run;
    bool entry;         // entry tile (else window tile)
    int64_t y0;         // first row of the tile in kc/vc (entry) or the raw cache (window)
    int c_lo, c_hi;     // visible items are columns [c_lo, c_hi) of the tile
    int zero_lo, zero_hi;  // V rows to clear before the PV MMA (in-bounds rows past the visible ones)
};

__device__ __forceinline__ Tile tile_info(const DenseArgs &a, const Sched &sc, int U) {
    int lo = 0, hi = a.B - 1;  // last b with cum[b] <= U
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sc.cum[mid] <= U) lo = mid;
        else hi = mid - 1;
    }
    Tile u;
    u.b = lo;
    const int64_t p = sc.p[u.b];
    const int64_t E = sc.E[u.b];
    const int n_ent = (int)((E + kN - 1) / kN);
    const int run_tiles = n_ent + a.n_win_tiles;
    const int r = U - sc.cum[lo];
    u.hg = r / run_tiles;
    u.t = r - u.hg * run_tiles;
    u.run = u.b * a.HG + u.hg;
    u.entry = u.t < n_ent;
    int64_t rows;  // rows of the tile inside its tensor (the rest read the TMA zero fill)
    if (u.entry) {
        u.y0 = (int64_t)u.t * kN;
        u.c_lo = 0;
        u.c_hi = (int)(E - u.y0 < kN ? E - u.y0 : kN);
        rows = a.E_cap - u.y0;
    } else {
        const int k = u.t - n_ent;
        u.y0 = p - a.window + 1 + (int64_t)k * kN;
        // window token y0 + c is visible iff 0 <= y0 + c <= p, c + 128k < window and
        // y0 + c < N_cap
        int64_t lo_c = -u.y0 > 0 ? -u.y0 : 0;
        int64_t hi_c = p - u.y0 + 1;
        if (hi_c > kN) hi_c = kN;
        if (hi_c > a.window - (int64_t)k * kN) hi_c = a.window - (int64_t)k * kN;
        if (hi_c > a.N_cap - u.y0) hi_c = a.N_cap - u.y0;
        if (hi_c < 0) hi_c = 0;
        if (lo_c > hi_c) lo_c = hi_c;
        u.c_lo = (int)lo_c;
        u.c_hi = (int)hi_c;
        rows = a.N_cap - u.y0;
    }
    // in-bounds rows past the visible ones hold real memory with any bits; rows
    // before c_lo are window rows at negative positions (zero fill)
    if (rows > kN) rows = kN;
    u.zero_lo = u.c_hi;
    u.zero_hi = rows > u.c_hi ? (int)rows : u.c_hi;
    return u;
}

__device__ __forceinline__ int range_begin(int c, int T, int G) { return (int)(((int64_t)c * T) / G); }

// The producer issues, at step s, K_s (s < n) and then V_{s - kVLag}
// (0 <= s - kVLag < n): V lags K so that a V tile lands about when its P is ready
// instead of waiting in shared memory through the softmax.  K tiles go through
// their own ring (consumed by the S issuer), V tiles through another (consumed by
// the PV issuer): each ring has a single consumer taking its fills in order, so a
// wait on a slot's fill can never be mistaken for the fill two before it.
constexpr int kVLag = 1;

__device__ __forceinline__ bool wait_bar(uint64_t *bar, unsigned parity, volatile int *abort) {
    for (unsigned long long i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    raise_flag(FLAG_ATTN_RANGE | 0x1000u);
    *abort = 1;
    return false;
}
__device__ __forceinline__ void arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
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

// 16 TMEM lanes (from the lane in taddr) x 64 columns, shape 16x256b repeated 8
// times: thread t gets, for k = 0..7, rows t/4 (v[4k], v[4k+1]) and t/4 + 8
// (v[4k+2], v[4k+3]), columns 8k + 2 (t % 4) and 8k + 2 (t % 4) + 1.
__device__ __forceinline__ void tmem_ld16x256_x8(uint32_t taddr, uint32_t *v) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16x256_x8(uint32_t taddr, const uint32_t *v) {
    asm volatile("tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
}
// 16 TMEM lanes (from the lane in taddr) x 128 columns, shape 16x256b repeated 16
// times: thread t gets, for k = 0..15, rows t/4 (v[4k], v[4k+1]) and t/4 + 8
// (v[4k+2], v[4k+3]), columns 8k + 2 (t % 4) and 8k + 2 (t % 4) + 1.
__device__ __forceinline__ void tmem_ld16x256_x16(uint32_t taddr, uint32_t *v) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]), "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16x256_x16(uint32_t taddr, const uint32_t *v) {
    asm volatile("tcgen05.st.sync.aligned.16x256b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]), "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]), "r"(v[37]), "r"(v[38]), "r"(v[39]), "r"(v[40]), "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]), "r"(v[46]), "r"(v[47]), "r"(v[48]), "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]), "r"(v[55]), "r"(v[56]), "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
                 : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_decode_dense_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                                const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kr,
                                const __grid_constant__ CUtensorMap tm_vr, DenseArgs a) {
    // the merge kernel (launched after this one with programmatic stream
    // serialization) may be scheduled now; it waits for this grid's completion
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    extern __shared__ __align__(16) unsigned char smem_raw[];  // rounded up to 1024 below, at run time
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *sQ = smem;                       // 16 KiB
    unsigned char *sKV = sQ + kQBytes;              // kRing x 32 KiB: K ring, then V ring
    unsigned char *sP = sKV + kRing * kTile;        // 2 x 16 KiB
    __shared__ Bars bars;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ int s_cum[kMaxB + 1];
    __shared__ int s_E[kMaxB];
    __shared__ int64_t s_p[kMaxB];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Launched with programmatic stream serialization: the barriers, the TMEM allocation
    // and the tensor-map prefetch overlap the preceding kernel (the new block's
    // compression, typically); every input is read after griddepcontrol.wait.
    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        for (int i = 0; i < kKRing; ++i) {
            mbar_init(&bars.k_full[i], 1);
            mbar_init(&bars.k_empty[i], 1);
        }
        for (int i = 0; i < kVRing; ++i) {
            mbar_init(&bars.v_full[i], 1);
            mbar_init(&bars.v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.p_full[i], 128);
            mbar_init(&bars.p_empty[i], 1);
            mbar_init(&bars.o_full[i], 1);
            mbar_init(&bars.o_empty[i], 128);
        }
        mbar_init(&bars.mma_fin[0], 1);
        mbar_init(&bars.mma_fin[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    if (warp == 3 && lane == 0) {
        for (const CUtensorMap *tm : {&tm_q, &tm_kc, &tm_vc, &tm_kr, &tm_vr})
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(tm) : "memory");
    }
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    build_sched(a, s_cum, s_E, s_p, blockIdx.x == 0);  // ends with a block barrier
    const Sched sc{s_cum, s_E, s_p, s_cum[a.B]};
    if (blockIdx.x == 0)
        for (int b = threadIdx.x; b <= a.B; b += blockDim.x) a.cum[b] = s_cum[b];  // for the merge
    const int G = gridDim.x;
    const int u_begin = range_begin(blockIdx.x, sc.total, G), u_end = range_begin(blockIdx.x + 1, sc.total, G);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (u_begin >= u_end) {  // no tile for this CTA
        if (warp == 0) tc::tmem_dealloc(s_tmem, 512);
        return;
    }
    const uint32_t tmem = s_tmem;
    const uint32_t tS[2] = {tmem, tmem + 128};
    const uint32_t tO[2] = {tmem + 256, tmem + 384};
    const int n_tiles = u_end - u_begin;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = -1;       // runs started
            int prev_run = -1;
            bool ok = true;
            int nk = 0, nv = 0;  // K and V tiles issued
            auto issue = [&](const Tile &u, bool is_v) {
                const int ring = is_v ? kVRing : kKRing;
                const int idx = is_v ? nv : nk;
                const int slot = idx % ring;
                uint64_t *empty = is_v ? &bars.v_empty[slot] : &bars.k_empty[slot];
                uint64_t *full = is_v ? &bars.v_full[slot] : &bars.k_full[slot];
                if (idx >= ring) ok = wait_bar(empty, (unsigned)(((idx / ring) - 1) & 1), &s_abort);
                if (!ok) return;
                unsigned char *dst = sKV + (is_v ? kKRing + slot : slot) * kTile;
                mbar_expect_tx(full, kTile);
                const CUtensorMap *tm = u.entry ? (is_v ? &tm_vc : &tm_kc) : (is_v ? &tm_vr : &tm_kr);
                const int y = (int)u.y0;
                tc::tma_load_3d(dst, tm, 0, y, u.b, full);
                tc::tma_load_3d(dst + kTBlk, tm, 64, y, u.b, full);
                if (is_v) ++nv;
                else ++nk;
            };
            Tile lag = tile_info(a, sc, u_begin);  // the tile whose V is issued next
            for (int step = 0; step < n_tiles + kVLag && ok; ++step) {
                if (step < n_tiles) {
                    const Tile u = tile_info(a, sc, u_begin + step);
                    if (u.run != prev_run) {
                        ++s;
                        prev_run = u.run;
                        // Q of the new run once every S of the previous run has completed
                        if (s >= 1) ok = wait_bar(&bars.q_empty, (unsigned)((s - 1) & 1), &s_abort);
                        if (!ok) break;
                        mbar_expect_tx(&bars.q_full, kQBytes);
                        const int qrow = u.b * a.H + u.hg * kH;
                        tc::tma_load_2d(sQ, &tm_q, 0, qrow, &bars.q_full);
                        tc::tma_load_2d(sQ + kQBlk, &tm_q, 64, qrow, &bars.q_full);
                    }
                    issue(u, false);
                }
                const int jv = step - kVLag;
                if (ok && jv >= 0 && jv < n_tiles) {
                    if (jv > 0) lag = tile_info(a, sc, u_begin + jv);
                    issue(lag, true);
                }
            }
            if (!ok) s_abort = 1;
            // let every copy this thread issued land before the CTA can exit
            volatile int never = 0;
            if (s >= 0) wait_bar(&bars.q_full, (unsigned)(s & 1), &never);
            for (int i = (nk > kKRing ? nk - kKRing : 0); i < nk; ++i)
                wait_bar(&bars.k_full[i % kKRing], (unsigned)((i / kKRing) & 1), &never);
            for (int i = (nv > kVRing ? nv - kVRing : 0); i < nv; ++i)
                wait_bar(&bars.v_full[i % kVRing], (unsigned)((i / kVRing) & 1), &never);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ S issuer
        // S(j) = Q K_j^T into S buffer j % 2 once Q of its run and K_j are there and
        // softmax group j % 2 has read S(j-2) (it arrived on p_full for tile j - 2).
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_bf16(kH, kN, false, false);
            bool ok = true;
            int rs = -1, prun = -1;  // runs of the S issued so far (count - 1)
            Tile ts = tile_info(a, sc, u_begin);
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int x = j & 1;
                const int rnew = ts.run != prun ? rs + 1 : rs;
                const int ks = j % kKRing;
                if (j >= 2) ok = wait_bar(&bars.p_full[x], (unsigned)(((j >> 1) - 1) & 1), &s_abort);
                ok = ok && wait_bar(&bars.q_full, (unsigned)(rnew & 1), &s_abort);
                ok = ok && wait_bar(&bars.k_full[ks], (unsigned)((j / kKRing) & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sKV + ks * kTile);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t da = tc::desc_sw128(aQ + (kk >> 2) * kQBlk + (kk & 3) * 32, 16, 1024);
                    const uint64_t db = tc::desc_sw128(aK + (kk >> 2) * kTBlk + (kk & 3) * 32, 16, 1024);
                    tc::mma_bf16(tS[x], da, db, idS, kk > 0 ? 1u : 0u);
                }
                tc::commit(&bars.s_full[x]);
                tc::commit(&bars.k_empty[ks]);
                rs = rnew;
                prun = ts.run;
                bool last_of_run = j + 1 == n_tiles;
                if (!last_of_run) {
                    ts = tile_info(a, sc, u_begin + j + 1);
                    last_of_run = ts.run != prun;
                }
                if (last_of_run) tc::commit(&bars.q_empty);  // Q may be replaced once these S complete
            }
            if (!ok) s_abort = 1;
            // every MMA this thread issued completes before TMEM is released
            tc::commit(&bars.mma_fin[0]);
            volatile int never = 0;
            wait_bar(&bars.mma_fin[0], 0u, &never);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ PV issuer
        // O_g += P(j) V_j for softmax group g = j % 2 once P(j) and V_j are there; a
        // group's piece (its tiles of one run in this range) starts with its O
        // buffer drained by the group's previous piece.
        if (lane == 0) {
            constexpr uint32_t idO = tc::idesc_bf16(kH, kD, false, true);
            bool ok = true;
            int pieces0 = 0, pieces1 = 0, prun0 = -1, prun1 = -1;
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int x = j & 1;
                const int run = tile_info(a, sc, u_begin + j).run;
                const int pieces = x ? pieces1 : pieces0;
                const bool start = run != (x ? prun1 : prun0);
                const int vs = j % kVRing;
                ok = wait_bar(&bars.p_full[x], (unsigned)((j >> 1) & 1), &s_abort);
                ok = ok && wait_bar(&bars.v_full[vs], (unsigned)((j / kVRing) & 1), &s_abort);
                if (ok && start && pieces >= 1)
                    ok = wait_bar(&bars.o_empty[x], (unsigned)((pieces - 1) & 1), &s_abort);
                if (!ok) break;
                tc::fence_after();
                const uint32_t aP = smem_u32(sP + x * kQBytes), aV = smem_u32(sKV + (kKRing + vs) * kTile);
#pragma unroll
                for (int kk = 0; kk < kN / 16; ++kk) {
                    const uint64_t da = tc::desc_sw128(aP + (kk >> 2) * kQBlk + (kk & 3) * 32, 16, 1024);
                    const uint64_t db = tc::desc_sw128(aV + kk * 16 * 128, kTBlk, 1024);
                    tc::mma_bf16(tO[x], da, db, idO, (start && kk == 0) ? 0u : 1u);
                }
                tc::commit(&bars.p_empty[x]);
                tc::commit(&bars.v_empty[vs]);
                if (x) {
                    pieces1 += start;
                    prun1 = run;
                } else {
                    pieces0 += start;
                    prun0 = run;
                }
                const bool piece_end = j + 2 >= n_tiles || tile_info(a, sc, u_begin + j + 2).run != run;
                if (piece_end) tc::commit(&bars.o_full[x]);
            }
            if (!ok) s_abort = 1;
            tc::commit(&bars.mma_fin[1]);
            volatile int never = 0;
            wait_bar(&bars.mma_fin[1], 0u, &never);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax + pieces
        // Group g (warps 4-7: g = 0, warps 8-11: g = 1) takes tiles j = g, g + 2, ...
        // with its own S buffer, P buffer and O accumulator, and writes one piece per
        // run it meets.  TMEM reads of shape 16x256b: thread t of warp w holds heads
        // 16w + t/4 and 16w + t/4 + 8, columns 8k + 2(t % 4) + {0, 1}; a head's
        // maximum and sum combine the four threads of a quad with two shuffles.
        const int x = (warp - 4) >> 2;
        const int wq = warp & 3;               // TMEM lane quadrant
        const int qd = lane & 3;
        const int hh[2] = {wq * 16 + (lane >> 2), wq * 16 + (lane >> 2) + 8};
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const int tid = threadIdx.x - 128 - 128 * x;  // 0..127 within the group
        unsigned char *myP = sP + x * kQBytes;
        bool ok = true;
        int pieces = 0;
        float m_used[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        int first = x;                         // the current piece's first tile
        int prun = -1;
        for (int j = x; j < n_tiles && ok; j += 2) {
            const Tile u = tile_info(a, sc, u_begin + j);
            if (u.run != prun) {
                prun = u.run;
                first = j;
                m_used[0] = m_used[1] = -INFINITY;
                l[0] = l[1] = 0.f;
            }
            ok = wait_bar(&bars.s_full[x], (unsigned)((j >> 1) & 1), &s_abort);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc::fence_after();
            uint32_t v[64];
            tmem_ld16x256_x16(tS[x] + lane_off, v);
            tc::tmem_wait_ld();
            if (u.c_lo > 0 || u.c_hi < kN) {
#pragma unroll
                for (int k = 0; k < 16; ++k)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int c = 8 * k + 2 * qd + e;
                        if (c < u.c_lo || c >= u.c_hi) {
                            v[4 * k + e] = __float_as_uint(-INFINITY);
                            v[4 * k + 2 + e] = __float_as_uint(-INFINITY);
                        }
                    }
            }
            float alpha[2] = {1.f, 1.f};
            bool rescale = false;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    mx4[k & 3] = fmaxf(mx4[k & 3], fmaxf(__uint_as_float(v[4 * k + 2 * i]),
                                                         __uint_as_float(v[4 * k + 2 * i + 1])));
                float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mx = mx == -INFINITY ? -INFINITY : mx * a.scale_log2;
                if (mx > m_used[i] + kRescale) {
                    if (m_used[i] != -INFINITY) {
                        alpha[i] = tc::ex2(m_used[i] - mx);
                        rescale = rescale || j > first;
                    }
                    l[i] *= (m_used[i] == -INFINITY) ? 0.f : alpha[i];
                    m_used[i] = mx;
                }
            }
            // P buffer and O of this group are free once the group's previous PV
            // (tile j - 2) has completed
            if (j >= 2) ok = wait_bar(&bars.p_empty[x], (unsigned)(((j >> 1) - 1) & 1), &s_abort);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (__any_sync(0xffffffffu, rescale)) {
                tc::fence_after();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t o[32];
                    tmem_ld16x256_x8(tO[x] + lane_off + hf * 64, o);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha[(e >> 1) & 1]);
                    tmem_st16x256_x8(tO[x] + lane_off + hf * 64, o);
                }
                tc::tmem_wait_st();
            }
            // P = 2^(s * scale_log2 - m) as bf16 pairs: row h, columns 8k + 2qd + {0, 1}
            // = bytes 4qd..4qd+3 of 16-byte chunk k of the 128-byte-swizzled row
            float sum[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float nm = m_used[i] == -INFINITY ? 0.f : -m_used[i];
                const int h = hh[i];
                unsigned char *row = myP + h * 128 + 4 * qd;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float p0 = tc::ex2(fmaf(__uint_as_float(v[4 * k + 2 * i]), a.scale_log2, nm));
                    const float p1 = tc::ex2(fmaf(__uint_as_float(v[4 * k + 2 * i + 1]), a.scale_log2, nm));
                    s0 += p0;
                    s1 += p1;
                    *reinterpret_cast<uint32_t *>(row + (k >> 3) * kQBlk + (((k & 7) ^ (h & 7)) << 4)) =
                        pack_bf16x2(p0, p1);
                }
                sum[i] = s0 + s1;
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], 1);
                sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], 2);
                l[i] += sum[i];
            }
            if (u.zero_hi > u.zero_lo) {
                // V rows past the visible items: clear them once the tile has landed
                // (the PV issuer consumes this fill only after this group's p_full, and
                // the slot's previous fill, V_{j-3}, was consumed before PV(j-2), which
                // this group waited for: the wait below sees this tile's fill)
                const int vs = j % kVRing;
                ok = wait_bar(&bars.v_full[vs], (unsigned)((j / kVRing) & 1), &s_abort);
                if (ok) {
                    unsigned char *tV = sKV + (kKRing + vs) * kTile;
                    const int nz = (u.zero_hi - u.zero_lo) * 16;  // 16-byte chunks over both column blocks
                    for (int i = tid; i < nz; i += 128) {
                        const int rr = u.zero_lo + (i >> 4), c = i & 15;
                        *reinterpret_cast<uint4 *>(tV + (c >> 3) * kTBlk + rr * 128 + ((c & 7) << 4)) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
            }
            tc::fence_proxy_async();
            tc::fence_before();
            arrive(&bars.p_full[x]);
            bool piece_end = j + 2 >= n_tiles;
            if (!piece_end) piece_end = tile_info(a, sc, u_begin + j + 2).run != u.run;
            if (!piece_end) continue;
            // the piece once its last PV is done: O (fp32), maximum and sum
            ok = __all_sync(0xffffffffu, ok) && wait_bar(&bars.o_full[x], (unsigned)(pieces & 1), &s_abort);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc::fence_after();
            const int slot = u_begin + first;  // the piece's first tile in the list
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t o[32];
                tmem_ld16x256_x8(tO[x] + lane_off + hf * 64, o);
                tc::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    __nv_bfloat16 *po = a.part_o + (int64_t)slot * (kH * kD) + (int64_t)hh[i] * kD + hf * 64 + 2 * qd;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<uint32_t *>(po + 8 * k) =
                            pack_bf16x2(__uint_as_float(o[4 * k + 2 * i]), __uint_as_float(o[4 * k + 2 * i + 1]));
                }
            }
            if (qd == 0) {
                float *pml = a.part_ml + (int64_t)slot * (2 * kH);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    pml[hh[i]] = m_used[i];
                    pml[kH + hh[i]] = l[i];
                }
            }
            tc::fence_before();
            arrive(&bars.o_empty[x]);
            ++pieces;
        }
        if (!ok) s_abort = 1;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// out[b, h] = sum_i 2^(m_i - M) O_i / sum_i 2^(m_i - M) l_i over the pieces i of
// the run (b, head group) -- one per CTA whose tile range meets the run, in CTA
// order -- and lse = (M + log2 L) ln 2.  Block (run, 8-head group); warp w takes
// head 8 * blockIdx.y + w, lane c the columns 4c..4c+3.  The tile prefix over the
// batch comes from the main kernel (its CTA 0 stores it in the workspace).
constexpr int kMergeWarps = 8;
constexpr int kMaxPieces = 2 * kMaxGrid;  // two softmax groups per CTA
__global__ void __launch_bounds__(kMergeWarps * 32) attn_decode_dense_merge_kernel(DenseArgs a, const int *cum, int G) {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    __shared__ int s_slot[kMaxPieces];
    __shared__ int s_n;
    const int run = blockIdx.x;  // b * HG + hg
    const int b = run / a.HG, hg = run - b * a.HG;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        const int T = __ldcg(cum + a.B), c0b = __ldcg(cum + b), c1b = __ldcg(cum + b + 1);
        const int tiles_b = (c1b - c0b) / a.HG;
        const int64_t g0 = c0b + (int64_t)hg * tiles_b, g1 = g0 + tiles_b;
        // CTAs c with floor(c T / G) < g1 and floor((c+1) T / G) > g0
        int c_first = 0, c_last = -1;
        if (tiles_b > 0 && T > 0) {
            c_first = (int)(((g0 + 1) * G + T - 1) / T) - 1;  // largest c with floor(c T / G) <= g0
            c_last = (int)((g1 * G + T - 1) / T) - 1;          // largest c with floor(c T / G) < g1
            if (c_first < 0) c_first = 0;
            if (c_last > G - 1) c_last = G - 1;
        }
        // in CTA c the run's tiles are [max(cb, g0), min(ce, g1)); softmax group x of c
        // took the ones at even (x = 0) or odd (x = 1) offsets from cb and wrote its
        // piece at the first of them
        int n = 0;
        for (int c0 = c_first; c0 <= c_last; c0 += 32) {
            const int c = c0 + lane;
            int sl[2] = {0, 0};
            bool pc[2] = {false, false};
            if (c <= c_last) {
                const int64_t cb = ((int64_t)c * T) / G, ce = ((int64_t)(c + 1) * T) / G;
                const int64_t lo = cb > g0 ? cb : g0, hi = ce < g1 ? ce : g1;
                if (lo < hi) {
                    pc[0] = true;
                    sl[0] = (int)lo;
                    if (lo + 1 < hi) {
                        pc[1] = true;
                        sl[1] = (int)lo + 1;
                    }
                }
            }
            // pieces in list order: lane by lane, the first tile before the second
            const unsigned m0 = __ballot_sync(0xffffffffu, pc[0]), m1 = __ballot_sync(0xffffffffu, pc[1]);
            const unsigned below = (1u << lane) - 1;
            const int pos = n + __popc(m0 & below) + __popc(m1 & below);
            if (pc[0] && pos < kMaxPieces) s_slot[pos] = sl[0];
            if (pc[1] && pos + 1 < kMaxPieces) s_slot[pos + 1] = sl[1];
            n += __popc(m0) + __popc(m1);
        }
        if (lane == 0) s_n = n < kMaxPieces ? n : kMaxPieces;
    }
    __syncthreads();
    const int n = s_n;
    const int hl = blockIdx.y * kMergeWarps + warp;
    // Up to kBatch pieces at a time with every load in flight at once: lane c's
    // columns 4c..4c+3 of each piece's O, and each piece's maximum and sum (every
    // lane loads them all; they are one 128-byte line per 32 heads).  The running
    // maximum M and the sums are rescaled when a later batch raises M.
    constexpr int kBatch = 32;
    float M = -INFINITY, L = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i0 = 0; i0 < n; i0 += kBatch) {
        uint2 ov[kBatch];
        float mv[kBatch], lv[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const bool in = i0 + k < n;
            const int64_t sl = in ? s_slot[i0 + k] : 0;
            const float *pml = a.part_ml + sl * (2 * kH);
            mv[k] = in ? __ldcg(pml + hl) : -INFINITY;
            lv[k] = in ? __ldcg(pml + kH + hl) : 0.f;
            ov[k] = in ? __ldcg(reinterpret_cast<const uint2 *>(a.part_o + sl * (kH * kD) + (int64_t)hl * kD) + lane)
                       : make_uint2(0u, 0u);
        }
        float bm = -INFINITY;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) bm = fmaxf(bm, mv[k]);
        if (bm == -INFINITY) continue;  // nothing visible in this batch (its O is not used)
        const float Mn = fmaxf(M, bm);
        if (M != -INFINITY && Mn != M) {
            const float r = tc::ex2(M - Mn);
            L *= r;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] *= r;
        }
        M = Mn;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const float wk = mv[k] == -INFINITY ? 0.f : tc::ex2(mv[k] - M);
            L = fmaf(wk, lv[k], L);
            acc[0] = fmaf(wk, bf16_lo(ov[k].x), acc[0]);
            acc[1] = fmaf(wk, bf16_hi(ov[k].x), acc[1]);
            acc[2] = fmaf(wk, bf16_lo(ov[k].y), acc[2]);
            acc[3] = fmaf(wk, bf16_hi(ov[k].y), acc[3]);
        }
    }
    const bool empty = !(L > 0.f);
    const float inv = empty ? 0.f : 1.f / L;
    const int h = hg * kH + hl;
    uint2 pk;
    pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2 *>(a.out + ((int64_t)b * a.H + h) * kD + lane * 4) = pk;
    if (a.lse && lane == 0) a.lse[(int64_t)b * a.H + h] = empty ? -INFINITY : (M + log2f(L)) * kLn2;
}

int t_max_of(int64_t E_cap, int window) {
    return (int)((E_cap + kN - 1) / kN) + (window + kN - 1) / kN;
}

}  // namespace

bool decode_dense_tc_shape(int B, int H, int d) { return d == kD && H % kH == 0 && H > 0 && B > 0 && B <= kMaxB; }

DecodeDenseWorkspace decode_dense_workspace(int B, int H, int64_t E_cap, int window) {
    DecodeDenseWorkspace w;
    const size_t slots = (size_t)B * (H / kH) * t_max_of(E_cap, window);  // one per tile of the list, at most
    w.off_o = 0;
    w.off_ml = (slots * kH * kD * sizeof(__nv_bfloat16) + 255) & ~(size_t)255;
    w.off_cum = w.off_ml + ((slots * 2 * kH * sizeof(float) + 255) & ~(size_t)255);
    w.total = w.off_cum + (((size_t)(B + 1) * sizeof(int) + 255) & ~(size_t)255);
    return w;
}

cudaError_t launch_attn_decode_dense_tc(const AttnArgs &a, int num_sms, cudaStream_t s) {
    const int B = a.rows;
    CUtensorMap tq, tkc, tvc, tkr, tvr;
    {
        const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)B * a.H};
        const uint64_t str[1] = {(uint64_t)kD};
        if (!make_tmap_bf16(&tq, a.q, 2, dims, str, kH)) return cudaErrorInvalidValue;
    }
    // a cache without rows gets a one-row map (never read: no tile of it exists)
    const void *kc = a.kc ? a.kc : a.q, *vc = a.vc ? a.vc : a.q;
    const void *kr = a.k_raw ? a.k_raw : a.q, *vr = a.v_raw ? a.v_raw : a.q;
    {
        const bool none = a.E_cap == 0 || !a.kc;
        const uint64_t dims[3] = {(uint64_t)kD, none ? 1 : (uint64_t)a.E_cap, none ? 1 : (uint64_t)B};
        const uint64_t str[2] = {none ? (uint64_t)kD : (uint64_t)a.c_se, none ? (uint64_t)kD : (uint64_t)a.c_sb};
        if (!make_tmap_bf16(&tkc, kc, 3, dims, str, kN)) return cudaErrorInvalidValue;
        if (!make_tmap_bf16(&tvc, vc, 3, dims, str, kN)) return cudaErrorInvalidValue;
    }
    {
        const bool none = a.window == 0 || !a.k_raw || a.N_cap == 0;
        const uint64_t dims[3] = {(uint64_t)kD, none ? 1 : (uint64_t)a.N_cap, none ? 1 : (uint64_t)B};
        const uint64_t str[2] = {none ? (uint64_t)kD : (uint64_t)a.r_st, none ? (uint64_t)kD : (uint64_t)a.r_sb};
        if (!make_tmap_bf16(&tkr, kr, 3, dims, str, kN)) return cudaErrorInvalidValue;
        if (!make_tmap_bf16(&tvr, vr, 3, dims, str, kN)) return cudaErrorInvalidValue;
    }
    DenseArgs g;
    g.B = B;
    g.H = a.H;
    g.HG = a.H / kH;
    g.m = a.m;
    g.window = a.window;
    g.n_win_tiles = (a.window + kN - 1) / kN;
    g.t_max = t_max_of(a.E_cap, a.window);
    g.E_cap = a.E_cap;
    g.N_cap = a.N_cap;
    g.ctx = a.pos;
    g.scale_log2 = a.scale * kLog2e;
    g.part_o = reinterpret_cast<__nv_bfloat16 *>(a.part_o);
    g.part_ml = a.part_lse;
    {
        const DecodeDenseWorkspace w = decode_dense_workspace(B, a.H, a.E_cap, a.window);
        g.cum = reinterpret_cast<int *>(reinterpret_cast<char *>(a.part_o) + w.off_cum);
    }
    g.out = static_cast<__nv_bfloat16 *>(a.out);
    g.lse = a.lse;
    static unsigned long long done = 0;
    cudaError_t e = smem_limit_once(attn_decode_dense_tc_kernel, (int)kSmemBytes, done);
    if (e != cudaSuccess) return e;
    const int64_t max_tiles = (int64_t)B * g.HG * g.t_max;
    int grid = (int)(max_tiles < num_sms ? max_tiles : num_sms);
    if (grid > kMaxGrid) grid = kMaxGrid;
    {
        cudaLaunchConfig_t mc = {};
        mc.gridDim = dim3((unsigned)grid);
        mc.blockDim = dim3(kThreads);
        mc.dynamicSmemBytes = kSmemBytes;
        mc.stream = s;
        cudaLaunchAttribute ma[1];
        ma[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        ma[0].val.programmaticStreamSerializationAllowed = 1;
        mc.attrs = ma;
        mc.numAttrs = 1;
        e = cudaLaunchKernelEx(&mc, attn_decode_dense_tc_kernel, tq, tkc, tvc, tkr, tvr, g);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * g.HG), kH / kMergeWarps);
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_decode_dense_merge_kernel, g, (const int *)g.cum, grid);
}

}  // namespace hsa
