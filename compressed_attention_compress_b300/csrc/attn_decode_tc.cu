// Decode attention (one query token per sequence) over the selected entries plus
// the window of a CSA layer, bf16, d = 128, H a multiple of 64, on the
// 5th-generation tensor cores.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制: CSA step 3 (MQA over
// the top-k compressed entries the indexer selected) and the sliding-window
// paragraph (the most recent raw tokens join the same softmax).
//
// A sequence's item slots (topk selected entries, then the window tokens) are cut
// into tiles of 128 items; tile j of a (sequence, 64-head group) is CTA j of a
// cluster of n_tiles CTAs.  Each CTA
//   - gathers its tile's K and V rows with cp.async into 128-byte-swizzled shared
//     memory (zero-filled for invalid slots, a 128-bit validity mask beside it);
//   - computes S = Q K^T (M = 64 heads, N = 128 items, K = d) into TMEM, one
//     thread issuing tcgen05.mma (row h of an M = 64 accumulator sits in TMEM lane
//     (h / 16) * 32 + h % 16, so lanes 0-15 of warp w hold heads 16w..16w+15);
//   - takes the masked softmax of its tile, one head per thread, writes P (bf16)
//     to shared memory and accumulates O = P V into TMEM;
//   - writes its unnormalised partial (O, maximum, sum) to the workspace with
//     coalesced stores.
// After a cluster barrier (its release/acquire also orders these global writes for
// the cluster) CTA r reads heads [r * hpc, (r + 1) * hpc) of all the partials from
// L2, combines them with the log-sum-exp rule and writes the output and the
// log-sum-exp.  The launch uses programmatic stream serialization: the barrier
// set-up and the TMEM allocation overlap the tail of the preceding kernel, and
// every CTA waits for that kernel's completion (griddepcontrol.wait) before it
// reads any input, since that kernel may have written the query, the positions,
// the cache or the selected indices.
// Every wait is bounded; a wait that gives up raises the device flag, and the CTA
// still reaches the cluster barrier and frees its TMEM.
#include <math.h>

#include <type_traits>

#include "internal.h"
#include "tc_common.cuh"

namespace hsa {

namespace {

constexpr int kH = 64;                  // heads per CTA = MMA M
constexpr int kD = 128;                 // head dim
constexpr int kN = 128;                 // items per tile = MMA N of S
constexpr int kThreads = 128;
constexpr int kMaxTiles = 16;           // cluster size limit
constexpr int kQBlk = kH * 128;         // 8 KiB: one 64-column block of Q or P
constexpr int kQBytes = 2 * kQBlk;      // 16 KiB
constexpr int kTBlk = kN * 128;         // 16 KiB: one 64-column block of a K or V tile
constexpr int kTile = 2 * kTBlk;        // 32 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitLimit = 1ull << 22;
// dynamic shared memory: 1 KiB for alignment | Q | K tile | V tile | P; the fp32
// partial O [64][128] (32 KiB) reuses the K tile once both MMAs are done
constexpr size_t kSmemBytes = 1024 + (size_t)kQBytes + 2 * (size_t)kTile + (size_t)kQBytes;

struct DecodeTcArgs {
    int B, H, topk, window, m, n_tiles, shared_kv;
    int64_t E_cap, N_cap, c_sb, c_se, r_sb, r_st;
    const int64_t *ctx;          // [B]: the query sits at p = ctx - 1
    const int32_t *idx, *cnt;    // [B, topk], [B] or null
    const __nv_bfloat16 *q, *kc, *vc, *k_raw, *v_raw;
    float scale_log2;
    __nv_bfloat16 *out;          // [B, H, d]
    float *lse;                  // [B, H] or null
    float *part_o;               // [B, H / 64, n_tiles, 64, d] fp32 partial O
    float *part_ml;              // [B, H / 64, n_tiles, 2, 64]: maximum (log2 units), sum
};
// V4 details (the V4 instantiation only): RMSNorm and partial RoPE of the query, sink
// and inverse rotation of the output
struct DecodeV4Args {
    int rope_dims;
    float eps;
    const float *gamma_q;        // [d] or null
    const float *sink;           // [H] or null
    double inv_freq[kMaxRopeDims / 2];
};
struct NoV4Args {};

// cos and sin of pos * inv_freq (inv_freq = theta^(-2k/rope_dims), formed on the host in
// double): the angle is formed and reduced modulo 2 pi in double precision, then
// sin/cos are taken in fp32 on the reduced angle (|r| <= pi)
__device__ __forceinline__ void rope_cs(int64_t pos, double inv_freq, float &c, float &s) {
    const double ang = (double)pos * inv_freq;
    const double two_pi = 6.283185307179586476925286766559;
    const double n = rint(ang * (1.0 / two_pi));
    const float r = (float)fma(-two_pi, n, ang);
    sincosf(r, &s, &c);
}

// Row h of Q (128-byte-swizzled, two 64-column blocks) <- R(p) N(q): RMSNorm with
// gamma, then channel pair k of the last rope_dims channels turned by the angle
// (cos, sin)[k] of the query position; one thread per row, in place.
__device__ __forceinline__ void prep_q_row(unsigned char *sQ, int h, const float *s_g, float eps, int rope_dims,
                                           const float *s_cs, const float *s_sn, int q_blk) {
    float ss = 0.f;
#pragma unroll 4
    for (int c = 0; c < kD / 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(sQ + (c >> 3) * q_blk + h * 128 + (((c & 7) ^ (h & 7)) << 4));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
            ss = fmaf(lo, lo, fmaf(hi, hi, ss));
        }
    }
    const float inv = 1.f / sqrtf(ss / (float)kD + eps);
    const int r0 = kD - rope_dims;  // first rotated channel
#pragma unroll 4
    for (int c = 0; c < kD / 8; ++c) {
        unsigned char *ptr = sQ + (c >> 3) * q_blk + h * 128 + (((c & 7) ^ (h & 7)) << 4);
        const uint4 u = *reinterpret_cast<const uint4 *>(ptr);
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int ch = c * 8 + 2 * e;  // channels ch, ch + 1: one rotation pair when ch >= r0
            float x0 = bf16_lo(w[e]) * inv * s_g[ch], x1 = bf16_hi(w[e]) * inv * s_g[ch + 1];
            if (ch >= r0) {
                const int k = (ch - r0) >> 1;
                const float cs = s_cs[k], sn = s_sn[k];
                const float y0 = x0 * cs - x1 * sn;
                x1 = x0 * sn + x1 * cs;
                x0 = y0;
            }
            w[e] = pack_bf16x2(x0, x1);
        }
        *reinterpret_cast<uint4 *>(ptr) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// chunk c (16 bytes) of row r of a 128-byte-swizzled K-major tile made of 64-column blocks
__device__ __forceinline__ uint32_t sw_off(int r, int c, int blk_bytes) {
    return (uint32_t)((c >> 3) * blk_bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}
// float4 chunk c4 of row h of the fp32 partial O staged in shared memory, rotated so
// that the 16 heads a warp stores at once spread over the banks
__device__ __forceinline__ int o_off(int h, int c4) { return h * kD + ((c4 ^ (h & 31)) << 2); }

__device__ __forceinline__ bool wait_phase0(uint64_t *bar) {
    for (unsigned long long i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, 0u)) return true;
    return false;
}

template <bool V4>
__global__ void __launch_bounds__(kThreads, 1)
    attn_decode_tc_kernel(DecodeTcArgs a, typename std::conditional<V4, DecodeV4Args, NoV4Args>::type v4) {
    extern __shared__ __align__(16) unsigned char smem_raw[];  // rounded up to 1024 at run time
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *sQ = smem;
    unsigned char *sK = sQ + kQBytes;
    unsigned char *sV = sK + kTile;
    unsigned char *sP = sV + kTile;
    float *sO = reinterpret_cast<float *>(sK);
    __shared__ uint32_t s_mask[kThreads / 32];
    __shared__ __align__(8) uint64_t bar_s, bar_o;
    __shared__ uint32_t s_tmem;
    // V4: the angles of the query position and gamma_q
    __shared__ float s_cs[V4 ? kMaxRopeDims / 2 : 1], s_sn[V4 ? kMaxRopeDims / 2 : 1], s_g[V4 ? kD : 1];

    const int j = blockIdx.x;  // tile == rank in the cluster
    const int b = blockIdx.y, hg = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(&bar_s, 1);
        mbar_init(&bar_o, 1);
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 256);  // S: columns [0, 128), O: [128, 256)
    // nothing written by the preceding kernel in the stream is read before this
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    // Q of this head group into 128-byte-swizzled K-major rows (cp.async group 0)
    {
        const __nv_bfloat16 *q = a.q + ((int64_t)b * a.H + (int64_t)hg * kH) * kD;
        for (int i = tid; i < kH * 16; i += kThreads) {
            const int h = i >> 4, c = i & 15;
            cp_async_16(smem_u32(sQ + sw_off(h, c, kQBlk)), q + (int64_t)h * kD + c * 8, 16);
        }
        cp_async_commit();
    }
    const int64_t p = a.ctx[b] - 1;
    int64_t E = num_entries(p, a.m);
    if (E > a.E_cap) E = a.E_cap;
    const int slot0 = j * kN;

    // ---- the item this thread resolves: slot slot0 + tid
    const __nv_bfloat16 *ksrc = nullptr, *vsrc = nullptr;
    {
        const int slot = slot0 + tid;
        if (slot < a.topk) {
            // the slot is inside the [B, topk] index array whatever the count: its load
            // goes out beside the count's instead of after it
            const int32_t e_any = a.idx[(int64_t)b * a.topk + slot];
            const int cntb = a.cnt ? min(max(a.cnt[b], 0), a.topk) : a.topk;
            const int32_t e = slot < cntb ? e_any : -1;
            if (e >= E) raise_flag(FLAG_ATTN_INDEX);
            if (e >= 0 && e < E) {
                ksrc = a.kc + (int64_t)b * a.c_sb + (int64_t)e * a.c_se;
                vsrc = a.vc + (int64_t)b * a.c_sb + (int64_t)e * a.c_se;
            }
        } else if (slot < a.topk + a.window) {
            const int64_t t = p - a.window + 1 + (slot - a.topk);
            if (t >= 0 && t <= p) {
                if (t >= a.N_cap) raise_flag(FLAG_ATTN_RANGE);
                else {
                    ksrc = a.k_raw + (int64_t)b * a.r_sb + t * a.r_st;
                    vsrc = a.v_raw + (int64_t)b * a.r_sb + t * a.r_st;
                }
            }
        }
    }
    const uint32_t bits = __ballot_sync(0xffffffffu, ksrc != nullptr);
    if (lane == 0) s_mask[warp] = bits;
    // ---- K rows (cp.async group 1), then V rows (group 2; empty when K and V are one
    // buffer): a half-warp copies one 256-byte row, the row pointer comes by shuffle
    // from the thread that resolved it
    auto gather = [&](unsigned char *dst, const __nv_bfloat16 *src) {
        const unsigned long long sv = reinterpret_cast<unsigned long long>(src);
        const int c = lane & 15;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
            const int rl = 2 * i + (lane >> 4);
            const unsigned long long rs = __shfl_sync(0xffffffffu, sv, rl);
            const int r = warp * 32 + rl;
            const __nv_bfloat16 *rp = reinterpret_cast<const __nv_bfloat16 *>(rs);
            cp_async_16(smem_u32(dst + sw_off(r, c, kTBlk)), rp ? (const void *)(rp + c * 8) : (const void *)a.q,
                        rp ? 16 : 0);  // zero-fill invalid rows
        }
    };
    gather(sK, ksrc);
    cp_async_commit();
    if (!a.shared_kv) gather(sV, vsrc);
    cp_async_commit();
    const unsigned char *tV = a.shared_kv ? sK : sV;
    if constexpr (V4) {
        // R(p) N(q) on Q in shared memory while the K and V rows are in flight
        if (tid < v4.rope_dims / 2) rope_cs(p, v4.inv_freq[tid], s_cs[tid], s_sn[tid]);
        for (int i = tid; i < kD; i += kThreads) s_g[i] = v4.gamma_q ? v4.gamma_q[i] : 1.f;
        cp_async_wait<2>();  // this thread's Q copies (group 0)
        __syncthreads();     // every thread's, the angles and gamma
        if (tid < kH) prep_q_row(sQ, tid, s_g, v4.eps, v4.rope_dims, s_cs, s_sn, kQBlk);
        // (the MMA reads Q through the async proxy: the fence below precedes the barrier)
    }

    // ---- S = Q K^T once Q and every thread's K rows have landed
    cp_async_wait<1>();
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t tS = tmem, tO = tmem + kN;
    if (tid == 0) {
        constexpr uint32_t idS = tc::idesc_bf16(kH, kN, false, false);
        const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t da = tc::desc_sw128(aQ + (kk >> 2) * kQBlk + (kk & 3) * 32, 16, 1024);
            const uint64_t db = tc::desc_sw128(aK + (kk >> 2) * kTBlk + (kk & 3) * 32, 16, 1024);
            tc::mma_bf16(tS, da, db, idS, kk > 0 ? 1u : 0u);
        }
        tc::commit(&bar_s);
    }
    cp_async_wait<0>();  // this thread's V rows
    tc::fence_proxy_async();

    // ---- softmax of the tile: thread (warp w, lane l < 16) owns head h = 16w + l
    bool ok = wait_phase0(&bar_s);
    ok = __syncthreads_and(ok) != 0;  // every thread's V rows, and S, or a give-up
    if (!ok && tid == 0) raise_flag(FLAG_ATTN_RANGE | 0x800u);
    tc::fence_after();
    const bool active = lane < 16;
    const int h = warp * 16 + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float m_tile = -INFINITY, l_tile = 0.f;
    if (ok) {
        uint32_t v[kN];
#pragma unroll
        for (int c = 0; c < kN / 32; ++c) tc::tmem_ld32(tS + lane_off + c * 32, v + c * 32);
        tc::tmem_wait_ld();
        uint32_t mw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) mw[q] = s_mask[q];
        if ((mw[0] & mw[1] & mw[2] & mw[3]) != 0xffffffffu) {
#pragma unroll
            for (int c = 0; c < kN; ++c)
                if (!((mw[c >> 5] >> (c & 31)) & 1u)) v[c] = __float_as_uint(-INFINITY);
        }
        float mx8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx8[q] = -INFINITY;
#pragma unroll
        for (int c = 0; c < kN; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], __uint_as_float(v[c]));
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        m_tile = mx == -INFINITY ? -INFINITY : mx * a.scale_log2;
        const float nm = m_tile == -INFINITY ? 0.f : -m_tile;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        // P = 2^(s * scale_log2 - m) in bf16 (invalid items read -inf: exponent 0)
#pragma unroll
        for (int cc = 0; cc < kN / 8; ++cc) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c0 = cc * 8 + 2 * e;
                const float p0 = tc::ex2(fmaf(__uint_as_float(v[c0]), a.scale_log2, nm));
                const float p1 = tc::ex2(fmaf(__uint_as_float(v[c0 + 1]), a.scale_log2, nm));
                acc[e] += p0 + p1;
                pk[e] = pack_bf16x2(p0, p1);
            }
            if (active)
                *reinterpret_cast<uint4 *>(sP + sw_off(h, cc, kQBlk)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        l_tile = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    // ---- O = P V once every head's P row is in shared memory
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (tid == 0 && ok) {
        constexpr uint32_t idO = tc::idesc_bf16(kH, kD, false, true);
        const uint32_t aP = smem_u32(sP), aV = smem_u32(tV);
#pragma unroll
        for (int kk = 0; kk < kN / 16; ++kk) {
            const uint64_t da = tc::desc_sw128(aP + (kk >> 2) * kQBlk + (kk & 3) * 32, 16, 1024);
            const uint64_t db = tc::desc_sw128(aV + kk * 16 * 128, kTBlk, 1024);
            tc::mma_bf16(tO, da, db, idO, kk > 0 ? 1u : 0u);
        }
        tc::commit(&bar_o);
    }
    bool ok_o = ok ? wait_phase0(&bar_o) : false;
    ok_o = __syncthreads_and(ok_o) != 0;
    if (ok && !ok_o && tid == 0) raise_flag(FLAG_ATTN_RANGE | 0x800u);
    tc::fence_after();
    // ---- this CTA's partial: unnormalised O, staged in the K tile (free now) and
    // written to the workspace with coalesced stores, maximum and sum
    const int S = a.n_tiles;
    const int64_t blk = ((int64_t)b * (a.H / kH) + hg) * S;  // partials of (sequence, head group)
    if (ok_o) {
        uint32_t o[kD];
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) tc::tmem_ld32(tO + lane_off + c * 32, o + c * 32);
        tc::tmem_wait_ld();
        if (active) {
#pragma unroll
            for (int c4 = 0; c4 < kD / 4; ++c4)
                *reinterpret_cast<float4 *>(sO + o_off(h, c4)) =
                    make_float4(__uint_as_float(o[4 * c4]), __uint_as_float(o[4 * c4 + 1]),
                                __uint_as_float(o[4 * c4 + 2]), __uint_as_float(o[4 * c4 + 3]));
        }
    }
    if (active) {  // a CTA that gave up contributes nothing (its O is never read)
        float *pml = a.part_ml + (blk + j) * (2 * kH);
        pml[h] = ok_o ? m_tile : -INFINITY;
        pml[kH + h] = ok_o ? l_tile : 0.f;
    }
    __syncthreads();
    if (ok_o) {
        float *po = a.part_o + (blk + j) * (kH * kD);
        for (int hr = warp; hr < kH; hr += kThreads / 32)  // warp w: rows w, w + 4, ...; lane: chunk
            *reinterpret_cast<float4 *>(po + hr * kD + lane * 4) =
                *reinterpret_cast<const float4 *>(sO + o_off(hr, lane));
    }
    cluster_sync_all();  // every partial of the cluster is written

    // ---- combine heads [j * hpc, (j + 1) * hpc) over the n_tiles partials (from L2);
    // all loads of a thread are issued before any is used
    const int hpc = (kH + S - 1) / S;
    const int h_lo = j * hpc, h_hi = min(kH, h_lo + hpc);
    const int work = h_hi > h_lo ? (h_hi - h_lo) * (kD / 4) : 0;
    for (int w = tid; w < work; w += kThreads) {
        const int hl = h_lo + w / (kD / 4);  // head within the group
        const int c4 = w % (kD / 4);
        float mv[kMaxTiles], lv[kMaxTiles];
        float4 ov[kMaxTiles];
#pragma unroll
        for (int r = 0; r < kMaxTiles; ++r) {
            if (r < S) {
                const float *pml = a.part_ml + (blk + r) * (2 * kH);
                mv[r] = __ldcg(pml + hl);
                lv[r] = __ldcg(pml + kH + hl);
                ov[r] = __ldcg(reinterpret_cast<const float4 *>(a.part_o + (blk + r) * (kH * kD) + hl * kD) + c4);
            } else {
                mv[r] = -INFINITY;
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < kMaxTiles; ++r) M = fmaxf(M, mv[r]);
        float Lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
            for (int r = 0; r < kMaxTiles; ++r) {
                if (mv[r] == -INFINITY) continue;  // nothing valid there (its O is not read)
                const float wgt = tc::ex2(mv[r] - M);
                Lsum = fmaf(wgt, lv[r], Lsum);
                acc.x = fmaf(wgt, ov[r].x, acc.x);
                acc.y = fmaf(wgt, ov[r].y, acc.y);
                acc.z = fmaf(wgt, ov[r].z, acc.z);
                acc.w = fmaf(wgt, ov[r].w, acc.w);
            }
        }
        const int hh = hg * kH + hl;
        __nv_bfloat16 *out = a.out + ((int64_t)b * a.H + hh) * kD + c4 * 4;
        if constexpr (!V4) {
            const bool empty = !(Lsum > 0.f);
            const float inv = empty ? 0.f : 1.f / Lsum;
            uint2 pk;
            pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2 *>(out) = pk;
            if (a.lse && c4 == 0) a.lse[(int64_t)b * a.H + hh] = empty ? -INFINITY : (M + log2f(Lsum)) * kLn2;
        } else {
            // the sink's logit z joins the denominator (e^z = 2^(z log2 e)), then the
            // output turns back by the query's position, R(-p)
            float Mx = M, Lt = Lsum, wa = 1.f;
            if (v4.sink) {
                const float zl = v4.sink[hh] * kLog2e;
                Mx = fmaxf(M, zl);
                wa = M == -INFINITY ? 0.f : tc::ex2(M - Mx);
                Lt = Lsum * wa + tc::ex2(zl - Mx);
            }
            const bool empty = !(Lt > 0.f);
            const float inv = empty ? 0.f : wa / Lt;
            float o4[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const int ch = c4 * 4 + e, r0 = kD - v4.rope_dims;
                if (ch >= r0) {
                    const int k = (ch - r0) >> 1;
                    const float cs = s_cs[k], sn = s_sn[k];
                    const float y0 = o4[e] * cs + o4[e + 1] * sn;
                    o4[e + 1] = -o4[e] * sn + o4[e + 1] * cs;
                    o4[e] = y0;
                }
            }
            uint2 pk;
            pk.x = pack_bf16x2(o4[0], o4[1]);
            pk.y = pack_bf16x2(o4[2], o4[3]);
            *reinterpret_cast<uint2 *>(out) = pk;
            if (a.lse && c4 == 0) a.lse[(int64_t)b * a.H + hh] = empty ? -INFINITY : (Mx + log2f(Lt)) * kLn2;
        }
    }
    // after a give-up, let this CTA's MMAs finish (again bounded) before TMEM is freed
    if (tid == 0 && !ok) wait_phase0(&bar_s);
    if (tid == 0 && ok && !ok_o) wait_phase0(&bar_o);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

}  // namespace

bool decode_tc_shape(int H, int d, int topk, int window) {
    return d == kD && H > 0 && H % kH == 0 && topk > 0 && window >= 0 && topk + window <= kMaxTiles * kN;
}

DecodeTcWorkspace decode_tc_workspace(int B, int H, int topk, int window) {
    DecodeTcWorkspace w;
    const size_t parts = (size_t)B * (H / kH) * ((topk + window + kN - 1) / kN);
    w.off_o = 0;
    w.off_ml = (parts * kH * kD * sizeof(float) + 255) & ~(size_t)255;
    w.total = w.off_ml + ((parts * 2 * kH * sizeof(float) + 255) & ~(size_t)255);
    return w;
}

bool decode_tc_supported(const AttnArgs &a) {
    return decode_tc_shape(a.H, a.d, a.topk, a.window) && a.idx != nullptr && a.T == 1 && a.pos_is_ctx &&
           a.part_o != nullptr && a.part_lse != nullptr;
}

cudaError_t launch_attn_decode_tc(const AttnArgs &a, cudaStream_t s) {
    DecodeTcArgs g;
    g.B = a.rows;
    g.H = a.H;
    g.topk = a.topk;
    g.window = a.window;
    g.m = a.m;
    g.n_tiles = (a.topk + a.window + kN - 1) / kN;
    g.shared_kv = a.shared_kv;
    g.E_cap = a.E_cap;
    g.N_cap = a.N_cap;
    g.c_sb = a.c_sb;
    g.c_se = a.c_se;
    g.r_sb = a.r_sb;
    g.r_st = a.r_st;
    g.ctx = a.pos;
    g.idx = a.idx;
    g.cnt = a.cnt;
    g.q = static_cast<const __nv_bfloat16 *>(a.q);
    g.kc = static_cast<const __nv_bfloat16 *>(a.kc);
    g.vc = static_cast<const __nv_bfloat16 *>(a.vc);
    g.k_raw = static_cast<const __nv_bfloat16 *>(a.k_raw);
    g.v_raw = static_cast<const __nv_bfloat16 *>(a.v_raw);
    g.scale_log2 = a.scale * kLog2e;
    g.out = static_cast<__nv_bfloat16 *>(a.out);
    g.lse = a.lse;
    g.part_o = a.part_o;
    g.part_ml = a.part_lse;
    static unsigned long long done = 0, np_done = 0, done4 = 0, np_done4 = 0;
    auto prepare = [&](auto kern, unsigned long long &dn, unsigned long long &npd) {
        cudaError_t e = smem_limit_once(kern, (int)kSmemBytes, dn);
        if (e != cudaSuccess) return e;
        if (g.n_tiles > 8) {
            int dev = 0;
            cudaGetDevice(&dev);
            const unsigned long long bit = 1ull << (dev & 63);
            if (!(npd & bit)) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e != cudaSuccess) return e;
                npd |= bit;
            }
        }
        return cudaSuccess;
    };
    cudaError_t e = a.v4 ? prepare(attn_decode_tc_kernel<true>, done4, np_done4)
                         : prepare(attn_decode_tc_kernel<false>, done, np_done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.n_tiles, a.rows, a.H / kH);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = g.n_tiles;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // the launch may overlap the tail of the previous kernel in the stream (set-up
    // only: every CTA waits for that kernel's completion before reading inputs)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (!a.v4) return cudaLaunchKernelEx(&cfg, attn_decode_tc_kernel<false>, g, NoV4Args{});
    DecodeV4Args v;
    v.rope_dims = a.rope_dims;
    v.eps = a.eps;
    v.gamma_q = a.gamma_q;
    v.sink = a.sink;
    for (int k = 0; k < kMaxRopeDims / 2; ++k) v.inv_freq[k] = a.inv_freq[k];
    return cudaLaunchKernelEx(&cfg, attn_decode_tc_kernel<true>, g, v);
}

}  // namespace hsa
