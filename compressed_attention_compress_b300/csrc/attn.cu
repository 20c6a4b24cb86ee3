// Attention over the hybrid set: selected (CSA) or all (HCA) compressed entries
// plus the raw sliding window, in one softmax per head.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制: CSA step 3 (Multi-Query
// Attention over the top-k compressed blocks), the HCA paragraph (dense over all
// compressed entries) and the sliding-window paragraph (the most recent 128 raw
// tokens join; compressed attention only sees complete blocks).
//
// A row is one query token with H heads sharing one KV head (MQA), so the H
// heads form the M dimension of the tensor-core tiles: S = Q[H x d] K^T[d x NT],
// online softmax in registers, O += P V.  The row's item list (entries, then
// window tokens) is cut into splits; each CTA handles one (split, row), gathers
// its items with cp.async into swizzled shared memory (double-buffered) and
// writes either the final output (one split) or an fp32 partial (o, lse) that
// the merge kernel combines with the log-sum-exp rule.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace hsa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct RowSet {
    int b;
    int64_t p, E, win0;
    int n_slots, n_win, n_items, n_splits;
};

__device__ __forceinline__ RowSet row_set(const AttnArgs &a, int row) {
    RowSet r;
    r.b = row / a.T;
    const int t = row - r.b * a.T;
    r.p = a.pos_is_ctx ? a.pos[r.b] - 1 : a.pos[r.b] + t;
    r.E = num_entries(r.p, a.m);
    if (r.E > a.E_cap) r.E = a.E_cap;
    const int64_t nw = r.p + 1 < (int64_t)a.window ? r.p + 1 : (int64_t)a.window;
    r.n_win = nw < 0 ? 0 : (int)nw;
    r.win0 = r.p - r.n_win + 1;
    if (a.idx) {
        int c = a.topk;
        if (a.cnt) {
            c = a.cnt[row];
            c = c < 0 ? 0 : (c > a.topk ? a.topk : c);
        }
        r.n_slots = c;
    } else {
        r.n_slots = (int)r.E;
    }
    r.n_items = r.n_slots + r.n_win;
    r.n_splits = a.split > 0 ? (r.n_items + a.split - 1) / a.split : 1;
    if (r.n_splits < 1) r.n_splits = 1;
    return r;
}

// Resolve item i of a row to an element offset of its K/V row, or -1 if masked.
// `raw` tells whether it comes from the raw cache.
__device__ __forceinline__ int64_t resolve_item(const AttnArgs &a, const RowSet &r, int row, int i, bool &raw) {
    if (i < r.n_slots) {
        raw = false;
        int64_t j = a.idx ? (int64_t)a.idx[(int64_t)row * a.topk + i] : (int64_t)i;
        if (j < 0) return -1;
        if (j >= r.E) {
            raise_flag(FLAG_ATTN_INDEX);
            return -1;
        }
        return r.b * a.c_sb + j * a.c_se;
    }
    raw = true;
    const int64_t t = r.win0 + (i - r.n_slots);
    if (t < 0 || t >= a.N_cap) {
        raise_flag(FLAG_ATTN_RANGE);
        return -1;
    }
    return r.b * a.r_sb + t * a.r_st;
}

// ------------------------------------------------------------ bf16 MMA path

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float *c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `c` of row `i` in a swizzled [rows][D] bf16 tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int i, int c) {
    return (uint32_t)(i * (D * 2) + ((c ^ (i & 7)) << 4));
}

template <int D, int NT, int NW>
__global__ void __launch_bounds__(NW * 32) attn_bf16_kernel(AttnArgs a) {
    constexpr int NTHR = NW * 32;
    constexpr int CH = D / 8;  // 16-byte chunks per row
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *sQ = smem;                                  // [NW*16][D]
    unsigned char *sK = sQ + NW * 16 * D * 2;                  // [2][NT][D]
    unsigned char *sV = sK + 2 * NT * D * 2;                   // [2][NT][D]
    int64_t *sOffK = reinterpret_cast<int64_t *>(sV + 2 * NT * D * 2);  // [2][NT]
    unsigned char *sRaw = reinterpret_cast<unsigned char *>(sOffK + 2 * NT);  // [2][NT]

    const int row = blockIdx.y;
    const RowSet r = row_set(a, row);
    const int split = blockIdx.x;
    if (split >= r.n_splits) return;
    const int i_begin = a.split > 0 ? split * a.split : 0;
    const int i_end = a.split > 0 ? min(r.n_items, i_begin + a.split) : r.n_items;
    const int ntiles = (i_end - i_begin + NT - 1) / NT;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const __nv_bfloat16 *kc = static_cast<const __nv_bfloat16 *>(a.kc);
    const __nv_bfloat16 *vc = static_cast<const __nv_bfloat16 *>(a.vc);
    const __nv_bfloat16 *kr = static_cast<const __nv_bfloat16 *>(a.k_raw);
    const __nv_bfloat16 *vr = static_cast<const __nv_bfloat16 *>(a.v_raw);

    // Q tile of this row (heads >= H are zero; H is a multiple of 16 here)
    {
        const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q) + (int64_t)row * a.H * D;
        for (int c = tid; c < NW * 16 * CH; c += NTHR) {
            const int h = c / CH, cc = c % CH;
            cp_async_16(smem_u32(sQ + swz<D>(h, cc)), q + (int64_t)h * D + cc * 8, h < a.H ? 16 : 0);
        }
    }

    auto resolve_tile = [&](int tile, int buf) {
        for (int it = tid; it < NT; it += NTHR) {
            const int i = i_begin + tile * NT + it;
            int64_t off = -1;
            bool raw = false;
            if (i < i_end) off = resolve_item(a, r, row, i, raw);
            sOffK[buf * NT + it] = off;
            sRaw[buf * NT + it] = raw;
        }
    };
    auto issue_tile = [&](int buf) {
        for (int c = tid; c < NT * CH; c += NTHR) {
            const int it = c / CH, cc = c % CH;
            const int64_t off = sOffK[buf * NT + it];
            const bool raw = sRaw[buf * NT + it];
            const __nv_bfloat16 *ks = (raw ? kr : kc) + (off < 0 ? 0 : off) + cc * 8;
            const __nv_bfloat16 *vs = (raw ? vr : vc) + (off < 0 ? 0 : off) + cc * 8;
            const int nb = off < 0 ? 0 : 16;
            cp_async_16(smem_u32(sK + buf * NT * D * 2 + swz<D>(it, cc)), ks, nb);
            cp_async_16(smem_u32(sV + buf * NT * D * 2 + swz<D>(it, cc)), vs, nb);
        }
    };

    if (ntiles > 0) resolve_tile(0, 0);
    __syncthreads();
    if (ntiles > 0) issue_tile(0);
    cp_async_commit();  // group: Q (+ tile 0)

    // per-thread state: rows g and g+8 of this warp's 16 heads
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY};
    float lrow[2] = {0.f, 0.f};
    uint32_t qa[D / 16][4];
    const float sl2 = a.scale * kLog2e;

    for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = tile & 1;
        if (tile + 1 < ntiles) resolve_tile(tile + 1, buf ^ 1);
        __syncthreads();
        if (tile + 1 < ntiles) issue_tile(buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (tile == 0) {
            // Q fragments (A operand) for this warp's 16 heads
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int q = lane >> 3, rr = lane & 7;
                const int h = warp * 16 + (q & 1) * 8 + rr;
                ldsm_x4(smem_u32(sQ + swz<D>(h, 2 * kk + (q >> 1))), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
            }
        }
        const unsigned char *tK = sK + buf * NT * D * 2;
        const unsigned char *tV = sV + buf * NT * D * 2;
        // S = Q K^T  (16 x NT per warp)
        float s[NT / 8][4];
#pragma unroll
        for (int n = 0; n < NT / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int n = 0; n < NT / 8; ++n) {
#pragma unroll
            for (int kk = 0; kk < D / 16; kk += 2) {
                const int q = lane >> 3, rr = lane & 7;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(tK + swz<D>(n * 8 + rr, 2 * kk + q)), b0, b1, b2, b3);
                mma_bf16(s[n], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma_bf16(s[n], qa[kk + 1][0], qa[kk + 1][1], qa[kk + 1][2], qa[kk + 1][3], b2, b3);
            }
        }
        // mask + online softmax (log2 domain)
        const int tq = lane & 3;
        float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < NT / 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = n * 8 + 2 * tq + (e & 1);
                const bool valid = sOffK[buf * NT + col] >= 0;
                const float x = valid ? s[n][e] * sl2 : -INFINITY;
                s[n][e] = x;
                tmax[e >> 1] = fmaxf(tmax[e >> 1], x);
            }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 1));
            tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 2));
        }
        float alpha[2], mnew[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            mnew[hh] = fmaxf(mrow[hh], tmax[hh]);
            alpha[hh] = mnew[hh] == -INFINITY ? 1.f : exp2f(mrow[hh] - mnew[hh]);
            mrow[hh] = mnew[hh];
        }
        float psum[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < NT / 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hh = e >> 1;
                const float pv = mnew[hh] == -INFINITY ? 0.f : exp2f(s[n][e] - mnew[hh]);
                s[n][e] = pv;
                psum[hh] += pv;
            }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) lrow[hh] = lrow[hh] * alpha[hh] + psum[hh];
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            o[n][0] *= alpha[0];
            o[n][1] *= alpha[0];
            o[n][2] *= alpha[1];
            o[n][3] *= alpha[1];
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < NT / 16; ++kk) {
            const uint32_t pa0 = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
            const uint32_t pa1 = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
            const uint32_t pa2 = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            const uint32_t pa3 = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int n = 0; n < D / 8; n += 2) {
                const int q = lane >> 3, rr = lane & 7;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(smem_u32(tV + swz<D>(kk * 16 + (q & 1) * 8 + rr, n + (q >> 1))), b0, b1, b2, b3);
                mma_bf16(o[n], pa0, pa1, pa2, pa3, b0, b1);
                mma_bf16(o[n + 1], pa0, pa1, pa2, pa3, b2, b3);
            }
        }
        __syncthreads();  // this buffer is refilled two iterations later
    }
    cp_async_wait<0>();

    // finalize: reduce l over the quad, normalise, write
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        lrow[hh] += __shfl_xor_sync(0xffffffffu, lrow[hh], 1);
        lrow[hh] += __shfl_xor_sync(0xffffffffu, lrow[hh], 2);
    }
    const int g = lane >> 2, tq = lane & 3;
    const bool direct = r.n_splits == 1;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int h = warp * 16 + g + hh * 8;
        if (h >= a.H) continue;
        const bool empty = lrow[hh] == 0.f;
        const float inv = empty ? 0.f : 1.f / lrow[hh];
        const float lse = empty ? -INFINITY : (mrow[hh] + log2f(lrow[hh])) * kLn2;
        if (direct) {
            __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + ((int64_t)row * a.H + h) * D;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                const uint32_t v = pack_bf16x2(o[n][2 * hh] * inv, o[n][2 * hh + 1] * inv);
                *reinterpret_cast<uint32_t *>(out + n * 8 + 2 * tq) = v;
            }
            if (a.lse && tq == 0) a.lse[(int64_t)row * a.H + h] = lse;
        } else {
            float *po = a.part_o + (((int64_t)row * a.max_splits + split) * a.H + h) * D;
#pragma unroll
            for (int n = 0; n < D / 8; ++n)
                *reinterpret_cast<float2 *>(po + n * 8 + 2 * tq) = make_float2(o[n][2 * hh] * inv, o[n][2 * hh + 1] * inv);
            if (tq == 0) a.part_lse[((int64_t)row * a.max_splits + split) * a.H + h] = lse;
        }
    }
}

template <int D, int NT, int NW>
cudaError_t launch_bf16_t(const AttnArgs &a, cudaStream_t s) {
    const size_t smem = (size_t)NW * 16 * D * 2 + 4 * (size_t)NT * D * 2 + 2 * NT * sizeof(int64_t) + 2 * NT;
    static unsigned long long done = 0;
    cudaError_t e = smem_limit_once(attn_bf16_kernel<D, NT, NW>, (int)smem, done);
    if (e != cudaSuccess) return e;
    const int splits = a.split > 0 ? a.max_splits : 1;
    dim3 grid(splits, a.rows);
    attn_bf16_kernel<D, NT, NW><<<grid, NW * 32, smem, s>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bf16_d(const AttnArgs &a, cudaStream_t s) {
    switch (a.H / 16) {
        case 1: return launch_bf16_t<D, 64, 1>(a, s);
        case 2: return launch_bf16_t<D, 64, 2>(a, s);
        case 3: return launch_bf16_t<D, 64, 3>(a, s);
        case 4: return launch_bf16_t<D, 64, 4>(a, s);
        case 5: return launch_bf16_t<D, 64, 5>(a, s);
        case 6: return launch_bf16_t<D, 64, 6>(a, s);
        case 7: return launch_bf16_t<D, 64, 7>(a, s);
        case 8: return launch_bf16_t<D, 64, 8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------ fp32 SIMT path
// One warp per (row, head); lanes own items for the logits and channels for the
// output.  Used for fp32 storage (exactness over speed).
template <int D>
__global__ void __launch_bounds__(128) attn_f32_kernel(AttnArgs a) {
    constexpr int CPL = D / 32;  // channels per lane
    const int warp_global = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (warp_global >= a.rows * a.H) return;
    const int row = warp_global / a.H, h = warp_global % a.H;
    const RowSet r = row_set(a, row);
    const float *q = static_cast<const float *>(a.q) + ((int64_t)row * a.H + h) * D;
    const float *kc = static_cast<const float *>(a.kc), *vc = static_cast<const float *>(a.vc);
    const float *kr = static_cast<const float *>(a.k_raw), *vr = static_cast<const float *>(a.v_raw);
    float qreg[D];
#pragma unroll
    for (int c = 0; c < D; ++c) qreg[c] = q[c];
    float o[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) o[c] = 0.f;
    float m = -INFINITY, l = 0.f;
    for (int i0 = 0; i0 < r.n_items; i0 += 32) {
        const int i = i0 + lane;
        bool raw = false;
        int64_t off = -1;
        if (i < r.n_items) off = resolve_item(a, r, row, i, raw);
        float x = -INFINITY;
        if (off >= 0) {
            const float *kk = (raw ? kr : kc) + off;
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) acc = fmaf(qreg[c], kk[c], acc);
            x = acc * a.scale;
        }
        float cmax = x;
#pragma unroll
        for (int o_ = 16; o_ > 0; o_ >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o_));
        const float mnew = fmaxf(m, cmax);
        if (mnew == -INFINITY) continue;
        const float alpha = expf(m - mnew);
        const float pv = off >= 0 ? expf(x - mnew) : 0.f;
        float psum = pv;
#pragma unroll
        for (int o_ = 16; o_ > 0; o_ >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o_);
        l = l * alpha + psum;
        m = mnew;
#pragma unroll
        for (int c = 0; c < CPL; ++c) o[c] *= alpha;
        const int nvalid = min(32, r.n_items - i0);
        for (int x_ = 0; x_ < nvalid; ++x_) {
            const float px = __shfl_sync(0xffffffffu, pv, x_);
            const int64_t ox = __shfl_sync(0xffffffffu, off, x_);
            const bool rx = __shfl_sync(0xffffffffu, (int)raw, x_);
            if (ox < 0 || px == 0.f) continue;
            const float *vv = (rx ? vr : vc) + ox;
#pragma unroll
            for (int c = 0; c < CPL; ++c) o[c] = fmaf(px, vv[lane + 32 * c], o[c]);
        }
    }
    const bool empty = l == 0.f;
    const float inv = empty ? 0.f : 1.f / l;
    float *out = static_cast<float *>(a.out) + ((int64_t)row * a.H + h) * D;
#pragma unroll
    for (int c = 0; c < CPL; ++c) out[lane + 32 * c] = o[c] * inv;
    if (a.lse && lane == 0) a.lse[(int64_t)row * a.H + h] = empty ? -INFINITY : m + logf(l);
}

// ------------------------------------------------------------ split merge
// out = sum_s exp(lse_s - lse) * o_s,  lse = ln sum_s exp(lse_s)  (rows with >1 split).
// One warp per (row, head): lanes own 4 channels each (d <= 128) and the split
// weights are computed once per warp; the loads of all splits are independent.
template <typename OutT>
__global__ void __launch_bounds__(128) attn_merge_kernel(AttnArgs a) {
    const int row = blockIdx.y;
    const int h = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (h >= a.H) return;
    const RowSet r = row_set(a, row);
    if (r.n_splits <= 1) return;
    const int D = a.d;
    const float *pl = a.part_lse + (int64_t)row * a.max_splits * a.H + h;
    float M = -INFINITY;
    for (int sp = lane; sp < r.n_splits; sp += 32) M = fmaxf(M, pl[(int64_t)sp * a.H]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int sp = lane; sp < r.n_splits; sp += 32) {
        const float ls = pl[(int64_t)sp * a.H];
        L += ls == -INFINITY ? 0.f : expf(ls - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const bool empty = M == -INFINITY || L == 0.f;
    const float invL = empty ? 0.f : 1.f / L;
    for (int c4 = lane; c4 < D / 4; c4 += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!empty) {
            const float *po = a.part_o + ((int64_t)row * a.max_splits * a.H + h) * D + c4 * 4;
#pragma unroll 4
            for (int sp = 0; sp < r.n_splits; ++sp) {
                const float ls = pl[(int64_t)sp * a.H];
                const float wgt = ls == -INFINITY ? 0.f : expf(ls - M) * invL;
                const float4 v = *reinterpret_cast<const float4 *>(po + (int64_t)sp * a.H * D);
                acc.x = fmaf(wgt, v.x, acc.x);
                acc.y = fmaf(wgt, v.y, acc.y);
                acc.z = fmaf(wgt, v.z, acc.z);
                acc.w = fmaf(wgt, v.w, acc.w);
            }
        }
        OutT *out = static_cast<OutT *>(a.out) + ((int64_t)row * a.H + h) * D + c4 * 4;
        if constexpr (sizeof(OutT) == 2) {
            uint2 pk;
            pk.x = pack_bf16x2(acc.x, acc.y);
            pk.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2 *>(out) = pk;
        } else {
            *reinterpret_cast<float4 *>(out) = acc;
        }
    }
    if (a.lse && lane == 0) a.lse[(int64_t)row * a.H + h] = empty ? -INFINITY : M + logf(L);
}

}  // namespace

int attn_split_size(bool bf16, bool dense, int H, int rows, int64_t max_items, int num_sms) {
    if (!bf16) return 0;
    // aim for about two CTAs per SM over the whole batch; splits are whole tiles
    int64_t want_ctas = 2ll * num_sms;
    int64_t per = (max_items * rows + want_ctas - 1) / want_ctas;
    int split = 64;
    while (split < 4096 && split < per) split <<= 1;
    (void)dense;
    (void)H;
    return split;
}

cudaError_t launch_attn_bf16(const AttnArgs &a, cudaStream_t s) {
    if (a.d == 128) return launch_bf16_d<128>(a, s);
    if (a.d == 64) return launch_bf16_d<64>(a, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_f32(const AttnArgs &a, cudaStream_t s) {
    const int64_t warps = (int64_t)a.rows * a.H;
    const int grid = (int)((warps + 3) / 4);
    switch (a.d) {
        case 32: attn_f32_kernel<32><<<grid, 128, 0, s>>>(a); break;
        case 64: attn_f32_kernel<64><<<grid, 128, 0, s>>>(a); break;
        case 96: attn_f32_kernel<96><<<grid, 128, 0, s>>>(a); break;
        case 128: attn_f32_kernel<128><<<grid, 128, 0, s>>>(a); break;
        case 160: attn_f32_kernel<160><<<grid, 128, 0, s>>>(a); break;
        case 192: attn_f32_kernel<192><<<grid, 128, 0, s>>>(a); break;
        case 224: attn_f32_kernel<224><<<grid, 128, 0, s>>>(a); break;
        case 256: attn_f32_kernel<256><<<grid, 128, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_attn_merge(const AttnArgs &a, bool bf16, cudaStream_t s) {
    if (a.split <= 0) return cudaSuccess;
    dim3 grid((a.H + 3) / 4, a.rows);
    if (bf16)
        attn_merge_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a);
    else
        attn_merge_kernel<float><<<grid, 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace hsa
