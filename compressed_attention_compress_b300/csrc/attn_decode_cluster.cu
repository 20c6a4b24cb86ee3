// Decode attention (one query token per sequence), bf16: one thread-block
// cluster per sequence.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制: CSA step 3 (MQA over the
// selected compressed entries), the HCA paragraph (dense over every entry) and
// the sliding-window paragraph (the most recent raw tokens join the same softmax).
//
// The sequence's items (selected or all entries, then the window tokens) are cut
// into S equal slices, one per CTA of an S-CTA cluster; heads are taken in groups
// of at most 64, one cluster per (sequence, head group).  Each CTA gathers its
// slice with cp.async into swizzled shared memory, runs the H heads as the M
// dimension of bf16 tensor-core tiles (S = Q K^T, online softmax, O += P V) and
// leaves its unnormalised partial (o, running max, running sum) in its own
// shared memory.  After a cluster barrier, CTA r combines heads
// [r*H/S, (r+1)*H/S) of all S partials through distributed shared memory with
// the log-sum-exp rule and writes the output.  No partial ever goes to global
// memory and no second kernel runs.  The slice layout depends only on the
// sequence itself, so each sequence's output is independent of the batch.
//
// For CSA the item space is static (topk slots + window slots; slots past cnt
// or holding -1 are masked), so the index loads are issued together with the
// position load, one memory round trip before the gathers.  When the caller
// passes one buffer as both K and V (V4's shared key/value entry), only one copy
// of each item is gathered.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace hsa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kStage = 64;  // items per copy stage

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
template <int D>
__device__ __forceinline__ uint32_t swz(int i, int c) {
    return (uint32_t)(i * (D * 2) + ((c ^ (i & 7)) << 4));
}

template <int D, int NW>
struct Smem {
    static constexpr int kQ = NW * 16 * D * 2;          // Q tile, bf16
    static constexpr int kKV = 2 * 2 * kStage * D * 2;  // K and V stages, double-buffered, bf16
    static constexpr int kO = NW * 16 * D * 4;          // fp32 partial O (reuses Q + KV)
    static constexpr int kMain = (kQ + kKV) > kO ? (kQ + kKV) : kO;
    static constexpr int kML = kMain;                    // float m[NW*16], l[NW*16]
    static constexpr int kTab = kML + 2 * NW * 16 * 4;  // int64 item table [per_max]
    static int total(int per_max) { return kTab + per_max * 8; }
};

template <int D, int NW, int S>
__global__ void __launch_bounds__(NW * 32) attn_decode_cluster_kernel(AttnArgs a) {
    constexpr int NTHR = NW * 32;
    constexpr int CH = D / 8;
    constexpr int HR = NW * 16;  // head rows (== H)
    using L = Smem<D, NW>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *sQ = smem;
    unsigned char *sK = smem + L::kQ;
    unsigned char *sV = sK + 2 * kStage * D * 2;
    float *sO = reinterpret_cast<float *>(smem);
    float *sM = reinterpret_cast<float *>(smem + L::kML);
    float *sL = sM + HR;
    int64_t *sTab = reinterpret_cast<int64_t *>(smem + L::kTab);  // offset | raw flag, or -1

    const int row = blockIdx.y;
    const int h0 = blockIdx.z * HR;  // this cluster's head group
    const int split = (int)cluster_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = row;  // decode: one query per sequence
    const bool dense = a.idx == nullptr;
    // launched with programmatic stream serialization: wait until the preceding grid
    // (normally the indexer) has completed and its writes are visible, before any
    // input is read (a no-op when there is no such dependency)
    asm volatile("griddepcontrol.wait;\n" ::: "memory");

    // ---- first round trip: Q, position, count and (CSA) this slice's indices
    {
        const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q) + ((int64_t)row * a.H + h0) * D;
        for (int c = tid; c < HR * CH; c += NTHR) {
            const int h = c / CH, cc = c % CH;
            cp_async_16(smem_u32(sQ + swz<D>(h, cc)), q + (int64_t)h * D + cc * 8, 16);
        }
        cp_async_commit();
    }
    const int64_t p = a.pos[b] - 1;  // decode: ctx_len - 1
    const int cnt = (!dense && a.cnt) ? a.cnt[b] : a.topk;
    int64_t E = num_entries(p, a.m);
    if (E > a.E_cap) E = a.E_cap;
    const int n_win = (int)(p + 1 < (int64_t)a.window ? (p + 1 < 0 ? 0 : p + 1) : a.window);
    // CSA: static slots [0, topk) + [topk, topk + window); HCA: [0, E) + window
    const int64_t n_ent_slots = dense ? E : a.topk;
    const int64_t total = n_ent_slots + (dense ? n_win : a.window);
    int per = (int)((total + S - 1) / S);
    per = (per + 15) / 16 * 16;
    const int64_t i_begin = (int64_t)split * per;
    const int n_my = (int)(i_begin >= total ? 0 : (total - i_begin < per ? total - i_begin : per));
    constexpr int64_t kRawBit = 1ll << 62;
    for (int it = tid; it < n_my; it += NTHR) {
        const int64_t i = i_begin + it;
        int64_t ent = -1;
        if (i < n_ent_slots) {
            int64_t j = i;
            if (!dense) {
                const int32_t jl = a.idx[(int64_t)b * a.topk + i];  // issued before cnt/pos are known
                j = (i < cnt) ? (int64_t)jl : -1;
            }
            if (j >= E) {
                raise_flag(FLAG_ATTN_INDEX);
                j = -1;
            }
            if (j >= 0) ent = (int64_t)b * a.c_sb + j * a.c_se;
        } else {
            const int64_t wslot = i - n_ent_slots;
            const int64_t t = dense ? p - n_win + 1 + wslot : p - a.window + 1 + wslot;
            if (t >= 0 && t <= p) {
                if (t >= a.N_cap) raise_flag(FLAG_ATTN_RANGE);
                else ent = ((int64_t)b * a.r_sb + t * a.r_st) | kRawBit;
            }
        }
        sTab[it] = ent;
    }
    __syncthreads();

    const __nv_bfloat16 *kc = static_cast<const __nv_bfloat16 *>(a.kc);
    const __nv_bfloat16 *vc = static_cast<const __nv_bfloat16 *>(a.vc);
    const __nv_bfloat16 *kr = static_cast<const __nv_bfloat16 *>(a.k_raw);
    const __nv_bfloat16 *vr = static_cast<const __nv_bfloat16 *>(a.v_raw);
    const int nst = (n_my + kStage - 1) / kStage;
    auto issue_stage = [&](int st) {
        if (st < nst) {
            const int buf = st & 1;
            for (int c = tid; c < kStage * CH; c += NTHR) {
                const int it = c / CH, cc = c % CH;
                const int ii = st * kStage + it;
                const int64_t ent = ii < n_my ? sTab[ii] : -1;
                const bool raw = ent >= 0 && (ent & kRawBit);
                const int64_t off = ent < 0 ? 0 : (ent & ~kRawBit);
                const int nb = ent < 0 ? 0 : 16;
                cp_async_16(smem_u32(sK + buf * kStage * D * 2 + swz<D>(it, cc)), (raw ? kr : kc) + off + cc * 8, nb);
                if (!a.shared_kv)  // one entry as key and value: the K copy serves both
                    cp_async_16(smem_u32(sV + buf * kStage * D * 2 + swz<D>(it, cc)), (raw ? vr : vc) + off + cc * 8,
                                nb);
            }
        }
        cp_async_commit();
    };
    issue_stage(0);
    issue_stage(1);

    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY};
    float lrow[2] = {0.f, 0.f};
    uint32_t qa[D / 16][4];
    const float sl2 = a.scale * kLog2e;

    cp_async_wait<2>();  // Q has landed
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int q = lane >> 3, rr = lane & 7;
        const int h = warp * 16 + (q & 1) * 8 + rr;
        ldsm_x4(smem_u32(sQ + swz<D>(h, 2 * kk + (q >> 1))), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }

    for (int st = 0; st < nst; ++st) {
        const int buf = st & 1;
        const int n_valid = min(kStage, n_my - st * kStage);  // items of this stage (CTA-uniform)
        cp_async_wait<1>();
        __syncthreads();
        const unsigned char *tK = sK + buf * kStage * D * 2;
        const unsigned char *tV = a.shared_kv ? tK : sV + buf * kStage * D * 2;
        float s[kStage / 8][4];
#pragma unroll
        for (int n = 0; n < kStage / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int n = 0; n < kStage / 8; ++n) {
            if (n * 8 >= n_valid) break;
#pragma unroll
            for (int kk = 0; kk < D / 16; kk += 2) {
                const int q = lane >> 3, rr = lane & 7;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(tK + swz<D>(n * 8 + rr, 2 * kk + q)), b0, b1, b2, b3);
                mma_bf16(s[n], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma_bf16(s[n], qa[kk + 1][0], qa[kk + 1][1], qa[kk + 1][2], qa[kk + 1][3], b2, b3);
            }
        }
        const int tq = lane & 3;
        float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < kStage / 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = st * kStage + n * 8 + 2 * tq + (e & 1);
                const bool valid = col < n_my && sTab[col] >= 0;
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
        for (int n = 0; n < kStage / 8; ++n) {
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
#pragma unroll
        for (int kk = 0; kk < kStage / 16; ++kk) {
            if (kk * 16 >= n_valid) break;
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
        __syncthreads();  // buffer consumed by every warp
        issue_stage(st + 2);
    }
    cp_async_wait<0>();
    __syncthreads();  // every warp is done with Q and the stages: their space now holds O

    // ---- this CTA's partial: unnormalised o, running max (log2 units), running sum
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        lrow[hh] += __shfl_xor_sync(0xffffffffu, lrow[hh], 1);
        lrow[hh] += __shfl_xor_sync(0xffffffffu, lrow[hh], 2);
    }
    {
        const int g = lane >> 2, tq = lane & 3;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int h = warp * 16 + g + hh * 8;
            float *orow = sO + h * D;
#pragma unroll
            for (int n = 0; n < D / 8; ++n)
                *reinterpret_cast<float2 *>(orow + n * 8 + 2 * tq) = make_float2(o[n][2 * hh], o[n][2 * hh + 1]);
            if (tq == 0) {
                sM[h] = mrow[hh];
                sL[h] = lrow[hh];
            }
        }
    }
    cluster_sync_all();

    // ---- combine heads [split*HPC, (split+1)*HPC) over the S partials (DSMEM);
    // all remote loads of a thread are issued before any is used
    constexpr int HPC = HR / S;
    const uint32_t o_base = smem_u32(sO), m_base = smem_u32(sM), l_base = smem_u32(sL);
    for (int w = tid; w < HPC * (D / 4); w += NTHR) {
        const int hl = split * HPC + w / (D / 4);  // head within the group
        const int h = h0 + hl;
        const int c4 = w % (D / 4);
        float mv[S], lv[S];
        float4 ov[S];
#pragma unroll
        for (int r = 0; r < S; ++r) {
            mv[r] = ld_dsmem_f32(map_rank(m_base + hl * 4, r));
            lv[r] = ld_dsmem_f32(map_rank(l_base + hl * 4, r));
            ov[r] = ld_dsmem_f32x4(map_rank(o_base + (hl * D + c4 * 4) * 4, r));
        }
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < S; ++r) M = fmaxf(M, mv[r]);
        float Lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
            for (int r = 0; r < S; ++r) {
                const float wgt = mv[r] == -INFINITY ? 0.f : exp2f(mv[r] - M);
                Lsum = fmaf(wgt, lv[r], Lsum);
                acc.x = fmaf(wgt, ov[r].x, acc.x);
                acc.y = fmaf(wgt, ov[r].y, acc.y);
                acc.z = fmaf(wgt, ov[r].z, acc.z);
                acc.w = fmaf(wgt, ov[r].w, acc.w);
            }
        }
        const bool empty = !(Lsum > 0.f);
        const float inv = empty ? 0.f : 1.f / Lsum;
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + ((int64_t)row * a.H + h) * D + c4 * 4;
        uint2 pk;
        pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(out) = pk;
        if (a.lse && c4 == 0) a.lse[(int64_t)row * a.H + h] = empty ? -INFINITY : (M + log2f(Lsum)) * kLn2;
    }
    cluster_sync_all();  // partials stay readable until every CTA of the cluster is done
}

template <int D, int NW>
cudaError_t launch_cluster_t(const AttnArgs &a, cudaStream_t s) {
    constexpr int S = 16;
    using L = Smem<D, NW>;
    static unsigned long long done = 0;
    static unsigned long long np_done = 0;
    // item table sized for the largest slice any sequence of this call can have
    const int64_t total_max = (a.idx ? (int64_t)a.topk : a.E_cap) + a.window;
    int per_max = (int)((total_max + S - 1) / S);
    per_max = (per_max + 15) / 16 * 16;
    const size_t smem = (size_t)L::total(per_max);
    if (smem > 220 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = smem_limit_once(attn_decode_cluster_kernel<D, NW, 16>, 220 * 1024, done);
    if (e != cudaSuccess) return e;
    {
        int dev = 0;
        cudaGetDevice(&dev);
        const unsigned long long bit = 1ull << (dev & 63);
        if (!(np_done & bit)) {
            e = cudaFuncSetAttribute(attn_decode_cluster_kernel<D, NW, 16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            np_done |= bit;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, a.rows, a.H / (NW * 16));
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // the launch may overlap the tail of the previous kernel in the stream; the
    // kernel's first instruction waits for that kernel's completion
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, attn_decode_cluster_kernel<D, NW, 16>, a);
}

template <int D>
cudaError_t launch_cluster_d(const AttnArgs &a, cudaStream_t s) {
    // heads are processed in groups of at most 64 (4 warps), one cluster per group
    switch (a.H / 16) {
        case 1: return launch_cluster_t<D, 1>(a, s);
        case 2: return launch_cluster_t<D, 2>(a, s);
        case 4: return launch_cluster_t<D, 4>(a, s);
        case 8: return launch_cluster_t<D, 4>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool decode_cluster_supported(int H, int d) {
    return (d == 64 || d == 128) && (H == 16 || H == 32 || H == 64 || H == 128);
}

cudaError_t launch_attn_decode_cluster(const AttnArgs &a, cudaStream_t s) {
    if (a.d == 128) return launch_cluster_d<128>(a, s);
    if (a.d == 64) return launch_cluster_d<64>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace hsa
