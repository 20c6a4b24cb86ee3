// V4's per-layer attention details around the attention kernels (QbitAI article
// "DeepSeek V4报告太详尽了！", section 混合注意力机制, the paragraphs after the CSA/HCA
// description): RMSNorm of the query and of the KV entries, rotary position
// encoding of their last `rope_dims` channels only, one entry serving as key and
// value (the caller passes the same buffer for both), the inverse rotation of the
// query's position on the output, and a learnable sink logit in the softmax
// denominator.
//
//   rmsnorm_rope_kernel   x <- R(pos) N(x) in place, one warp per row: queries
//                         before attention, compressed entries when they are
//                         written, raw tokens when they enter the window.
//   attn_finalize_kernel  (out, lse) of plain attention over the prepared
//                         vectors -> sink and inverse rotation:
//                         lse' = ln(e^lse + e^z), out' = R(-p) e^(lse - lse') out.
//
// Rotation: channel pair k (channels d - rd + 2k, d - rd + 2k + 1) turns by
// pos * theta^(-2k/rd).  The angle is formed and reduced in double precision so
// that positions up to millions keep it exact to well below a bf16 ulp; the
// frequencies theta^(-2k/rd) come with the launch, formed on the host in double.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace hsa {

namespace {

template <typename T>
__device__ __forceinline__ float load_e(const T *p);
template <>
__device__ __forceinline__ float load_e<float>(const float *p) {
    return *p;
}
template <>
__device__ __forceinline__ float load_e<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void store_e(T *p, float v);
template <>
__device__ __forceinline__ void store_e<float>(float *p, float v) {
    *p = v;
}
template <>
__device__ __forceinline__ void store_e<__nv_bfloat16>(__nv_bfloat16 *p, float v) {
    *p = __float2bfloat16_rn(v);
}

// cos and sin of pos * inv_freq[k] (inv_freq[k] = theta^(-2k/rd), formed on the host in
// double): the angle is formed and reduced modulo 2 pi in double precision, then
// sin/cos are taken in fp32 on the reduced angle (|r| <= pi)
__device__ __forceinline__ void rope_angle(int64_t pos, const double *inv_freq, int k, float &c, float &s) {
    const double ang = (double)pos * inv_freq[k];
    const double two_pi = 6.283185307179586476925286766559;
    const double n = rint(ang * (1.0 / two_pi));
    const float r = (float)fma(-two_pi, n, ang);
    sincosf(r, &s, &c);
}

constexpr int kMaxPerLane = 16;  // d <= 512

template <typename T>
__global__ void __launch_bounds__(128) rmsnorm_rope_kernel(NormRopeArgs a) {
    const int b = blockIdx.y;
    const int64_t w = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t n = a.n_begin[b] + w / a.H;
    const int h = (int)(w % a.H);
    if (n >= a.n_end[b]) return;
    if (n < 0 || n >= a.n_cap) {
        if (lane == 0) raise_flag(FLAG_ATTN_RANGE);
        return;
    }
    T *x = static_cast<T *>(a.x) + b * a.x_sb + n * a.x_sn + (int64_t)h * a.d;
    const int per = a.d / 32;  // consecutive channels per lane (even)
    const int c0 = lane * per;
    float v[kMaxPerLane];
    float ss = 0.f;
    for (int e = 0; e < per; ++e) {
        v[e] = load_e<T>(x + c0 + e);
        ss = fmaf(v[e], v[e], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.f / sqrtf(ss / (float)a.d + a.eps);
    for (int e = 0; e < per; ++e) v[e] = v[e] * inv * (a.gamma ? a.gamma[c0 + e] : 1.f);
    if (a.rope_dims > 0) {
        const int64_t pos = (a.pos_base ? a.pos_base[b] : 0) + n * a.pos_stride + a.pos_offset;
        for (int e = 0; e < per; e += 2) {
            const int c = c0 + e;
            if (c < a.d - a.rope_dims) continue;
            float cs, sn;
            rope_angle(pos, a.inv_freq, (c - (a.d - a.rope_dims)) >> 1, cs, sn);
            const float u = v[e], t = v[e + 1];
            v[e] = u * cs - t * sn;
            v[e + 1] = u * sn + t * cs;
        }
    }
    for (int e = 0; e < per; ++e) store_e<T>(x + c0 + e, v[e]);
}

template <typename T>
__global__ void __launch_bounds__(128) attn_finalize_kernel(FinalizeArgs a) {
    const int64_t row = blockIdx.y;  // b * T + t
    const int h = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (h >= a.H) return;
    const int b = (int)(row / a.T), t = (int)(row - (row / a.T) * a.T);
    const int64_t p = a.q_pos0[b] + t;
    T *o = static_cast<T *>(a.out) + (row * a.H + h) * a.d;
    float scale = 1.f;
    if (a.sink) {
        float *lp = a.lse + row * a.H + h;
        const float L = *lp, z = a.sink[h];
        const float Mx = fmaxf(L, z);
        const float newL = Mx == -INFINITY ? -INFINITY : Mx + logf(expf(L - Mx) + expf(z - Mx));
        scale = L == -INFINITY ? 0.f : expf(L - newL);
        __syncwarp();
        if (lane == 0) *lp = newL;
    }
    const int per = a.d / 32;
    const int c0 = lane * per;
    for (int e = 0; e < per; e += 2) {
        const int c = c0 + e;
        float u = load_e<T>(o + c) * scale, w = load_e<T>(o + c + 1) * scale;
        if (a.rope_dims > 0 && c >= a.d - a.rope_dims) {
            float cs, sn;
            rope_angle(p, a.inv_freq, (c - (a.d - a.rope_dims)) >> 1, cs, sn);
            const float uu = u * cs + w * sn;  // rotation by -angle
            w = -u * sn + w * cs;
            u = uu;
        }
        store_e<T>(o + c, u);
        store_e<T>(o + c + 1, w);
    }
}

}  // namespace

cudaError_t launch_rmsnorm_rope(const NormRopeArgs &a, bool bf16, cudaStream_t s) {
    const int64_t warps = a.max_rows * a.H;
    if (warps <= 0 || a.B <= 0) return cudaSuccess;
    dim3 grid((unsigned)((warps + 3) / 4), a.B);
    if (bf16)
        rmsnorm_rope_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a);
    else
        rmsnorm_rope_kernel<float><<<grid, 128, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attn_finalize(const FinalizeArgs &a, bool bf16, cudaStream_t s) {
    if (a.B * (int64_t)a.T == 0) return cudaSuccess;
    dim3 grid((a.H + 3) / 4, (unsigned)(a.B * (int64_t)a.T));
    if (bf16)
        attn_finalize_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a);
    else
        attn_finalize_kernel<float><<<grid, 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace hsa
