// KV compression: every m consecutive K (and V) tokens fold into one entry,
// C[b, j, :] = sum_{r<m} w[r] * X[b, j*m + r, :]   (QbitAI article "DeepSeek V4报告太详尽了！",
// section 混合注意力机制: CSA step 1 and the HCA paragraph, m' = 128 with no overlap).
//
// HBM-bound: every input byte is read once with 16-byte vector loads, rows are
// coalesced (consecutive threads own consecutive 16-byte channel chunks of the
// same token), the weighted sum is accumulated in fp32 in the order r = 0..m-1
// and rounded once to the storage type.  K and V are handled by the same launch
// (blockIdx.y selects the tensor).
#include "common.cuh"
#include "internal.h"

namespace hsa {

__device__ __forceinline__ float load_elem(const float *p) { return *p; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_elem(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_elem(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T, int U>
__global__ void __launch_bounds__(256) compress_kernel(CompressArgs a) {
    constexpr int V = ElemTraits<T>::kVec;
    extern __shared__ float s_w[];
    for (int r = threadIdx.x; r < a.m; r += blockDim.x) s_w[r] = a.w[r];
    __syncthreads();

    const T *__restrict__ x = static_cast<const T *>(blockIdx.y == 0 ? a.k : a.v);
    T *__restrict__ out = static_cast<T *>(blockIdx.y == 0 ? a.kc : a.vc);
    const int nvec = a.d / V;
    const int64_t per_b = a.max_blocks * nvec;
    const int64_t total = per_b * a.B;
    for (int64_t item = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; item < total;
         item += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(item / per_b);
        const int64_t rem = item - b * per_b;
        const int64_t jl = rem / nvec;
        const int c = (int)(rem - jl * nvec);
        const int64_t j0 = a.tok_begin[b] / a.m, j1 = a.tok_end[b] / a.m;
        const int64_t j = j0 + jl;
        if (j >= j1) continue;
        if (a.tok_begin[b] < 0 || (j + 1) * a.m > a.N_cap || j >= a.E_cap) {
            raise_flag(FLAG_COMPRESS_RANGE);
            continue;
        }
        const char *src = reinterpret_cast<const char *>(x + b * a.in_sb + j * a.m * a.in_st + c * V);
        const int64_t step = a.in_st * (int64_t)sizeof(T);
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
        int r = 0;
        for (; r + U <= a.m; r += U) {
            int4 buf[U];
#pragma unroll
            for (int u = 0; u < U; ++u) buf[u] = ld_nc_v4(src + (r + u) * step);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float wr = s_w[r + u];
                const uint32_t *p = reinterpret_cast<const uint32_t *>(&buf[u]);
                if constexpr (V == 8) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[2 * e] = fmaf(wr, bf16_lo(p[e]), acc[2 * e]);
                        acc[2 * e + 1] = fmaf(wr, bf16_hi(p[e]), acc[2 * e + 1]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[e] = fmaf(wr, __uint_as_float(p[e]), acc[e]);
                }
            }
        }
        for (; r < a.m; ++r) {
            const int4 bv = ld_nc_v4(src + r * step);
            const float wr = s_w[r];
            const uint32_t *p = reinterpret_cast<const uint32_t *>(&bv);
            if constexpr (V == 8) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[2 * e] = fmaf(wr, bf16_lo(p[e]), acc[2 * e]);
                    acc[2 * e + 1] = fmaf(wr, bf16_hi(p[e]), acc[2 * e + 1]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] = fmaf(wr, __uint_as_float(p[e]), acc[e]);
            }
        }
        int4 o;
        uint32_t *op = reinterpret_cast<uint32_t *>(&o);
        if constexpr (V == 8) {
#pragma unroll
            for (int e = 0; e < 4; ++e) op[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) op[e] = __float_as_uint(acc[e]);
        }
        *reinterpret_cast<int4 *>(out + b * a.out_sb + j * a.out_se + c * V) = o;
    }
}

// V4 entries (one tensor; the entry is both key and value): one warp per entry, lane l
// owns channels [l * d/32, (l+1) * d/32).  The weighted sum runs in fp32 in the order
// r = 0..m-1; then RMSNorm over the row (gamma, eps) and the rotation of channel pair
// k of the last rope_dims channels by ((j+1)m - 1) * theta^(-2k/rope_dims) (angle
// formed and reduced in double), rounded once to the storage type.
template <typename T>
__global__ void __launch_bounds__(128) compress_v4_kernel(CompressArgs a, CompressV4Args v) {
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int64_t j0 = a.tok_begin[b] / a.m, j1 = a.tok_end[b] / a.m;
    const int64_t j = j0 + (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (j >= j1) return;
    if (a.tok_begin[b] < 0 || (j + 1) * a.m > a.N_cap || j >= a.E_cap) {
        if (lane == 0) raise_flag(FLAG_COMPRESS_RANGE);
        return;
    }
    const int per = a.d / 32;  // even, <= 16
    const int c0 = lane * per;
    const T *x = static_cast<const T *>(a.k) + b * a.in_sb + j * a.m * a.in_st + c0;
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    for (int r = 0; r < a.m; ++r) {
        const float wr = a.w[r];
#pragma unroll
        for (int e = 0; e < 16; ++e)
            if (e < per) acc[e] = fmaf(wr, load_elem(x + (int64_t)r * a.in_st + e), acc[e]);
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e)
        if (e < per) ss = fmaf(acc[e], acc[e], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.f / sqrtf(ss / (float)a.d + v.eps);
    const int64_t pos = (j + 1) * a.m - 1;
    T *out = static_cast<T *>(a.kc) + b * a.out_sb + j * a.out_se + c0;
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
        if (e >= per) break;
        const int c = c0 + e;
        float x0 = acc[e] * inv * (v.gamma ? v.gamma[c] : 1.f);
        float x1 = acc[e + 1] * inv * (v.gamma ? v.gamma[c + 1] : 1.f);
        if (c >= a.d - v.rope_dims) {
            const double ang = (double)pos * v.inv_freq[(c - (a.d - v.rope_dims)) >> 1];
            const double two_pi = 6.283185307179586476925286766559;
            const float rr = (float)fma(-two_pi, rint(ang * (1.0 / two_pi)), ang);
            float sn, cs;
            sincosf(rr, &sn, &cs);
            const float y0 = x0 * cs - x1 * sn;
            x1 = x0 * sn + x1 * cs;
            x0 = y0;
        }
        store_elem(out + e, x0);
        store_elem(out + e + 1, x1);
    }
}

cudaError_t launch_compress_v4(const CompressArgs &a, const CompressV4Args &v, bool bf16, cudaStream_t s) {
    if (a.B <= 0 || a.max_blocks <= 0) return cudaSuccess;
    dim3 grid((unsigned)((a.max_blocks + 3) / 4), a.B);
    if (bf16)
        compress_v4_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a, v);
    else
        compress_v4_kernel<float><<<grid, 128, 0, s>>>(a, v);
    return cudaGetLastError();
}

// Few long blocks (HCA, m = 128, one block per sequence in a decode step): one CTA
// per (block, sequence, K or V) copies the block's m rows into shared memory with
// every 16-byte load in flight at once, then each thread folds its channels over
// r = 0..m-1 with the same fmaf sequence as compress_kernel (bit-identical
// entries), instead of one thread walking the m rows one load group at a time.
template <typename T>
__global__ void __launch_bounds__(128) compress_staged_kernel(CompressArgs a) {
    // a kernel launched after this one with programmatic stream serialization may start
    // its set-up now; it waits for this grid's completion before reading anything
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    extern __shared__ __align__(16) unsigned char s_raw[];
    float *s_w = reinterpret_cast<float *>(s_raw);
    T *s_x = reinterpret_cast<T *>(s_raw + ((a.m * sizeof(float) + 15) & ~(size_t)15));
    const int b = blockIdx.y;
    const bool is_v = blockIdx.z == 1;
    const int64_t j = a.tok_begin[b] / a.m + blockIdx.x;
    if (j >= a.tok_end[b] / a.m) return;
    if (a.tok_begin[b] < 0 || (j + 1) * a.m > a.N_cap || j >= a.E_cap) {
        if (threadIdx.x == 0) raise_flag(FLAG_COMPRESS_RANGE);
        return;
    }
    const T *x = static_cast<const T *>(is_v ? a.v : a.k) + b * a.in_sb + j * a.m * a.in_st;
    const int cpr = a.d * (int)sizeof(T) / 16;  // 16-byte chunks per row
    for (int i = threadIdx.x; i < a.m * cpr; i += blockDim.x) {
        const int r = i / cpr, c = i - r * cpr;
        cp_async_16(smem_u32(reinterpret_cast<unsigned char *>(s_x) + (size_t)i * 16),
                    reinterpret_cast<const unsigned char *>(x + r * a.in_st) + c * 16, 16);
    }
    cp_async_commit();
    for (int r = threadIdx.x; r < a.m; r += blockDim.x) s_w[r] = a.w[r];
    cp_async_wait<0>();
    __syncthreads();
    T *out = static_cast<T *>(is_v ? a.vc : a.kc) + b * a.out_sb + j * a.out_se;
    for (int e = threadIdx.x; e < a.d; e += blockDim.x) {
        float acc = 0.f;
#pragma unroll 8
        for (int r = 0; r < a.m; ++r) acc = fmaf(s_w[r], load_elem(s_x + (size_t)r * a.d + e), acc);
        store_elem(out + e, acc);
    }
}

cudaError_t launch_compress(const CompressArgs &a, bool bf16, int num_sms, cudaStream_t s) {
    const int V = bf16 ? 8 : 4;
    const int64_t total = a.max_blocks * (a.d / V) * a.B;
    if (total <= 0) return cudaSuccess;
    const size_t staged = ((a.m * sizeof(float) + 15) & ~(size_t)15) + (size_t)a.m * a.d * (bf16 ? 2 : 4);
    if (a.m >= 16 && staged <= 96 * 1024 && a.max_blocks * a.B <= 8ll * num_sms && a.max_blocks <= 65535 &&
        a.B <= 65535) {
        static unsigned long long done_bf16 = 0, done_f32 = 0;
        cudaError_t e = bf16 ? smem_limit_once(compress_staged_kernel<__nv_bfloat16>, 96 * 1024, done_bf16)
                             : smem_limit_once(compress_staged_kernel<float>, 96 * 1024, done_f32);
        if (e != cudaSuccess) return e;
        const dim3 grid((unsigned)a.max_blocks, (unsigned)a.B, 2);
        if (bf16)
            compress_staged_kernel<__nv_bfloat16><<<grid, 128, staged, s>>>(a);
        else
            compress_staged_kernel<float><<<grid, 128, staged, s>>>(a);
        return cudaGetLastError();
    }
    const int threads = 256;
    int64_t want = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms * 8;
    const int grid_x = (int)(want < cap ? want : cap);
    const size_t smem = sizeof(float) * a.m;
    dim3 grid(grid_x, 2);
    if (bf16) {
        if (a.m >= 8)
            compress_kernel<__nv_bfloat16, 8><<<grid, threads, smem, s>>>(a);
        else
            compress_kernel<__nv_bfloat16, 4><<<grid, threads, smem, s>>>(a);
    } else {
        if (a.m >= 8)
            compress_kernel<float, 8><<<grid, threads, smem, s>>>(a);
        else
            compress_kernel<float, 4><<<grid, threads, smem, s>>>(a);
    }
    return cudaGetLastError();
}

// ------------------------------------------------------- state-cache append
// Decode-time compression with a partial-block state (the incremental form of the
// same fold): for each new token at position p, r = p mod m, the running fp32 sum
// of the current block is reset at r = 0 and takes fmaf(w[r], x, sum) -- the same
// operations in the same order as compress_kernel -- and at r = m - 1 the block's
// entry p / m is rounded and written.  The raw tokens of earlier blocks are never
// read again, so the raw cache only has to keep the attention window.
template <typename T>
__global__ void __launch_bounds__(128) compress_append_kernel(CompressAppendArgs a) {
    constexpr int V = ElemTraits<T>::kVec;
    const int nvec = a.d / V;
    const int item = blockIdx.x * blockDim.x + threadIdx.x;
    if (item >= a.B * nvec) return;
    const int b = item / nvec, c = item - b * nvec;
    const bool is_v = blockIdx.y == 1;
    const T *x = static_cast<const T *>(is_v ? a.v_new : a.k_new) + b * a.new_sb + c * V;
    float *st = (is_v ? a.state_v : a.state_k) + b * a.state_sb + c * V;
    T *out = static_cast<T *>(is_v ? a.vc : a.kc) + b * a.out_sb + c * V;
    const int64_t p0 = a.pos0[b];
    if (p0 < 0) {
        raise_flag(FLAG_COMPRESS_RANGE);
        return;
    }
    float acc[V];
    {
        const float4 s0 = *reinterpret_cast<const float4 *>(st);
        acc[0] = s0.x; acc[1] = s0.y; acc[2] = s0.z; acc[3] = s0.w;
        if constexpr (V == 8) {
            const float4 s1 = *reinterpret_cast<const float4 *>(st + 4);
            acc[4] = s1.x; acc[5] = s1.y; acc[6] = s1.z; acc[7] = s1.w;
        }
    }
    for (int t = 0; t < a.T; ++t) {
        const int64_t p = p0 + t;
        const int r = (int)(p % a.m);
        const float wr = a.w[r];
        const int4 xv = ld_nc_v4(x + (int64_t)t * a.new_st);
        const uint32_t *xp = reinterpret_cast<const uint32_t *>(&xv);
        if (r == 0) {
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = 0.f;
        }
        if constexpr (V == 8) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] = fmaf(wr, bf16_lo(xp[e]), acc[2 * e]);
                acc[2 * e + 1] = fmaf(wr, bf16_hi(xp[e]), acc[2 * e + 1]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = fmaf(wr, __uint_as_float(xp[e]), acc[e]);
        }
        if (r == a.m - 1) {
            const int64_t j = p / a.m;
            if (j >= a.E_cap) {
                raise_flag(FLAG_COMPRESS_RANGE);
                continue;
            }
            int4 o;
            uint32_t *op = reinterpret_cast<uint32_t *>(&o);
            if constexpr (V == 8) {
#pragma unroll
                for (int e = 0; e < 4; ++e) op[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) op[e] = __float_as_uint(acc[e]);
            }
            *reinterpret_cast<int4 *>(out + j * a.out_se) = o;
        }
    }
    *reinterpret_cast<float4 *>(st) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if constexpr (V == 8) *reinterpret_cast<float4 *>(st + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

cudaError_t launch_compress_append(const CompressAppendArgs &a, bool bf16, cudaStream_t s) {
    const int V = bf16 ? 8 : 4;
    const int items = a.B * (a.d / V);
    if (items <= 0 || a.T <= 0) return cudaSuccess;
    dim3 grid((items + 127) / 128, 2);
    if (bf16)
        compress_append_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a);
    else
        compress_append_kernel<float><<<grid, 128, 0, s>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------ learned compression
// Attention-like pooling with learned weights (QbitAI article, 混合注意力机制: CSA step 1
// merges every m tokens "through an attention-like mechanism with learned weights";
// HCA has no overlap).  Entry j pools the L tokens t_r = (j+1)*m - L + r (t_r >= 0)
// with a = softmax_r(<u, K[t_r]> + bias[r]); the same weights pool K and V.  One warp
// per entry: lanes score the window's tokens (one token row per lane), the warp
// takes the softmax, then every lane accumulates its d/32 channels over the window.
template <typename T>
__global__ void __launch_bounds__(128) compress_learned_kernel(CompressLearnedArgs a) {
    extern __shared__ float s_dyn[];
    float *s_u = s_dyn;                        // [d]
    float *s_sc = s_dyn + a.d + (threadIdx.x >> 5) * a.L;  // [4][L]
    for (int c = threadIdx.x; c < a.d; c += blockDim.x) s_u[c] = a.u[c];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (item >= (int64_t)a.B * a.max_blocks) return;
    const int b = (int)(item / a.max_blocks);
    const int64_t j = a.tok_begin[b] / a.m + (item - (int64_t)b * a.max_blocks);
    if (j >= a.tok_end[b] / a.m) return;
    if (a.tok_begin[b] < 0 || (j + 1) * a.m > a.N_cap || j >= a.E_cap) {
        if (lane == 0) raise_flag(FLAG_COMPRESS_RANGE);
        return;
    }
    const T *kb = static_cast<const T *>(a.k) + b * a.in_sb;
    const T *vb = static_cast<const T *>(a.v) + b * a.in_sb;
    const int64_t t0 = (j + 1) * a.m - a.L;
    // scores, one window token per lane
    for (int r = lane; r < a.L; r += 32) {
        const int64_t t = t0 + r;
        float sc = -INFINITY;
        if (t >= 0) {
            // the token row in 16-byte vectors (rows are 16-byte aligned)
            constexpr int V = ElemTraits<T>::kVec;
            const char *row = reinterpret_cast<const char *>(kb + t * a.in_st);
            float dot = 0.f;
            for (int c = 0; c < a.d; c += V) {
                const int4 x = ld_nc_v4(row + c * sizeof(T));
                const uint32_t *xp = reinterpret_cast<const uint32_t *>(&x);
                if constexpr (V == 8) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        dot = fmaf(s_u[c + 2 * e], bf16_lo(xp[e]), dot);
                        dot = fmaf(s_u[c + 2 * e + 1], bf16_hi(xp[e]), dot);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) dot = fmaf(s_u[c + e], __uint_as_float(xp[e]), dot);
                }
            }
            sc = dot + a.bias[r];
        }
        s_sc[r] = sc;
    }
    __syncwarp();
    float M = -INFINITY;
    for (int r = lane; r < a.L; r += 32) M = fmaxf(M, s_sc[r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float Z = 0.f;
    for (int r = lane; r < a.L; r += 32) Z += s_sc[r] == -INFINITY ? 0.f : expf(s_sc[r] - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
    const float invZ = 1.f / Z;
    // weighted sums over the window, d / 32 channels per lane
    const int per = a.d / 32, c0 = lane * per;
    float ak[16], av[16];
    for (int e = 0; e < per; ++e) ak[e] = av[e] = 0.f;
    for (int r = 0; r < a.L; ++r) {
        const float sc = s_sc[r];
        if (sc == -INFINITY) continue;  // uniform across the warp
        const float w = expf(sc - M) * invZ;
        const int64_t t = t0 + r;
        const T *kr = kb + t * a.in_st + c0;
        const T *vr = vb + t * a.in_st + c0;
        for (int e = 0; e < per; ++e) {
            ak[e] = fmaf(w, load_elem(kr + e), ak[e]);
            av[e] = fmaf(w, load_elem(vr + e), av[e]);
        }
    }
    T *ko = static_cast<T *>(a.kc) + b * a.out_sb + j * a.out_se + c0;
    T *vo = static_cast<T *>(a.vc) + b * a.out_sb + j * a.out_se + c0;
    for (int e = 0; e < per; ++e) {
        store_elem(ko + e, ak[e]);
        store_elem(vo + e, av[e]);
    }
}

cudaError_t launch_compress_learned(const CompressLearnedArgs &a, bool bf16, cudaStream_t s) {
    const int64_t items = (int64_t)a.B * a.max_blocks;
    if (items <= 0) return cudaSuccess;
    const size_t smem = sizeof(float) * ((size_t)a.d + 4 * (size_t)a.L);
    const unsigned grid = (unsigned)((items + 3) / 4);
    if (bf16)
        compress_learned_kernel<__nv_bfloat16><<<grid, 128, smem, s>>>(a);
    else
        compress_learned_kernel<float><<<grid, 128, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace hsa
