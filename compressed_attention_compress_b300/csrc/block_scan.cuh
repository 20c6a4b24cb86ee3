// Block-wide exclusive prefix sums built from warp shuffles (no library primitives).
#pragma once

#include <cuda_runtime.h>

namespace hsa {

__device__ __forceinline__ int warp_inclusive_sum(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Exclusive prefix sum of `v` over the block (threads in threadIdx.x order).
// `scratch` holds at least 33 ints of shared memory; `total` receives the sum.
// Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_sum(int v, int *scratch, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    const int inc = warp_inclusive_sum(v);
    __syncthreads();  // scratch may still be read by a previous call
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nwarps ? scratch[lane] : 0;
        const int wi = warp_inclusive_sum(w);
        if (lane < nwarps) scratch[lane] = wi - w;
        if (lane == 31) scratch[32] = wi;
    }
    __syncthreads();
    total = scratch[32];
    return scratch[warp] + inc - v;
}

// Exclusive prefix sums of two values at once (the same barriers as one);
// `scratch` holds at least 66 ints of shared memory.
__device__ __forceinline__ int2 block_exclusive_sum2(int a, int b, int *scratch, int &total_a, int &total_b) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    const int ia = warp_inclusive_sum(a), ib = warp_inclusive_sum(b);
    __syncthreads();  // scratch may still be read by a previous call
    if (lane == 31) {
        scratch[warp] = ia;
        scratch[33 + warp] = ib;
    }
    __syncthreads();
    if (warp == 0) {
        const int wa = lane < nwarps ? scratch[lane] : 0, wb = lane < nwarps ? scratch[33 + lane] : 0;
        const int xa = warp_inclusive_sum(wa), xb = warp_inclusive_sum(wb);
        if (lane < nwarps) {
            scratch[lane] = xa - wa;
            scratch[33 + lane] = xb - wb;
        }
        if (lane == 31) {
            scratch[32] = xa;
            scratch[65] = xb;
        }
    }
    __syncthreads();
    total_a = scratch[32];
    total_b = scratch[65];
    return make_int2(scratch[warp] + ia - a, scratch[33 + warp] + ib - b);
}

}  // namespace hsa
