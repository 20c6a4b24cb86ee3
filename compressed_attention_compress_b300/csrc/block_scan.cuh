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

}  // namespace hsa
