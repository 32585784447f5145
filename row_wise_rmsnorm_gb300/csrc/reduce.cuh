// reduce.cuh -- fixed-order column reduction of the backward's dgamma/dbeta partials.
// Included by api.cu only (one definition of the kernel in the library).
#pragma once

#include <cuda_runtime.h>

namespace mt {

// Column sums of the [P, D] partials in a fixed order: slice s of the block sums
// rows s, s + SL, s + 2 SL, ... in ascending order, then thread row 0 adds the SL
// slice sums in ascending order. blockIdx.y selects dgamma (0) or dbeta (1).
constexpr int kReduceSlices = 16;
__global__ void __launch_bounds__(32 * kReduceSlices)
param_reduce_kernel(const float *__restrict__ part, int P, int D, float *__restrict__ out0,
                    float *__restrict__ out1) {
    __shared__ float sm[kReduceSlices][33];
    const float *src = part + (size_t)blockIdx.y * (size_t)P * (size_t)D;
    float *dst = blockIdx.y == 0 ? out0 : out1;
    const int col = blockIdx.x * 32 + threadIdx.x;
    float s = 0.f;
    if (col < D) {
#pragma unroll 4
        for (int q = threadIdx.y; q < P; q += kReduceSlices) s += src[(size_t)q * D + col];
    }
    sm[threadIdx.y][threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.y == 0 && col < D) {
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < kReduceSlices; ++i) tot += sm[i][threadIdx.x];
        dst[col] = tot;
    }
}

}  // namespace mt
