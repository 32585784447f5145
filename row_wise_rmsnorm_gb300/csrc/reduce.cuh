// reduce.cuh -- fixed-order column reduction of the backward's dgamma/dbeta partials.
// Included by api.cu only (one definition of the kernel in the library).
#pragma once

#include <cuda_runtime.h>

#include "kernels.cuh"

namespace mt {

// Column sums of the [P, D] partials in a fixed order. A block owns 32 columns (one per
// lane, so each warp load is one 128-byte line) and spreads the partial rows over its
// W = kReduceWarps warps: warp w sums rows w, w + W, w + 2W, ... in ascending order,
// kReduceBatch loads in flight before each group of adds (rows past P add nothing);
// warp 0 then adds the W warp sums in ascending order. Many small blocks keep the
// loads spread over many SMs. blockIdx.y selects dgamma (0) or dbeta (1). The kernel is
// launched as a programmatic dependent of the backward: pdl_enter() holds it until the
// backward grid has finished and its partials are visible.
constexpr int kReduceWarps = 32;
constexpr int kReduceCols = 32;
constexpr int kReduceBatch = 16;
__global__ void __launch_bounds__(32 * kReduceWarps)
param_reduce_kernel(const float *__restrict__ part, int P, int D, float *__restrict__ out0,
                    float *__restrict__ out1) {
    pdl_enter();
    __shared__ float sm[kReduceWarps][33];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const float *src = part + (size_t)blockIdx.y * (size_t)P * (size_t)D;
    float *dst = blockIdx.y == 0 ? out0 : out1;
    const int col = blockIdx.x * kReduceCols + lane;
    float s = 0.f;
    if (col < D) {
        for (int p = w; p < P; p += kReduceBatch * kReduceWarps) {
            float v[kReduceBatch];
#pragma unroll
            for (int i = 0; i < kReduceBatch; ++i) {
                const int q = p + i * kReduceWarps;
                v[i] = q < P ? __ldcg(src + (size_t)q * D + col) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kReduceBatch; ++i)
                if (p + i * kReduceWarps < P) s += v[i];
        }
    }
    sm[w][lane] = s;
    __syncthreads();
    if (w == 0 && col < D) {
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < kReduceWarps; ++i) tot += sm[i][lane];
        dst[col] = tot;
    }
}

}  // namespace mt
