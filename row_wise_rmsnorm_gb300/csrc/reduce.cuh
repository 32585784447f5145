// reduce.cuh -- fixed-order column reduction of the backward's dgamma/dbeta partials.
// Included by api.cu only (one definition of the kernel in the library).
#pragma once

#include <cuda_runtime.h>

#include "kernels.cuh"

namespace mt {

// Column sums of the [P, D] partials in a fixed order. A block owns 32*V columns: lane l
// loads columns l*V .. l*V+V-1 of a partial row with one V-wide access (one 128-byte
// line per warp load for V = 1, 512 bytes for V = 4). Warp w sums partial rows
// w, w + W, w + 2W, ... in ascending order, kReduceBatch loads in flight before each
// group of adds (rows past P add nothing); then thread c < 32*V adds the W warp sums of
// column c in ascending warp order. blockIdx.y selects dgamma (0) or dbeta (1). V = 4
// needs D % 4 == 0. The host picks V = 4 only when D is wide enough for one block per
// SM, so small D keeps its loads spread over many SMs. The kernel is launched as a
// programmatic dependent of the backward: pdl_enter() holds it until the backward grid
// has finished and its partials are visible.
constexpr int kReduceBatch = 12;

template <int V> struct VecF;
template <> struct VecF<1> {
    using T = float;
    __device__ static T zero() { return 0.f; }
    __device__ static void add(T &a, const T &b) { a += b; }
    __device__ static float get(const T &a, int) { return a; }
};
template <> struct VecF<4> {
    using T = float4;
    __device__ static T zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ static void add(T &a, const T &b) { a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w; }
    __device__ static float get(const T &a, int e) {
        return (e == 0) ? a.x : (e == 1) ? a.y : (e == 2) ? a.z : a.w;
    }
};

template <int V, int W>
__global__ void __launch_bounds__(32 * W)
param_reduce_kernel(const float *__restrict__ part, int P, int D, float *__restrict__ out0,
                    float *__restrict__ out1) {
    pdl_enter();
    using F = VecF<V>;
    using T = typename F::T;
    __shared__ T sm[W][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const float *src = part + (size_t)blockIdx.y * (size_t)P * (size_t)D;
    float *dst = blockIdx.y == 0 ? out0 : out1;
    const int col0 = blockIdx.x * 32 * V;
    const int col = col0 + lane * V;
    T s = F::zero();
    if (col < D) {
        for (int p = w; p < P; p += kReduceBatch * W) {
            T v[kReduceBatch];
#pragma unroll
            for (int i = 0; i < kReduceBatch; ++i) {
                const int q = p + i * W;
                v[i] = q < P ? __ldcg(reinterpret_cast<const T *>(src + (size_t)q * D + col)) : F::zero();
            }
#pragma unroll
            for (int i = 0; i < kReduceBatch; ++i)
                if (p + i * W < P) F::add(s, v[i]);
        }
    }
    sm[w][lane] = s;
    __syncthreads();
    if (threadIdx.x < 32 * V) {
        const int c = col0 + threadIdx.x;
        if (c < D) {
            const int l = threadIdx.x / V, e = threadIdx.x % V;
            float tot = 0.f;
#pragma unroll 8
            for (int i = 0; i < W; ++i) tot += F::get(sm[i][l], e);
            dst[c] = tot;
        }
    }
}

// Narrow form (32 columns, 32 warps per block) and wide form (128 columns, 16 warps; 4 when
// there are at most 4 batches of partial rows).
constexpr int kReduceNarrowWarps = 32;
constexpr int kReduceWideWarps = 16;

}  // namespace mt
