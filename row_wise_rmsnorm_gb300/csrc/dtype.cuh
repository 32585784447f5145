// dtype.cuh -- storage types of the normalization kernels and their 8-element chunk I/O.
//
// Activations (X, R, S, Y, dX), parameters (gamma, beta) and cotangents (dY, dS) are
// stored as fp16, bf16 or fp32; all arithmetic, statistics and parameter gradients are
// fp32 (meTile "Kernel coverage and training scope", "Exact native normalization
// contract": storage FP16 or FP32 with weight, bias and cotangents in either type, FP32
// statistics and accumulation; bf16 is this library's addition). The vector kernels
// move a row in chunks of 8 consecutive elements: one 16-byte access for a 2-byte type,
// two for fp32. A chunk is handed to the arithmetic as four fp32 pairs (elements 2p and
// 2p+1 in pair p). Widening is exact; narrowing rounds to nearest even.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mt {

// Storage type codes; the values match mt_dtype_t in mt_norm.h.
enum DType : int { kF16 = 0, kBF16 = 1, kF32 = 2 };

template <int DT> struct Store;
template <> struct Store<kF16> { using T = __half; };
template <> struct Store<kBF16> { using T = __nv_bfloat16; };
template <> struct Store<kF32> { using T = float; };

// A chunk is PPC fp32 pairs (2*PPC consecutive elements): PPC = 4 (8 elements) in
// general, PPC = 2 (4 elements, one 16-byte unit) for kernels whose arrays are all fp32.
// 16-byte units in one chunk of type DT:
template <int DT, int PPC = 4>
__host__ __device__ constexpr int chunk_units() {
    return (int)sizeof(typename Store<DT>::T) * 2 * PPC / 16;
}

// ------------------------------------------------------------- conversions ---

__device__ __forceinline__ float2 h2_to_f2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
__device__ __forceinline__ float2 b2_to_f2(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}
__device__ __forceinline__ uint32_t f2_to_h2(float2 f) {
    __half2 h = __floats2half2_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t f2_to_b2(float2 f) {
    __nv_bfloat162 h = __float22bfloat162_rn(f);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// One 16-byte unit of a 2-byte type as four fp32 pairs, and back.
template <int DT>
__device__ __forceinline__ void unpack_unit(const uint4 &u, float2 (&f)[4]) {
    static_assert(DT == kF16 || DT == kBF16, "2-byte types only");
    if constexpr (DT == kF16) {
        f[0] = h2_to_f2(u.x); f[1] = h2_to_f2(u.y); f[2] = h2_to_f2(u.z); f[3] = h2_to_f2(u.w);
    } else {
        f[0] = b2_to_f2(u.x); f[1] = b2_to_f2(u.y); f[2] = b2_to_f2(u.z); f[3] = b2_to_f2(u.w);
    }
}
template <int DT>
__device__ __forceinline__ uint4 pack_unit(const float2 (&f)[4]) {
    static_assert(DT == kF16 || DT == kBF16, "2-byte types only");
    uint4 u;
    if constexpr (DT == kF16) {
        u.x = f2_to_h2(f[0]); u.y = f2_to_h2(f[1]); u.z = f2_to_h2(f[2]); u.w = f2_to_h2(f[3]);
    } else {
        u.x = f2_to_b2(f[0]); u.y = f2_to_b2(f[1]); u.z = f2_to_b2(f[2]); u.w = f2_to_b2(f[3]);
    }
    return u;
}

// The chunk's 16-byte units (chunk_units<DT, PPC>() of them, read from `units`, `stride`
// apart) as PPC fp32 pairs.
template <int DT, int PPC = 4>
__device__ __forceinline__ void unpack_chunk(const uint4 *units, int stride, float2 (&f)[PPC]) {
    if constexpr (DT == kF32) {
#pragma unroll
        for (int u = 0; u < PPC / 2; ++u) {
            const uint4 a = units[u * stride];
            f[2 * u] = make_float2(__uint_as_float(a.x), __uint_as_float(a.y));
            f[2 * u + 1] = make_float2(__uint_as_float(a.z), __uint_as_float(a.w));
        }
    } else {
        static_assert(PPC == 4, "a 2-byte chunk is one 16-byte unit of 8 elements");
        unpack_unit<DT>(units[0], f);
    }
}

// ------------------------------------------------------------ global I/O ---
// p points at the chunk's first element (8 elements, 16-byte aligned).

enum Hint : int { kStream = 0, kReadOnly = 1 };

template <int H>
__device__ __forceinline__ uint4 ld_unit(const void *p) {
    if constexpr (H == kStream) return __ldcs(reinterpret_cast<const uint4 *>(p));
    else return __ldg(reinterpret_cast<const uint4 *>(p));
}

// Load a chunk as fp32 pairs; all zeros when !valid (nothing is read).
template <int DT, int H, int PPC = 4>
__device__ __forceinline__ void ld_chunk(const void *p, bool valid, float2 (&f)[PPC]) {
    if constexpr (DT == kF32) {
#pragma unroll
        for (int u = 0; u < PPC / 2; ++u) {
            const uint4 a = valid ? ld_unit<H>(static_cast<const float *>(p) + 4 * u)
                                  : make_uint4(0, 0, 0, 0);
            f[2 * u] = make_float2(__uint_as_float(a.x), __uint_as_float(a.y));
            f[2 * u + 1] = make_float2(__uint_as_float(a.z), __uint_as_float(a.w));
        }
    } else {
        static_assert(PPC == 4, "a 2-byte chunk is one 16-byte unit of 8 elements");
        unpack_unit<DT>(valid ? ld_unit<H>(p) : make_uint4(0, 0, 0, 0), f);
    }
}

// Load a parameter chunk (gamma, beta) as fp32 pairs through the read-only path.
template <int DT>
__device__ __forceinline__ void ld_param(const typename Store<DT>::T *p, float2 (&f)[4]) {
    if constexpr (DT == kF32) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        f[0] = make_float2(a.x, a.y);
        f[1] = make_float2(a.z, a.w);
        f[2] = make_float2(b.x, b.y);
        f[3] = make_float2(b.z, b.w);
    } else {
        unpack_unit<DT>(__ldg(reinterpret_cast<const uint4 *>(p)), f);
    }
}

// Round a chunk to DT (nearest even) and store it with streaming (evict-first) stores.
template <int DT, int PPC = 4>
__device__ __forceinline__ void st_chunk(void *p, const float2 (&f)[PPC]) {
    if constexpr (DT == kF32) {
#pragma unroll
        for (int u = 0; u < PPC / 2; ++u)
            __stcs(reinterpret_cast<float4 *>(p) + u,
                   make_float4(f[2 * u].x, f[2 * u].y, f[2 * u + 1].x, f[2 * u + 1].y));
    } else {
        static_assert(PPC == 4, "a 2-byte chunk is one 16-byte unit of 8 elements");
        __stcs(reinterpret_cast<uint4 *>(p), pack_unit<DT>(f));
    }
}

template <int DT>
__device__ __forceinline__ const typename Store<DT>::T *as(const void *p) {
    return static_cast<const typename Store<DT>::T *>(p);
}
template <int DT>
__device__ __forceinline__ typename Store<DT>::T *as(void *p) {
    return static_cast<typename Store<DT>::T *>(p);
}

// --------------------------------------------------- scalar (any alignment) ---
// Element access with the type chosen at run time, for the fallback kernels that serve
// misaligned bases and widths that are not a multiple of 8.

// A 2-byte element is read as 16 bits and widened by its type (fp16 through the
// conversion instruction, bf16 by placing the bits in the upper half of an fp32).
__device__ __forceinline__ float widen16(unsigned short u, int dt) {
    return (dt == kBF16) ? __uint_as_float((uint32_t)u << 16) : __half2float(__ushort_as_half(u));
}

__device__ __forceinline__ float ld_elem(const void *p, int64_t i, int dt) {
    if (dt == kF32) return __ldg(static_cast<const float *>(p) + i);
    return widen16(__ldg(static_cast<const unsigned short *>(p) + i), dt);
}

__device__ __forceinline__ float ld_elem_stream(const void *p, int64_t i, int dt) {
    if (dt == kF32) return __ldcs(static_cast<const float *>(p) + i);
    return widen16(__ldcs(static_cast<const unsigned short *>(p) + i), dt);
}

__device__ __forceinline__ void st_elem(void *p, int64_t i, float v, int dt) {
    if (dt == kF16) static_cast<__half *>(p)[i] = __float2half_rn(v);
    else if (dt == kBF16) static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    else static_cast<float *>(p)[i] = v;
}

}  // namespace mt
