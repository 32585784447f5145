// launch.cuh -- launch shapes and per-op planning for the normalization kernels.
//
// A launch shape is (TPR threads per row, RPC rows per CTA, CH chunks per thread,
// VEC fp16 elements per chunk). VEC = 8 (one 16-byte access per chunk) is legal when
// D % 8 == 0 and every row base is 16-byte aligned; VEC = 1 covers everything else.
// The first shape whose width covers D is taken. Forward rows up to 1024 wide get one
// warp each (four rows per CTA, two for the fused op at 1024); wider rows get a row
// group of 64-512 threads, one row per CTA (on GB300 this beat a persistent pipelined
// forward at every width measured). The
// aligned backward is persistent and pipelined (pipe.cuh), with few CTAs so that the
// dgamma/dbeta partials stay small.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>

#include "kernels.cuh"
#include "pipe.cuh"

namespace mt {

// Forward shapes for 16-byte-aligned rows, per op: X(max_D, TPR, RPC, CH, PACK, MINB).
// PACK runs norm_fwd_packed_kernel (the row kept as fp16 chunks; RMSNorm and LayerNorm
// only), otherwise norm_fwd_vec8_kernel (the row kept as fp32 pairs). MINB is the
// resident-CTA floor per SM the kernel is compiled for, which caps its registers per
// thread (0: the compiler's choice). Every entry was timed on GB300 against its
// neighbours and compiles without spills.
#ifndef MT_FWD_SHAPES_RMS
#define MT_FWD_SHAPES_RMS(X)           \
    X(256, 32, 4, 1, false, 0)         \
    X(512, 32, 4, 2, false, 0)         \
    X(1024, 32, 4, 4, false, 0)        \
    X(2048, 128, 1, 2, true, 16)       \
    X(4096, 128, 1, 4, true, 12)       \
    X(8192, 256, 1, 4, true, 6)        \
    X(16384, 512, 1, 4, true, 3)
#endif
#ifndef MT_FWD_SHAPES_LAYER
#define MT_FWD_SHAPES_LAYER(X)         \
    X(256, 32, 4, 1, false, 0)         \
    X(512, 32, 4, 2, false, 0)         \
    X(1024, 32, 4, 4, false, 0)        \
    X(2048, 128, 1, 2, true, 16)       \
    X(4096, 64, 1, 8, true, 8)         \
    X(8192, 512, 1, 2, true, 4)        \
    X(16384, 512, 1, 4, false, 0)
#endif
#ifndef MT_FWD_SHAPES_FUSED
#define MT_FWD_SHAPES_FUSED(X)         \
    X(256, 32, 4, 1, false, 16)        \
    X(512, 32, 4, 2, false, 16)        \
    X(1024, 64, 2, 2, false, 16)       \
    X(2048, 128, 1, 2, false, 16)      \
    X(4096, 512, 1, 1, false, 4)       \
    X(8192, 512, 1, 2, false, 4)       \
    X(16384, 512, 1, 4, false, 0)
#endif

#define MT_FWD_SHAPES_VEC1(X) \
    X(64, 32, 4, 2)           \
    X(128, 32, 4, 4)          \
    X(256, 32, 4, 8)          \
    X(512, 32, 4, 16)         \
    X(1024, 32, 4, 32)        \
    X(2048, 128, 1, 16)       \
    X(4096, 256, 1, 16)       \
    X(8192, 512, 1, 16)       \
    X(16384, 1024, 1, 16)

#define MT_BWD_SHAPES_VEC1(X) \
    X(64, 32, 8, 2)           \
    X(128, 32, 8, 4)          \
    X(256, 32, 8, 8)          \
    X(512, 32, 8, 16)         \
    X(1024, 64, 4, 16)        \
    X(2048, 128, 4, 16)       \
    X(4096, 256, 2, 16)       \
    X(8192, 512, 1, 16)       \
    X(16384, 512, 1, 32)

// Pipelined persistent backward shapes for 16-byte-aligned rows, RMSNorm and the fused
// op (the first table) and LayerNorm: X(max_D, TPR, RPC, CH, STAGES, CTAS). STAGES is the
// largest ring depth (pipe_stages() cuts it to fit shared memory); CTAS the resident CTAs
// per SM the kernel is compiled for, which caps its registers per thread. The persistent
// grid is the resident CTA count, one dgamma/dbeta partial row per CTA. LayerNorm keeps
// two sums per thread and column, so its narrow shapes use single-row-group CTAs.
#ifndef MT_BWD_PIPE_SHAPES_RMS
#define MT_BWD_PIPE_SHAPES_RMS(X)   \
    X(256, 32, 16, 1, 8, 2)         \
    X(512, 64, 8, 1, 8, 2)          \
    X(1024, 128, 4, 1, 8, 2)        \
    X(2048, 256, 2, 1, 8, 2)        \
    X(4096, 512, 1, 1, 4, 2)        \
    X(8192, 512, 1, 2, 3, 1)        \
    X(16384, 512, 1, 4, 3, 1)
#endif
#ifndef MT_BWD_PIPE_SHAPES_LAYER
#define MT_BWD_PIPE_SHAPES_LAYER(X) \
    X(256, 32, 16, 1, 8, 1)         \
    X(512, 64, 1, 1, 8, 16)         \
    X(1024, 128, 1, 1, 6, 6)        \
    X(2048, 256, 1, 1, 6, 3)        \
    X(4096, 512, 1, 1, 4, 2)        \
    X(8192, 512, 1, 2, 3, 1)        \
    X(16384, 512, 1, 4, 3, 1)
#endif

// Ring depth: the table's depth, cut so that ring + parameter slots fit the dynamic
// shared memory a CTA may use (227 KB per SM, shared by `ctas` resident CTAs), and
// never below 2.
constexpr size_t kMaxDynSmem = 226 * 1024;
constexpr int pipe_stages(int base, int narr, int npar, int ch, int threads, int ctas) {
    const size_t slot = (size_t)ch * threads * 16;
    const int fit = (int)(((kMaxDynSmem / ctas / slot) - npar) / narr);
    const int s = base < fit ? base : fit;
    return s < 2 ? 2 : s;
}

struct LaunchPlan {
    const void *kernel = nullptr;
    int threads = 0;
    int grid = 0;       // forward: ceil(N / RPC); backward: persistent CTA count P
    size_t smem = 0;    // dynamic shared memory bytes
    int rows_per_cta = 0;
};

// Host helpers defined in api.cu (cached per device; thread-safe).
void record_cuda_error(cudaError_t e);  // what mt_last_cuda_error() reports on this thread
cudaError_t device_sm_count(int device, int *sms);
cudaError_t cached_occupancy(const void *kernel, int threads, size_t smem, int device,
                             int *blocks_per_sm);

template <int OP, int TPR, int RPC, int CH, int VEC, bool PACK = false, int MINB = 1>
cudaError_t fwd_plan_shape(int64_t N, LaunchPlan *p) {
    static_assert(!(PACK && OP == kAddRms), "the fused op keeps its fp32 sum");
    if constexpr (VEC == 8 && PACK)
        p->kernel = reinterpret_cast<const void *>(&norm_fwd_packed_kernel<OP, TPR, RPC, CH, MINB>);
    else if constexpr (VEC == 8)
        p->kernel = reinterpret_cast<const void *>(&norm_fwd_vec8_kernel<OP, TPR, RPC, CH, MINB>);
    else
        p->kernel = reinterpret_cast<const void *>(&norm_fwd_kernel<OP, TPR, RPC, CH, VEC>);
    p->threads = TPR * RPC;
    p->grid = (int)((N + RPC - 1) / RPC);
    p->smem = 0;
    p->rows_per_cta = RPC;
    return cudaSuccess;
}

// Persistent grid: as many CTAs as fit on the device at once, at most one per row slot.
inline cudaError_t persistent_grid(LaunchPlan *p, int64_t N, int device) {
    int per_sm = 0, sms = 0;
    cudaError_t e = cached_occupancy(p->kernel, p->threads, p->smem, device, &per_sm);
    if (e != cudaSuccess) return e;
    e = device_sm_count(device, &sms);
    if (e != cudaSuccess) return e;
    const int64_t slots = (N + p->rows_per_cta - 1) / p->rows_per_cta;
    const int64_t cap = (int64_t)sms * (int64_t)std::max(per_sm, 1);
    p->grid = (int)std::min(slots, cap);
    return cudaSuccess;
}

template <int OP>
cudaError_t fwd_plan(int64_t N, int D, bool vec8, int device, LaunchPlan *p) {
    (void)device;
#define MT_TRY8(maxd, tpr, rpc, ch, pack, minb) \
    if (D <= maxd) return fwd_plan_shape<OP, tpr, rpc, ch, 8, pack, minb>(N, p);
#define MT_TRY(maxd, tpr, rpc, ch) \
    if (D <= maxd) return fwd_plan_shape<OP, tpr, rpc, ch, VEC>(N, p);
    if (vec8) {
        if constexpr (OP == kRms) {
            MT_FWD_SHAPES_RMS(MT_TRY8)
        } else if constexpr (OP == kLayer) {
            MT_FWD_SHAPES_LAYER(MT_TRY8)
        } else {
            MT_FWD_SHAPES_FUSED(MT_TRY8)
        }
    } else {
        constexpr int VEC = 1;
        MT_FWD_SHAPES_VEC1(MT_TRY)
    }
#undef MT_TRY
#undef MT_TRY8
    return cudaErrorInvalidValue;
}

template <int OP, int TPR, int RPC, int CH, int VEC, bool HAS_DS>
cudaError_t bwd_plan_shape(int64_t N, int D, int device, LaunchPlan *p) {
    constexpr int NV = (OP == kLayer) ? 2 : 1;
    p->kernel = reinterpret_cast<const void *>(&norm_bwd_kernel<OP, TPR, RPC, CH, VEC, HAS_DS>);
    p->threads = TPR * RPC;
    p->smem = (RPC > 1) ? (size_t)NV * (size_t)D * sizeof(float) : 0;
    p->rows_per_cta = RPC;
    return persistent_grid(p, N, device);
}

template <int OP, int TPR, int RPC, int CH, int STAGES, bool HAS_DS, int CTAS>
cudaError_t bwd_pipe_plan_shape(int64_t N, int device, LaunchPlan *p) {
    constexpr int NARR = HAS_DS ? 3 : 2;
    constexpr int NPAR = (CH <= 2) ? 0 : 1;
    constexpr int S = pipe_stages(STAGES, NARR, NPAR, CH, TPR * RPC, CTAS);
    static_assert(Ring<S, NARR, CH, TPR * RPC, NPAR>::kBytes <= kMaxDynSmem, "ring too large");
    p->kernel = reinterpret_cast<const void *>(
        &norm_bwd_pipe_kernel<OP, TPR, RPC, CH, S, HAS_DS, CTAS>);
    p->threads = TPR * RPC;
    p->smem = Ring<S, NARR, CH, TPR * RPC, NPAR>::kBytes;
    p->rows_per_cta = RPC;
    return persistent_grid(p, N, device);
}

template <int OP, bool HAS_DS>
cudaError_t bwd_plan(int64_t N, int D, bool vec8, int device, LaunchPlan *p) {
#define MT_TRY(maxd, tpr, rpc, ch) \
    if (D <= maxd) return bwd_plan_shape<OP, tpr, rpc, ch, VEC, HAS_DS>(N, D, device, p);
#define MT_TRY_PIPE(maxd, tpr, rpc, ch, st, ctas) \
    if (D <= maxd) return bwd_pipe_plan_shape<OP, tpr, rpc, ch, st, HAS_DS, ctas>(N, device, p);
    if (vec8) {
        if constexpr (OP == kLayer) {
            MT_BWD_PIPE_SHAPES_LAYER(MT_TRY_PIPE)
        } else {
            MT_BWD_PIPE_SHAPES_RMS(MT_TRY_PIPE)
        }
    } else {
        constexpr int VEC = 1;
        MT_BWD_SHAPES_VEC1(MT_TRY)
    }
#undef MT_TRY
#undef MT_TRY_PIPE
    return cudaErrorInvalidValue;
}

// Per-op entry points, one translation unit each (compiled in parallel).
cudaError_t fwd_plan_rms(int64_t N, int D, bool vec8, int device, LaunchPlan *p);
cudaError_t fwd_plan_layer(int64_t N, int D, bool vec8, int device, LaunchPlan *p);
cudaError_t fwd_plan_add(int64_t N, int D, bool vec8, int device, LaunchPlan *p);
cudaError_t bwd_plan_rms(int64_t N, int D, bool vec8, int device, LaunchPlan *p);
cudaError_t bwd_plan_layer(int64_t N, int D, bool vec8, int device, LaunchPlan *p);
cudaError_t bwd_plan_add(int64_t N, int D, bool vec8, bool has_ds, int device, LaunchPlan *p);

}  // namespace mt
