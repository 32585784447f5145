// launch.cuh -- launch shapes and per-op, per-dtype planning for the normalization kernels.
//
// A vector launch shape is (TPR threads per row, RPC rows per CTA, CH chunks of 8
// elements per thread). The vector kernels are legal when D % 8 == 0 and every row base
// is 16-byte aligned; the scalar kernels (one element per access, types chosen at run
// time) cover everything else, and every dtype combination the vector tables do not
// list. The first shape whose width covers D is taken. Forward rows up to 1024 wide get
// one warp each (four rows per CTA, two for the fused op at 1024); wider rows get a row
// group of 64-512 threads, one row per CTA (on GB300 this beat a persistent pipelined
// forward at every width measured); aligned rows wider than 16384 are streamed twice
// by one CTA each. The aligned backward is persistent and pipelined
// (pipe.cuh), with few CTAs so that the dgamma/dbeta partials stay small.
//
// Storage types: activations XT, parameters WT, cotangents GT (dtype.cuh). The full
// tables were tuned for fp16 and serve every combination whose three types match; the
// others (fp32 parameters or cotangents with 2-byte activations, and all-fp32 in the
// backward) use short tables. A backward ring that cannot hold two stages, and any
// combination not listed, take the scalar kernel.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>

#include "kernels.cuh"
#include "mt_norm.h"
#include "pipe.cuh"

namespace mt {

// Forward shapes for 16-byte-aligned rows, per op: X(max_D, TPR, RPC, CH, PACK, MINB).
// PACK runs norm_fwd_packed_kernel (the row kept as the loaded 2-byte chunks; RMSNorm and
// LayerNorm with fp16/bf16 activations only), otherwise norm_fwd_vec8_kernel (the row
// kept as fp32 pairs). MINB is the resident-CTA floor per SM the kernel is compiled for,
// which caps its registers per thread (0: the compiler's choice). Every entry was timed
// on GB300 against its neighbours and compiles without spills.
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
// LayerNorm rows of 8192 and 16384 columns: 256-thread row groups with the row packed in
// registers and 5 / 4 resident CTAs per SM (back to back on GB300: LayerNorm 2048 x 16384
// forward 26.5 -> 24.4 us against 512 threads with the row as fp32 pairs, where 5 CTAs per
// SM or 1024-thread rows lost; 4096 x 8192 26.8 us with 512 threads and 4 CTAs, 23.8 us
// with 6 CTAs, which spills, 23.9 us with 5).
#ifndef MT_FWD_SHAPES_LAYER
#define MT_FWD_SHAPES_LAYER(X)         \
    X(256, 32, 4, 1, false, 0)         \
    X(512, 32, 4, 2, false, 0)         \
    X(1024, 32, 4, 4, false, 0)        \
    X(2048, 128, 1, 2, true, 16)       \
    X(4096, 64, 1, 8, true, 8)         \
    X(8192, 256, 1, 4, true, 5)        \
    X(16384, 256, 1, 8, true, 4)
#endif
#ifndef MT_FWD_SHAPES_FUSED
#define MT_FWD_SHAPES_FUSED(X)         \
    X(256, 32, 4, 1, false, 16)        \
    X(512, 32, 4, 2, false, 16)        \
    X(1024, 64, 2, 2, false, 16)       \
    X(2048, 128, 1, 2, false, 12)      \
    X(4096, 512, 1, 1, false, 4)       \
    X(8192, 512, 1, 2, false, 3)
#endif
// (The fused op's 16384-wide rows take the streaming kernel below: 4096 x 16384 in 83.1
// us against 96.2 us for the register-resident row, which holds the fp32 sum x + r.)
// Short forward table (fp32 parameters with 2-byte activations), every op.
#define MT_FWD_SHAPES_SHORT(X)         \
    X(1024, 32, 4, 4, false, 0)        \
    X(4096, 512, 1, 1, false, 4)       \
    X(16384, 512, 1, 4, false, 0)

// Scalar fallback shapes: X(max_D, TPR, RPC, CH), CH elements per thread.
#define MT_FWD_SHAPES_SCALAR(X) \
    X(64, 32, 4, 2)             \
    X(128, 32, 4, 4)            \
    X(256, 32, 4, 8)            \
    X(512, 32, 4, 16)           \
    X(1024, 32, 4, 32)          \
    X(2048, 128, 1, 16)         \
    X(4096, 256, 1, 16)         \
    X(8192, 512, 1, 16)         \
    X(16384, 1024, 1, 16)

#define MT_BWD_SHAPES_SCALAR(X) \
    X(64, 32, 8, 2)             \
    X(128, 32, 8, 4)            \
    X(256, 32, 8, 8)            \
    X(512, 32, 8, 16)           \
    X(1024, 64, 4, 16)          \
    X(2048, 128, 4, 16)         \
    X(4096, 256, 2, 16)         \
    X(8192, 512, 1, 16)         \
    X(16384, 512, 1, 32)

// Pipelined persistent backward shapes for 16-byte-aligned rows, per op (RMSNorm, the fused
// op, LayerNorm): X(max_D, TPR, RPC, CH, STAGES, CTAS). STAGES is the
// largest ring depth (pipe_stages() cuts it to fit shared memory); CTAS the resident CTAs
// per SM the kernel is compiled for, which caps its registers per thread. The persistent
// grid is the resident CTA count, one dgamma/dbeta partial row per CTA. From 1024 to
// 4096 columns RMSNorm and LayerNorm run one 512-thread CTA per SM holding several row
// groups of 16 elements per thread with a 3-deep ring (measured faster than two CTAs of
// 8 elements per thread: fewer per-row instructions per byte).
// 8192 and 16384 columns (RMSNorm) and 16384 (LayerNorm) keep a 2-deep ring: measured
// back to back on GB300 against 3 stages, LayerNorm 2048 x 16384 48.5 -> 46.0 us, RMSNorm
// 4096 x 16384 69.5 -> 68.1 us, RMSNorm 8192 x 8192 (256 threads of 4 chunks) 69.2 ->
// 67.5 us: a smaller start-up burst gets each CTA's first row in sooner.
#ifndef MT_BWD_PIPE_SHAPES_RMS
#define MT_BWD_PIPE_SHAPES_RMS(X)   \
    X(256, 32, 16, 1, 8, 2)         \
    X(512, 64, 8, 1, 8, 2)          \
    X(1024, 64, 8, 2, 3, 1)         \
    X(2048, 128, 4, 2, 3, 1)        \
    X(4096, 256, 2, 2, 3, 1)        \
    X(8192, 256, 1, 4, 2, 1)        \
    X(16384, 512, 1, 4, 2, 1)
#endif
#ifndef MT_BWD_PIPE_SHAPES_FUSED
#define MT_BWD_PIPE_SHAPES_FUSED(X) \
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
    X(1024, 64, 8, 2, 3, 1)         \
    X(2048, 128, 4, 2, 3, 1)        \
    X(4096, 256, 2, 2, 3, 1)        \
    X(8192, 512, 1, 2, 3, 1)        \
    X(16384, 512, 1, 4, 2, 1)
#endif
// All-fp32 backward: an fp32 chunk takes two ring units per array, so these shapes keep
// 2-3 ring stages; 16384-wide fp32 rows (128 KB per stage) take the scalar kernel.
#ifndef MT_BWD_PIPE_SHAPES_F32
#define MT_BWD_PIPE_SHAPES_F32(X)   \
    X(1024, 128, 4, 1, 8, 2)        \
    X(2048, 256, 2, 1, 8, 2)        \
    X(4096, 512, 1, 1, 4, 1)        \
    X(8192, 512, 1, 2, 3, 1)
#endif
#define MT_BWD_PIPE_SHAPES_F32_LAYER(X) \
    X(1024, 128, 1, 1, 6, 6)            \
    X(2048, 256, 1, 1, 6, 3)            \
    X(4096, 512, 1, 1, 4, 1)            \
    X(8192, 512, 1, 2, 3, 1)
// Short backward tables: one shape per width class.
#define MT_BWD_PIPE_SHAPES_RMS_SHORT(X) \
    X(1024, 128, 4, 1, 8, 2)            \
    X(4096, 512, 1, 1, 4, 2)            \
    X(16384, 512, 1, 4, 3, 1)
#define MT_BWD_PIPE_SHAPES_LAYER_SHORT(X) \
    X(1024, 128, 1, 1, 6, 6)              \
    X(4096, 512, 1, 1, 4, 2)              \
    X(16384, 512, 1, 4, 3, 1)

// Aligned rows wider than the tables above cover, forward (every op past 16384 columns, the
// fused op past 8192): the two-pass streaming kernel, one CTA per row, X(max_D, TPR, UN,
// MINB), MINB the resident-CTA floor per SM the kernel is compiled for (1: none); fp32
// rows take half as many chunks in flight (stream_un: the same bytes).
// Each entry gives whole batches of UN chunks per thread at the width it was measured on
// (16384: 4 chunks per thread; 24576: 12; 32768 and 65536: 8 and 16). At 16384 columns
// the register-resident RMSNorm and LayerNorm rows stay faster (RMSNorm 8192 x 16384
// 81.2 us against 84.2 streamed, LayerNorm 2048 x 16384 29.6 against 35.1).
// Measured on GB300 against the cluster split the backward keeps (fp16 forward): RMSNorm
// 4096 x 32768 108.0 -> 90.1 us, LayerNorm 1024 x 131072 189.1 -> 137.6 us, fused op
// 2048 x 65536 239.8 -> 199.7 us, LayerNorm 4096 x 24576 139.9 -> 77.5 us (256 threads;
// 89.9 us at 512); 1024 x 131072 at 1024 threads with 4 chunks 124.4 us, 2 chunks 135.6.
// Floors of 2 or 4 resident CTAs per SM did not help.
#ifndef MT_FWD_STREAM_SHAPES
#define MT_FWD_STREAM_SHAPES(X) \
    X(16384, 512, 2, 1)         \
    X(24576, 256, 4, 1)         \
    X(65536, 512, 4, 1)         \
    X(MT_MAX_COLS, 1024, 4, 1)
#endif

// Rows wider than 16384 columns that are not streamed (the backward; forwards of rows that
// are misaligned or not a multiple of 8 wide): a cluster of CL = 2, 4 or 8 CTAs per row, each CTA a
// slice of ceil(D / CL) columns (rounded up to 8). The shapes below, X(max slice, TPR,
// RPC, CH, ...), are tried in order; the first whose slice needs at most kMaxCluster CTAs
// is taken (CL the smallest power of two that covers D with it).
constexpr int kMaxCluster = 8;
// The all-fp32 backward's slices are 8192 columns (two ring stages of 16384 fp32 columns
// do not fit), so its widest rows need 16 CTAs: a non-portable cluster size, which the
// kernel opts into; where 16-CTA clusters cannot be resident the scalar kernel runs.
constexpr int kMaxClusterF32Bwd = 16;
#define MT_FWD_WIDE_SCALAR(X) X(16384, 1024, 1, 16)
#ifndef MT_BWD_WIDE_PIPE
#define MT_BWD_WIDE_PIPE(X) X(16384, 512, 1, 4, 3, 1)
#endif
#define MT_BWD_WIDE_PIPE_F32(X) X(8192, 512, 1, 2, 3, 1)
#define MT_BWD_WIDE_SCALAR(X) X(16384, 512, 1, 32)

// The cluster split of a D-column row over CTAs of at most `cap` columns: false when
// more than max_cl CTAs would be needed.
inline bool wide_split(int D, int cap, int *cl, int *slice, int max_cl = kMaxCluster) {
    int c = 2;
    while ((int64_t)c * cap < D) c *= 2;
    if (c > max_cl) return false;
    *cl = c;
    *slice = (((D + c - 1) / c) + 7) / 8 * 8;
    return true;
}

// Ring depth: the table's depth, cut so that the ring plus the parameter slots fit the
// dynamic shared memory a CTA may use (227 KB per SM, shared by `ctas` resident CTAs);
// 0 when not even two stages fit.
constexpr size_t kMaxDynSmem = 226 * 1024;
constexpr int pipe_stages(int base, size_t stage_bytes, size_t param_bytes, int ctas) {
    return (param_bytes + 2 * stage_bytes > kMaxDynSmem / ctas)
               ? 0
               : ((int)((kMaxDynSmem / ctas - param_bytes) / stage_bytes) < base
                      ? (int)((kMaxDynSmem / ctas - param_bytes) / stage_bytes)
                      : base);
}

// Returned by a vector plan for a dtype combination or shape it does not cover: the
// caller takes the scalar kernel.
constexpr cudaError_t kNoVectorPlan = cudaErrorNotSupported;

struct LaunchPlan {
    const void *kernel = nullptr;
    int threads = 0;
    int grid = 0;       // CTAs. forward: ceil(N / RPC) (x cluster); backward: persistent
    size_t smem = 0;    // dynamic shared memory bytes
    int rows_per_cta = 0;
    int cluster = 1;    // CTAs per cluster (> 1: a row split across the cluster)
    int slice = 0;      // columns per CTA of a split row
    bool waits = false; // the kernel has bounded waits: pass it the device status word
    bool warm = false;  // forward that warms L2 a wave ahead: pass it FwdArgs::ahead
    // Row owners of a backward, one dgamma/dbeta partial row each.
    int owners() const { return grid / cluster; }
};

// Host helpers defined in api.cu (cached per device; thread-safe).
void record_cuda_error(cudaError_t e);  // what mt_last_cuda_error() reports on this thread
// Called before every kernel launch: cudaSuccess, except in the test build (compiled with
// MT_TEST_HOOKS), where an armed injected failure is returned instead of launching.
cudaError_t launch_hook();
// Launch p.kernel(*arg) on `stream` with the programmatic-stream-serialization attribute.
cudaError_t launch_pdl(const LaunchPlan &p, void *arg, cudaStream_t stream);
cudaError_t device_sm_count(int device, int *sms);
cudaError_t cached_occupancy(const void *kernel, int threads, size_t smem, int device,
                             int *blocks_per_sm);
// Clusters of `cluster` CTAs that can be resident at once (cached per kernel and shape).
cudaError_t cached_cluster_occupancy(const void *kernel, int threads, size_t smem, int cluster,
                                     int device, int *clusters);
// Address of the device's status word: the error bits of bounded waits (cached per device).
cudaError_t device_status_word(int device, unsigned **word);

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

// Persistent grid of clusters for a split row: as many clusters as fit at once, at most
// one CTA per SM (which bounds the partial rows to SMs / cluster) and one per row.
inline cudaError_t persistent_cluster_grid(LaunchPlan *p, int64_t N, int device) {
    int per_sm = 0, sms = 0, fit = 0;
    cudaError_t e = cached_occupancy(p->kernel, p->threads, p->smem, device, &per_sm);
    if (e != cudaSuccess) return e;
    if ((e = device_sm_count(device, &sms)) != cudaSuccess) return e;
    e = cached_cluster_occupancy(p->kernel, p->threads, p->smem, p->cluster, device, &fit);
    if (e != cudaSuccess) return e;
    if (fit == 0 && p->cluster > kMaxCluster) return kNoVectorPlan;  // not resident: scalar
    const int64_t owners = std::min<int64_t>({(int64_t)std::max(fit, 1),
                                              (int64_t)std::max(sms / p->cluster, 1), N});
    p->grid = (int)owners * p->cluster;
    return cudaSuccess;
}

// Forward grid of a split row: one cluster per row.
inline cudaError_t cluster_row_grid(LaunchPlan *p, int64_t N) {
    if (N * p->cluster > (int64_t)INT32_MAX) return cudaErrorInvalidConfiguration;
    p->grid = (int)N * p->cluster;
    return cudaSuccess;
}

// ------------------------------------------------------------------ forward ---

template <int OP, int TPR, int RPC, int CH>
cudaError_t fwd_scalar_shape(int64_t N, LaunchPlan *p) {
    p->kernel = reinterpret_cast<const void *>(&norm_fwd_kernel<OP, TPR, RPC, CH>);
    p->threads = TPR * RPC;
    p->grid = (int)((N + RPC - 1) / RPC);
    p->smem = 0;
    p->rows_per_cta = RPC;
    return cudaSuccess;
}

template <int OP, int TPR, int RPC, int CH>
cudaError_t fwd_scalar_wide(int64_t N, int D, int cap, LaunchPlan *p) {
    if (!wide_split(D, cap, &p->cluster, &p->slice)) return cudaErrorInvalidValue;
    p->kernel = reinterpret_cast<const void *>(&norm_fwd_kernel<OP, TPR, RPC, CH, true>);
    p->threads = TPR * RPC;
    p->smem = 0;
    p->rows_per_cta = RPC;
    return cluster_row_grid(p, N);
}

template <int OP>
cudaError_t fwd_plan_scalar(int64_t N, int D, LaunchPlan *p) {
#define MT_TRY(maxd, tpr, rpc, ch) \
    if (D <= maxd) return fwd_scalar_shape<OP, tpr, rpc, ch>(N, p);
    MT_FWD_SHAPES_SCALAR(MT_TRY)
#undef MT_TRY
#define MT_TRY(cap, tpr, rpc, ch) return fwd_scalar_wide<OP, tpr, rpc, ch>(N, D, cap, p);
    MT_FWD_WIDE_SCALAR(MT_TRY)
#undef MT_TRY
}

// The register floors (MINB) were set for 2-byte types; with fp32 activations or
// parameters the compiler chooses (MINB 0), since the floors would force spills there.
template <int OP, int XT, int WT, int TPR, int RPC, int CH, bool PACK, int MINB>
cudaError_t fwd_vec_shape(int64_t N, LaunchPlan *p) {
    constexpr int minb = (XT == kF32 || WT == kF32) ? 0 : MINB;
    if constexpr (PACK && OP != kAddRms && XT != kF32) {
        p->kernel = reinterpret_cast<const void *>(
            &norm_fwd_packed_kernel<OP, TPR, RPC, CH, minb, XT, WT>);
        p->warm = (OP == kRms);  // (see the kernel)
    } else
        p->kernel = reinterpret_cast<const void *>(
            &norm_fwd_vec8_kernel<OP, TPR, RPC, CH, minb, XT, WT>);
    p->threads = TPR * RPC;
    p->smem = 0;
    p->rows_per_cta = RPC;
    p->grid = (int)((N + RPC - 1) / RPC);
    return cudaSuccess;
}

template <int OP, int XT, int WT, int TPR, int UN, int MINB>
cudaError_t fwd_stream_shape(int64_t N, LaunchPlan *p) {
    p->kernel = reinterpret_cast<const void *>(
        &norm_fwd_stream_kernel<OP, TPR, stream_un(XT, UN), MINB, XT, WT>);
    p->threads = TPR;
    p->smem = 0;
    p->rows_per_cta = 1;
    p->grid = (int)N;
    p->warm = true;
    return cudaSuccess;
}

// Vector forward for activations XT and parameters WT; SHORT selects the short table.
template <int OP, int XT, int WT, bool SHORT>
cudaError_t fwd_plan_vec(int64_t N, int D, LaunchPlan *p) {
#define MT_TRY(maxd, tpr, rpc, ch, pack, minb) \
    if (D <= maxd) return fwd_vec_shape<OP, XT, WT, tpr, rpc, ch, pack, minb>(N, p);
    if constexpr (SHORT) {
        MT_FWD_SHAPES_SHORT(MT_TRY)
    } else if constexpr (OP == kRms) {
        MT_FWD_SHAPES_RMS(MT_TRY)
    } else if constexpr (OP == kLayer) {
        MT_FWD_SHAPES_LAYER(MT_TRY)
    } else {
        MT_FWD_SHAPES_FUSED(MT_TRY)
    }
#undef MT_TRY
    // wider rows: streamed, one CTA per row
#define MT_TRY(maxd, tpr, un, minb) \
    if (D <= maxd) return fwd_stream_shape<OP, XT, WT, tpr, un, minb>(N, p);
    MT_FWD_STREAM_SHAPES(MT_TRY)
#undef MT_TRY
    return kNoVectorPlan;
}

// ----------------------------------------------------------------- backward ---

template <int OP, int TPR, int RPC, int CH, bool HAS_DS>
cudaError_t bwd_scalar_shape(int64_t N, int D, int device, LaunchPlan *p) {
    constexpr int NV = (OP == kLayer) ? 2 : 1;
    p->kernel = reinterpret_cast<const void *>(&norm_bwd_kernel<OP, TPR, RPC, CH, HAS_DS>);
    p->threads = TPR * RPC;
    p->smem = (RPC > 1) ? (size_t)NV * (size_t)D * sizeof(float) : 0;
    p->rows_per_cta = RPC;
    return persistent_grid(p, N, device);
}

template <int OP, int TPR, int RPC, int CH, bool HAS_DS>
cudaError_t bwd_scalar_wide(int64_t N, int D, int cap, int device, LaunchPlan *p) {
    if (!wide_split(D, cap, &p->cluster, &p->slice)) return cudaErrorInvalidValue;
    p->kernel = reinterpret_cast<const void *>(&norm_bwd_kernel<OP, TPR, RPC, CH, HAS_DS, true>);
    p->threads = TPR * RPC;
    p->smem = 0;
    p->rows_per_cta = RPC;
    return persistent_cluster_grid(p, N, device);
}

template <int OP, bool HAS_DS>
cudaError_t bwd_plan_scalar(int64_t N, int D, int device, LaunchPlan *p) {
#define MT_TRY(maxd, tpr, rpc, ch) \
    if (D <= maxd) return bwd_scalar_shape<OP, tpr, rpc, ch, HAS_DS>(N, D, device, p);
    MT_BWD_SHAPES_SCALAR(MT_TRY)
#undef MT_TRY
#define MT_TRY(cap, tpr, rpc, ch) return bwd_scalar_wide<OP, tpr, rpc, ch, HAS_DS>(N, D, cap, device, p);
    MT_BWD_WIDE_SCALAR(MT_TRY)
#undef MT_TRY
}

template <int OP, int XT, int WT, int GT, int TPR, int RPC, int CH, int STAGES, bool HAS_DS,
          int CTAS, bool CLU = false>
cudaError_t bwd_pipe_shape(int64_t N, int device, LaunchPlan *p) {
    constexpr int NPAR = (CH <= 2) ? 0 : 1;
    using G = PipeGeom<CH, XT, WT, GT>;
    using R1 = Ring<1, G::CK, TPR * RPC, G::UX, G::UG, HAS_DS, G::UW, NPAR>;
    constexpr int S1 = pipe_stages(STAGES, R1::kStageBytes, R1::kParamBytes, CTAS);
    // Split rows of the fused op with fp16 dS: read dS into registers instead of through
    // the ring when that is what makes the ring three deep (and the exchange pipelined).
    // Measured on GB300 (backward, back to back): fp16 8192 x 16392 239.9 -> 214.3 us,
    // 1024 x 131072 234.0 -> 216.5 us; with bf16 the same kernel was slower (2048 x 65536
    // 191.0 -> 262.5 us, every width alike; the cause was not found), so bf16 keeps dS in
    // a 2-deep ring.
    using R2 = Ring<1, G::CK, TPR * RPC, G::UX, G::UG, false, G::UW, NPAR>;
    constexpr int S2 = pipe_stages(STAGES, R2::kStageBytes, R2::kParamBytes, CTAS);
    constexpr bool DSD = CLU && HAS_DS && GT == kF16 && S1 < 3 && S2 >= 3;
    constexpr int S = DSD ? S2 : S1;
    if constexpr (S < 2) {
        (void)N; (void)device; (void)p;
        return kNoVectorPlan;
    } else {
        using R = Ring<S, G::CK, TPR * RPC, G::UX, G::UG, HAS_DS && !DSD, G::UW, NPAR>;
        static_assert(R::kBytes <= kMaxDynSmem, "ring too large");
        p->kernel = reinterpret_cast<const void *>(
            &norm_bwd_pipe_kernel<OP, TPR, RPC, CH, S, HAS_DS, CTAS, XT, WT, GT, CLU, DSD>);
        p->threads = TPR * RPC;
        p->smem = R::kBytes;
        p->rows_per_cta = RPC;
        p->waits = CLU;  // the split row's push exchange
        if constexpr (CLU) return persistent_cluster_grid(p, N, device);
        return persistent_grid(p, N, device);
    }
}

// Vector backward for activations XT, parameters WT and cotangents GT; SHORT selects the
// short tables.
template <int OP, int XT, int WT, int GT, bool HAS_DS, bool SHORT>
cudaError_t bwd_plan_vec(int64_t N, int D, int device, LaunchPlan *p) {
#define MT_TRY(maxd, tpr, rpc, ch, st, ctas) \
    if (D <= maxd) return bwd_pipe_shape<OP, XT, WT, GT, tpr, rpc, ch, st, HAS_DS, ctas>(N, device, p);
    if constexpr (XT == kF32 && WT == kF32 && GT == kF32 && OP == kLayer) {
        MT_BWD_PIPE_SHAPES_F32_LAYER(MT_TRY)
    } else if constexpr (XT == kF32 && WT == kF32 && GT == kF32) {
        MT_BWD_PIPE_SHAPES_F32(MT_TRY)
    } else if constexpr (SHORT && OP == kLayer) {
        MT_BWD_PIPE_SHAPES_LAYER_SHORT(MT_TRY)
    } else if constexpr (SHORT) {
        MT_BWD_PIPE_SHAPES_RMS_SHORT(MT_TRY)
    } else if constexpr (OP == kLayer) {
        MT_BWD_PIPE_SHAPES_LAYER(MT_TRY)
    } else if constexpr (OP == kAddRms) {
        MT_BWD_PIPE_SHAPES_FUSED(MT_TRY)
    } else {
        MT_BWD_PIPE_SHAPES_RMS(MT_TRY)
    }
#undef MT_TRY
    // wider rows: split across a cluster (a shape whose ring does not fit falls through)
    constexpr int max_cl = (XT == kF32 && WT == kF32 && GT == kF32) ? kMaxClusterF32Bwd : kMaxCluster;
#define MT_TRY(cap, tpr, rpc, ch, st, ctas)                                                      \
    if (wide_split(D, cap, &p->cluster, &p->slice, max_cl)) {                                   \
        const cudaError_t e =                                                                   \
            bwd_pipe_shape<OP, XT, WT, GT, tpr, rpc, ch, st, HAS_DS, ctas, true>(N, device, p); \
        if (e != kNoVectorPlan) return e;                                                       \
    }
    if constexpr (XT == kF32 && WT == kF32 && GT == kF32) {
        MT_BWD_WIDE_PIPE_F32(MT_TRY)
    } else {
        MT_BWD_WIDE_PIPE(MT_TRY)
    }
#undef MT_TRY
    return kNoVectorPlan;
}

// ------------------------------------------------------------ entry points ---
// The dtype combinations the vector kernels cover for activations XT: parameters and
// cotangents each of the activation type or fp32 (all three matching: the full tables;
// otherwise the short ones). All-fp32 uses the full forward tables and its own backward
// table (an fp32 row takes twice the ring). Anything else returns kNoVectorPlan.
// Each (op, XT) pair is instantiated in its own translation unit (ops_<op>_<type>.cu),
// so the kernels compile in parallel.

template <int OP, int XT>
cudaError_t fwd_plan_for(int64_t N, int D, int wdt, LaunchPlan *p) {
    if constexpr (XT == kF32) {
        return (wdt == kF32) ? fwd_plan_vec<OP, kF32, kF32, false>(N, D, p) : kNoVectorPlan;
    } else {
        if (wdt == XT) return fwd_plan_vec<OP, XT, XT, false>(N, D, p);
        if (wdt == kF32) return fwd_plan_vec<OP, XT, kF32, true>(N, D, p);
        return kNoVectorPlan;
    }
}

template <int OP, int XT, int WT, int GT>
cudaError_t bwd_plan_ds(int64_t N, int D, bool has_ds, int device, LaunchPlan *p) {
    constexpr bool SHORT = !(WT == XT && GT == XT) || XT == kF32;
    if constexpr (OP == kAddRms) {
        if (has_ds) return bwd_plan_vec<OP, XT, WT, GT, true, SHORT>(N, D, device, p);
    }
    return bwd_plan_vec<OP, XT, WT, GT, false, SHORT>(N, D, device, p);
}

template <int OP, int XT>
cudaError_t bwd_plan_for(int64_t N, int D, int wdt, int gdt, bool has_ds, int device,
                         LaunchPlan *p) {
    if constexpr (XT == kF32) {
        if (wdt != kF32 || gdt != kF32) return kNoVectorPlan;
        return bwd_plan_ds<OP, kF32, kF32, kF32>(N, D, has_ds, device, p);
    } else {
        const bool w32 = (wdt == kF32), g32 = (gdt == kF32);
        if ((!w32 && wdt != XT) || (!g32 && gdt != XT)) return kNoVectorPlan;
        if (!w32 && !g32) return bwd_plan_ds<OP, XT, XT, XT>(N, D, has_ds, device, p);
        if (!w32 && g32) return bwd_plan_ds<OP, XT, XT, kF32>(N, D, has_ds, device, p);
        if (w32 && !g32) return bwd_plan_ds<OP, XT, kF32, XT>(N, D, has_ds, device, p);
        return bwd_plan_ds<OP, XT, kF32, kF32>(N, D, has_ds, device, p);
    }
}

#define MT_EXTERN_PLANS(OP, XT)                                                            \
    extern template cudaError_t fwd_plan_for<OP, XT>(int64_t, int, int, LaunchPlan *);     \
    extern template cudaError_t bwd_plan_for<OP, XT>(int64_t, int, int, int, bool, int,    \
                                                     LaunchPlan *);
#define MT_INSTANTIATE_PLANS(OP, XT)                                               \
    template cudaError_t fwd_plan_for<OP, XT>(int64_t, int, int, LaunchPlan *);    \
    template cudaError_t bwd_plan_for<OP, XT>(int64_t, int, int, int, bool, int,   \
                                              LaunchPlan *);

#define MT_ALL_PLANS(M) \
    M(kRms, kF16) M(kRms, kBF16) M(kRms, kF32) \
    M(kLayer, kF16) M(kLayer, kBF16) M(kLayer, kF32) \
    M(kAddRms, kF16) M(kAddRms, kBF16) M(kAddRms, kF32)
#ifndef MT_PLANS_TU
MT_ALL_PLANS(MT_EXTERN_PLANS)
#endif

// Scalar plans (ops_scalar.cu).
cudaError_t fwd_plan_scalar_op(int op, int64_t N, int D, LaunchPlan *p);
cudaError_t bwd_plan_scalar_op(int op, int64_t N, int D, bool has_ds, int device, LaunchPlan *p);

}  // namespace mt
