// softmax_api.cu -- launch planning and C entry points of the row softmax / log-softmax
// and the per-row cross-entropy (include/mt_norm.h documents the contracts).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <initializer_list>

#include "launch.cuh"
#include "mt_norm.h"
#include "softmax.cuh"

namespace mt {
namespace {

// Softmax shapes, X(max_D, TPR, RPC, CH): 8-element chunks for aligned rows (a warp per
// row up to 1024 columns, one CTA per row above), single elements otherwise.
#ifndef MT_SOFTMAX_SHAPES_VEC8
#define MT_SOFTMAX_SHAPES_VEC8(X) \
    X(256, 32, 4, 1)              \
    X(1024, 32, 4, 4)             \
    X(4096, 128, 1, 4)            \
    X(16384, 512, 1, 4)
#endif
// Rows wider than 16384 (up to MT_MAX_SOFTMAX_COLS): the two-pass streaming kernels,
// X(max_D, TPR, UN, MINB): one CTA of TPR threads per row, UN chunks (or elements) in
// flight per thread and operand (the backward loads two operands; fp32 rows take half as
// many chunks, the same bytes), MINB the resident-CTA floor per SM the kernel is compiled
// for (1: none). Measured on GB300 (forward / backward, us): 2048 x 32768 fp16 47.0 / 73.6
// (backward at 256 threads 77.3); 1024 x 65536 fp16 52.8 / 92.8 (256 threads 54.8 / 94.4,
// 128 threads 60.4 / 105.8); 512 x 131072 bf16 forward 56.5 at 2 chunks, 62.5 at 4;
// 256 x 262144 fp16 forward 58.1 - 61.5 at 4 chunks, 61.5 at 2, 63.0 at 512 threads;
// floors of 2 or 4 resident CTAs per SM did not help.
// The forward's entries add CIT, the batches of UN chunks per thread kept in shared memory
// between the passes (softmax_stream_fwd_kernel; 0: none): rows wider than 131072 keep
// their first 3 of 8 batches (192 KB of an fp16 row), one CTA per SM.
#ifndef MT_SOFTMAX_SHAPES_STREAM_FWD
#define MT_SOFTMAX_SHAPES_STREAM_FWD(X) \
    X(65536, 512, 4, 1, 0)              \
    X(131072, 1024, 2, 1, 0)            \
    X(MT_MAX_SOFTMAX_COLS, 1024, 4, 1, 3)
#endif
// Backward of rows wider than 65536: split over a thread-block cluster of CL = 2, 4 or 8
// CTAs (the smallest power of two whose slices of ceil(D / CL) columns fit the cap),
// X(cap, TPR, UN, MINB) per CTA. Measured on GB300 (backward, us): 256 x 262144 fp16
// 93.8 unsplit, 84.5 with 65536-column slices, 81.4 with 32768; 512 x 131072 bf16 80.3,
// 84.4, 78.4; 2048 x 131072 fp16 277.6, 285.6, 266.6.
#ifndef MT_SOFTMAX_SHAPES_STREAM_CLU_BWD
#define MT_SOFTMAX_SHAPES_STREAM_CLU_BWD(X) X(32768, 512, 4, 1)
#endif
#ifndef MT_SOFTMAX_SHAPES_STREAM_BWD
#define MT_SOFTMAX_SHAPES_STREAM_BWD(X) X(65536, 512, 2, 1)
#endif
#define MT_SOFTMAX_SHAPES_SCALAR(X) \
    X(256, 32, 4, 8)                \
    X(1024, 32, 4, 32)              \
    X(4096, 256, 1, 16)             \
    X(16384, 1024, 1, 16)

// Cross-entropy: X(max_D, TPR, RPC, MINB, UN): a row group of TPR threads per row, RPC
// rows per CTA (one-warp row groups only), MINB a floor on resident CTAs per SM for the
// register allocator (0: the compiler's choice), UN chunks in flight per thread. Narrow
// row groups with many chunks per thread, narrower still in the forward (whose
// per-element work is larger): each entry measured on GB300 against its neighbours
// (forward of 4096 x 32768 bf16: 128 threads 55.8 us, 256 threads 59.3 us, 512 threads
// 92.5 us, and 8 chunks in flight 54.1 us against 4; forward of 16384 x 4096: one warp
// per row, four rows per CTA, 35.2 us, 64 threads 39.0 us, 256 threads 80.1 us; 8 chunks
// in flight lose at 1024 columns: 53.4 us against 47.3 us for 65536 rows).
#ifndef MT_CE_FWD_SHAPES
#define MT_CE_FWD_SHAPES(X) \
    X(1024, 32, 2, 0, 4)    \
    X(4096, 32, 4, 0, 4)    \
    X(16384, 64, 1, 0, 8)   \
    X(MT_MAX_CE_COLS, 128, 1, 0, 8)
#endif
#ifndef MT_CE_BWD_SHAPES
#define MT_CE_BWD_SHAPES(X) \
    X(1024, 32, 4, 0, 4)    \
    X(4096, 64, 1, 0, 8)    \
    X(16384, 128, 1, 0, 8)  \
    X(MT_MAX_CE_COLS, 256, 1, 0, 4)
#endif

mt_status_t fail(cudaError_t e) {
    record_cuda_error(e);
    return MT_ERR_CUDA;
}

bool valid_dtype(int dt) { return dt == kF16 || dt == kBF16 || dt == kF32; }
size_t dtype_bytes(int dt) { return dt == kF32 ? 4 : 2; }

bool aligned16(std::initializer_list<const void *> ptrs) {
    for (const void *p : ptrs)
        if (p != nullptr && ((uintptr_t)p & 15u) != 0) return false;
    return true;
}

struct Span {
    const void *p;
    size_t bytes;
};
bool overlaps(std::initializer_list<Span> outs, std::initializer_list<Span> ins) {
    auto hit = [](const Span &a, const Span &b) {
        if (!a.p || !b.p || !a.bytes || !b.bytes) return false;
        const uintptr_t x = (uintptr_t)a.p, y = (uintptr_t)b.p;
        return x < y + b.bytes && y < x + a.bytes;
    };
    for (auto o = outs.begin(); o != outs.end(); ++o) {
        for (const Span &i : ins)
            if (hit(*o, i)) return true;
        for (auto o2 = o + 1; o2 != outs.end(); ++o2)
            if (hit(*o, *o2)) return true;
    }
    return false;
}

template <bool BWD, bool LOG, int XT>
cudaError_t softmax_plan_vec(int64_t N, int D, LaunchPlan *p) {
#define MT_TRY(maxd, tpr, rpc, ch)                                                            \
    if (D <= maxd) {                                                                          \
        p->kernel = BWD ? reinterpret_cast<const void *>(&softmax_bwd_vec8_kernel<tpr, rpc, ch, LOG, XT>) \
                        : reinterpret_cast<const void *>(&softmax_fwd_vec8_kernel<tpr, rpc, ch, LOG, XT>); \
        p->threads = tpr * rpc;                                                               \
        p->grid = (int)((N + rpc - 1) / rpc);                                                 \
        p->rows_per_cta = rpc;                                                                \
        return cudaSuccess;                                                                   \
    }
    MT_SOFTMAX_SHAPES_VEC8(MT_TRY)
#undef MT_TRY
    return cudaErrorInvalidValue;
}

template <bool BWD, bool LOG>
cudaError_t softmax_plan_scalar(int64_t N, int D, LaunchPlan *p) {
#define MT_TRY(maxd, tpr, rpc, ch)                                                                   \
    if (D <= maxd) {                                                                                 \
        p->kernel = reinterpret_cast<const void *>(&softmax_scalar_kernel<tpr, rpc, ch, LOG, BWD>);  \
        p->threads = tpr * rpc;                                                                      \
        p->grid = (int)((N + rpc - 1) / rpc);                                                        \
        p->rows_per_cta = rpc;                                                                       \
        return cudaSuccess;                                                                          \
    }
    MT_SOFTMAX_SHAPES_SCALAR(MT_TRY)
#undef MT_TRY
    return cudaErrorInvalidValue;
}

template <bool BWD, bool LOG, bool VEC8, int XT>
cudaError_t softmax_plan_stream(int64_t N, int D, LaunchPlan *p) {
    if constexpr (BWD) {
#define MT_TRY(cap, tpr, un, minb)                                                                  \
    if (D > 65536 && wide_split(D, cap, &p->cluster, &p->slice)) {                                  \
        p->kernel = reinterpret_cast<const void *>(                                                 \
            &softmax_stream_bwd_kernel<tpr, VEC8, XT, LOG, stream_un(XT, un), minb, true>);         \
        p->threads = tpr;                                                                           \
        p->rows_per_cta = 1;                                                                        \
        return cluster_row_grid(p, N);                                                              \
    }
        MT_SOFTMAX_SHAPES_STREAM_CLU_BWD(MT_TRY)
#undef MT_TRY
    }
#define MT_TRY(maxd, tpr, un, minb)                                                                 \
    if (D <= maxd) {                                                                                \
        p->kernel = reinterpret_cast<const void *>(&softmax_stream_bwd_kernel<tpr, VEC8, XT, LOG, stream_un(XT, un), minb>); \
        p->threads = tpr;                                                                           \
        p->grid = (int)N;                                                                           \
        p->rows_per_cta = 1;                                                                        \
        return cudaSuccess;                                                                         \
    }
#define MT_TRY_F(maxd, tpr, un, minb, cit)                                                          \
    if (D <= maxd) {                                                                                \
        constexpr int cu = VEC8 ? chunk_units<XT>() : 1;                                            \
        constexpr int c = VEC8 ? cit : 0;                                                           \
        p->kernel = reinterpret_cast<const void *>(                                                 \
            &softmax_stream_fwd_kernel<tpr, VEC8, XT, LOG, stream_un(XT, un), minb, c>);            \
        p->threads = tpr;                                                                           \
        p->grid = (int)N;                                                                           \
        p->rows_per_cta = 1;                                                                        \
        p->smem = (size_t)c * stream_un(XT, un) * cu * tpr * 16;                                    \
        if (p->smem > 0) {                                                                          \
            int device = 0, per_sm = 0;                                                             \
            cudaError_t e = cudaGetDevice(&device);                                                 \
            if (e == cudaSuccess) e = cached_occupancy(p->kernel, tpr, p->smem, device, &per_sm);   \
            return e;                                                                               \
        }                                                                                           \
        return cudaSuccess;                                                                         \
    }
    if constexpr (BWD) {
        MT_SOFTMAX_SHAPES_STREAM_BWD(MT_TRY)
    } else {
        MT_SOFTMAX_SHAPES_STREAM_FWD(MT_TRY_F)
    }
#undef MT_TRY
#undef MT_TRY_F
    return cudaErrorInvalidValue;
}

template <bool BWD, bool LOG>
cudaError_t softmax_plan(int64_t N, int D, bool vec8, int xdt, LaunchPlan *p) {
    if (D > 16384) {
        if (!vec8) return softmax_plan_stream<BWD, LOG, false, kF32>(N, D, p);  // types at run time
        if (xdt == kF16) return softmax_plan_stream<BWD, LOG, true, kF16>(N, D, p);
        if (xdt == kBF16) return softmax_plan_stream<BWD, LOG, true, kBF16>(N, D, p);
        return softmax_plan_stream<BWD, LOG, true, kF32>(N, D, p);
    }
    if (vec8) {
        if (xdt == kF16) return softmax_plan_vec<BWD, LOG, kF16>(N, D, p);
        if (xdt == kBF16) return softmax_plan_vec<BWD, LOG, kBF16>(N, D, p);
        return softmax_plan_vec<BWD, LOG, kF32>(N, D, p);
    }
    return softmax_plan_scalar<BWD, LOG>(N, D, p);
}

template <bool BWD, bool VEC8, int XT>
cudaError_t ce_plan_t(int64_t N, int D, LaunchPlan *p) {
#define MT_TRY(maxd, tpr, rpc, minb, un)                                                            \
    if (D <= maxd) {                                                                                \
        if constexpr (BWD)                                                                          \
            p->kernel = reinterpret_cast<const void *>(&ce_bwd_kernel<tpr, rpc, VEC8, XT, minb, un>); \
        else                                                                                        \
            p->kernel = reinterpret_cast<const void *>(&ce_fwd_kernel<tpr, rpc, VEC8, XT, minb, un>); \
        p->threads = tpr * rpc;                                                                     \
        p->grid = (int)((N + rpc - 1) / rpc);                                                       \
        p->rows_per_cta = rpc;                                                                      \
        return cudaSuccess;                                                                         \
    }
    if constexpr (BWD) {
        MT_CE_BWD_SHAPES(MT_TRY)
    } else {
        MT_CE_FWD_SHAPES(MT_TRY)
    }
#undef MT_TRY
    return cudaErrorInvalidValue;
}

template <bool BWD>
cudaError_t ce_plan(int64_t N, int D, bool vec8, int xdt, LaunchPlan *p) {
    if (!vec8) return ce_plan_t<BWD, false, kF32>(N, D, p);  // scalar: the type is read at run time
    if (xdt == kF16) return ce_plan_t<BWD, true, kF16>(N, D, p);
    if (xdt == kBF16) return ce_plan_t<BWD, true, kBF16>(N, D, p);
    return ce_plan_t<BWD, true, kF32>(N, D, p);
}

// N = 0 is a valid, empty batch.
mt_status_t check_rows(int64_t N, int64_t D, int64_t max_cols) {
    if (N < 0 || D < 1) return MT_ERR_INVALID_ARG;
    if (D > max_cols || N > (int64_t)INT32_MAX) return MT_ERR_UNSUPPORTED;
    return MT_OK;
}

mt_status_t softmax_impl(bool bwd, int dt, const void *in, const void *dY, void *out, int64_t N,
                         int64_t D, int log_softmax, mt_stream_t stream) {
    if (!valid_dtype(dt)) return MT_ERR_INVALID_ARG;
    mt_status_t s = check_rows(N, D, MT_MAX_SOFTMAX_COLS);
    if (s != MT_OK) return s;
    if (N == 0) return MT_OK;
    if (!in || !out || (bwd && !dY)) return MT_ERR_INVALID_ARG;
    const size_t act = (size_t)N * (size_t)D * dtype_bytes(dt);
    if (overlaps({{out, act}}, {{in, act}, {dY, bwd ? act : 0}})) return MT_ERR_INVALID_ARG;
    SoftmaxArgs a{};
    a.X = in;
    a.dY = dY;
    a.Y = out;
    a.N = N;
    a.D = (int)D;
    a.xdt = dt;
    a.gdt = dt;
    const bool vec8 = (D % 8 == 0) && aligned16({in, dY, out});
    LaunchPlan p;
    const bool log = log_softmax != 0;
    const cudaError_t e = bwd ? (log ? softmax_plan<true, true>(N, (int)D, vec8, dt, &p)
                                     : softmax_plan<true, false>(N, (int)D, vec8, dt, &p))
                              : (log ? softmax_plan<false, true>(N, (int)D, vec8, dt, &p)
                                     : softmax_plan<false, false>(N, (int)D, vec8, dt, &p));
    if (e != cudaSuccess) return fail(e);
    a.slice = p.slice;
    const cudaError_t le = launch_pdl(p, &a, reinterpret_cast<cudaStream_t>(stream));
    return le == cudaSuccess ? MT_OK : fail(le);
}

mt_status_t check_ce_options(int reduction, float label_smoothing, float z_loss) {
    if (reduction != MT_REDUCTION_NONE && reduction != MT_REDUCTION_SUM &&
        reduction != MT_REDUCTION_MEAN)
        return MT_ERR_INVALID_ARG;
    if (!std::isfinite(label_smoothing) || label_smoothing < 0.f || label_smoothing > 1.f)
        return MT_ERR_INVALID_ARG;
    if (!std::isfinite(z_loss) || z_loss < 0.f) return MT_ERR_INVALID_ARG;
    return MT_OK;
}

}  // namespace
}  // namespace mt

using namespace mt;

extern "C" mt_status_t mt_softmax_forward(mt_dtype_t dtype, const void *X, void *Y, int64_t N,
                                          int64_t D, int log_softmax, mt_stream_t stream) {
    return softmax_impl(false, (int)dtype, X, nullptr, Y, N, D, log_softmax, stream);
}

extern "C" mt_status_t mt_softmax_backward(mt_dtype_t dtype, const void *Y, const void *dY,
                                           void *dX, int64_t N, int64_t D, int log_softmax,
                                           mt_stream_t stream) {
    return softmax_impl(true, (int)dtype, Y, dY, dX, N, D, log_softmax, stream);
}

extern "C" mt_status_t mt_cross_entropy_forward(mt_dtype_t dtype, const void *logits,
                                                const int64_t *targets, int64_t N, int64_t D,
                                                int64_t ignore_index, float label_smoothing,
                                                float z_loss, mt_reduction_t reduction,
                                                float *loss_rows, float *lse, float *loss_out,
                                                float *n_valid, mt_stream_t stream) {
    const int dt = (int)dtype;
    const bool reduce = reduction != MT_REDUCTION_NONE;
    if (!valid_dtype(dt)) return MT_ERR_INVALID_ARG;
    mt_status_t s = check_ce_options((int)reduction, label_smoothing, z_loss);
    if (s != MT_OK) return s;
    if ((s = check_rows(N, D, MT_MAX_CE_COLS)) != MT_OK) return s;
    if (reduce && (!loss_out || !n_valid || loss_out == n_valid)) return MT_ERR_INVALID_ARG;
    if (N == 0) {
        // an empty batch: the sum is 0, the mean over no valid row is 0 (as when every
        // row is ignored), and no row is valid
        if (!reduce) return MT_OK;
        cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
        cudaError_t e = cudaMemsetAsync(loss_out, 0, sizeof(float), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(n_valid, 0, sizeof(float), st);
        return e == cudaSuccess ? MT_OK : fail(e);
    }
    if (!logits || !targets || !loss_rows || !lse) return MT_ERR_INVALID_ARG;
    const size_t act = (size_t)N * (size_t)D * dtype_bytes(dt), row = (size_t)N * 4;
    if (!reduce) { loss_out = nullptr; n_valid = nullptr; }
    if (overlaps({{loss_rows, row}, {lse, row}, {loss_out, 4}, {n_valid, 4}},
                 {{logits, act}, {targets, (size_t)N * 8}}))
        return MT_ERR_INVALID_ARG;
    CeArgs a{};
    a.X = logits;
    a.T = targets;
    a.loss = loss_rows;
    a.lse = lse;
    a.N = N;
    a.D = (int)D;
    a.ignore_index = ignore_index;
    a.eps = label_smoothing;
    a.z = z_loss;
    a.reduction = (int)reduction;
    a.xdt = dt;
    const bool vec8 = (D % 8 == 0) && aligned16({logits});
    LaunchPlan p;
    cudaError_t e = ce_plan<false>(N, (int)D, vec8, dt, &p);
    if (e != cudaSuccess) return fail(e);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((e = launch_pdl(p, &a, st)) != cudaSuccess) return fail(e);
    if (reduce) {
        constexpr int B = 1024;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(B);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const float *cl = loss_rows;
        e = launch_hook();
        if (e == cudaSuccess)
            e = cudaLaunchKernelEx(&cfg, ce_loss_reduce_kernel<B>, cl, targets, N, ignore_index,
                                   (int)reduction, loss_out, n_valid);
        if (e != cudaSuccess) return fail(e);
    }
    return MT_OK;
}

extern "C" mt_status_t mt_cross_entropy_backward(mt_dtype_t dtype, const void *logits,
                                                 const int64_t *targets, const float *lse,
                                                 int64_t N, int64_t D, int64_t ignore_index,
                                                 float label_smoothing, float z_loss,
                                                 mt_reduction_t reduction, const float *dloss,
                                                 const float *n_valid, void *dlogits,
                                                 mt_stream_t stream) {
    const int dt = (int)dtype;
    if (!valid_dtype(dt)) return MT_ERR_INVALID_ARG;
    mt_status_t s = check_ce_options((int)reduction, label_smoothing, z_loss);
    if (s != MT_OK) return s;
    if ((s = check_rows(N, D, MT_MAX_CE_COLS)) != MT_OK) return s;
    if (N == 0) return MT_OK;  // an empty batch: no logit gradient to write
    if (!logits || !targets || !lse || !dloss || !dlogits ||
        (reduction == MT_REDUCTION_MEAN && !n_valid))
        return MT_ERR_INVALID_ARG;
    const size_t act = (size_t)N * (size_t)D * dtype_bytes(dt), row = (size_t)N * 4;
    const size_t dl = (reduction == MT_REDUCTION_NONE) ? row : 4;
    if (overlaps({{dlogits, act}}, {{logits, act}, {targets, (size_t)N * 8}, {lse, row},
                                    {dloss, dl}, {n_valid, n_valid ? 4u : 0u}}))
        return MT_ERR_INVALID_ARG;
    CeArgs a{};
    a.X = logits;
    a.T = targets;
    a.lse = const_cast<float *>(lse);
    a.dloss = dloss;
    a.n_valid = n_valid;
    a.dX = dlogits;
    a.N = N;
    a.D = (int)D;
    a.ignore_index = ignore_index;
    a.eps = label_smoothing;
    a.z = z_loss;
    a.reduction = (int)reduction;
    a.xdt = dt;
    const bool vec8 = (D % 8 == 0) && aligned16({logits, dlogits});
    LaunchPlan p;
    cudaError_t e = ce_plan<true>(N, (int)D, vec8, dt, &p);
    if (e != cudaSuccess) return fail(e);
    if ((e = launch_pdl(p, &a, reinterpret_cast<cudaStream_t>(stream))) != cudaSuccess)
        return fail(e);
    return MT_OK;
}
