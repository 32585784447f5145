// gemv_api.cu -- launch planning and C entry points of the fused normalization + GEMV
// (include/mt_norm.h documents the contracts; gemv.cuh the kernel).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "gemv.cuh"
#include "launch.cuh"
#include "mt_norm.h"

namespace mt {
namespace {

// Features per CTA at most: two 8-feature chunks per thread (kGemvSliceChunks); the
// normalized slice (slice x 8 rows x 4 bytes) stays within 128 KB of shared memory.
constexpr int kGemvMaxSlice = kGemvSliceChunks * 8 * kGemvWarps * 32;

// Features per CTA for a cluster of cl: ceil(K / cl) rounded up to whole 8-feature chunks.
int gemv_slice(int K, int cl) { return ((K + cl - 1) / cl + 7) / 8 * 8; }
// W ring stages per thread (features in flight + 1), and the CTAs per SM the launch
// shape aims for.
#ifndef MT_GEMV_STAGES
#define MT_GEMV_STAGES 12
#endif
#ifndef MT_GEMV_CTAS_PER_SM
#define MT_GEMV_CTAS_PER_SM 2
#endif
constexpr int kGemvStages = MT_GEMV_STAGES;

mt_status_t gemv_fail(cudaError_t e) {
    record_cuda_error(e);
    return MT_ERR_CUDA;
}

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

template <int OP, int MT, int LPF, bool VEC>
const void *gemv_kernel() {
    return reinterpret_cast<const void *>(&norm_gemv_kernel<OP, MT, LPF, kGemvStages, VEC>);
}

template <int OP, int MT>
cudaError_t gemv_pick(int lpf, bool vec, int slice, LaunchPlan *p) {
    if (!vec) {
        p->kernel = gemv_kernel<OP, MT, 32, false>();
        p->smem = gemv_smem<MT, 32, kGemvStages>(slice);
        return cudaSuccess;
    }
    if (lpf == 32) {
        p->kernel = gemv_kernel<OP, MT, 32, true>();
        p->smem = gemv_smem<MT, 32, kGemvStages>(slice);
    } else if (lpf == 16) {
        p->kernel = gemv_kernel<OP, MT, 16, true>();
        p->smem = gemv_smem<MT, 16, kGemvStages>(slice);
    } else {
        p->kernel = gemv_kernel<OP, MT, 8, true>();
        p->smem = gemv_smem<MT, 8, kGemvStages>(slice);
    }
    return cudaSuccess;
}

template <int OP>
cudaError_t gemv_pick_rows(int M, int lpf, bool vec, int slice, LaunchPlan *p) {
    switch (M) {
        case 1: return gemv_pick<OP, 1>(lpf, vec, slice, p);
        case 2: return gemv_pick<OP, 2>(lpf, vec, slice, p);
        case 3: return gemv_pick<OP, 3>(lpf, vec, slice, p);
        case 4: return gemv_pick<OP, 4>(lpf, vec, slice, p);
        default: return gemv_pick<OP, 8>(lpf, vec, slice, p);
    }
}

// Launch shape: the widest column tile (lanes per feature 32, 16, 8) and the smallest
// cluster along K that give at least MT_GEMV_CTAS_PER_SM CTAs per SM, with at most kGemvMaxSlice
// features per CTA and, where K allows, at least four features per feature group.
cudaError_t gemv_plan(int op, int M, int N, int K, bool vec, int device, LaunchPlan *p,
                      int *slice) {
    int sms = 0;
    cudaError_t e = device_sm_count(device, &sms);
    if (e != cudaSuccess) return e;
    const int64_t want = MT_GEMV_CTAS_PER_SM * (int64_t)sms;
    int lpf = 32;
    if (vec) {
        while (lpf > 8 && (int64_t)((N + 8 * lpf - 1) / (8 * lpf)) * kMaxCluster < want) lpf /= 2;
    }
    const int64_t tiles = (N + 8 * lpf - 1) / (8 * lpf);
    const int fg = kGemvWarps * (32 / lpf);
    int cl = 1;
    while (cl < kMaxCluster && (tiles * cl < want || gemv_slice(K, cl) > kGemvMaxSlice)) cl *= 2;
    while (cl > 1 && gemv_slice(K, cl) < 4 * fg && gemv_slice(K, cl / 2) <= kGemvMaxSlice)
        cl /= 2;
    *slice = gemv_slice(K, cl);
    if (*slice > kGemvMaxSlice || tiles * cl > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
    e = (op == kRms) ? gemv_pick_rows<kRms>(M, lpf, vec, *slice, p)
                     : gemv_pick_rows<kLayer>(M, lpf, vec, *slice, p);
    if (e != cudaSuccess) return e;
    p->threads = kGemvWarps * 32;
    p->grid = (int)(tiles * cl);
    p->cluster = cl;
    p->rows_per_cta = M;
    int per_sm = 0;  // raises the kernel's dynamic shared memory limit to p->smem
    return cached_occupancy(p->kernel, p->threads, p->smem, device, &per_sm);
}

mt_status_t norm_gemv_impl(int op, const void *X, const void *gamma, const void *beta,
                           const void *W, void *Y, int64_t M, int64_t N, int64_t K, float eps,
                           mt_stream_t stream) {
    if (M < 0 || N < 0 || K < 1) return MT_ERR_INVALID_ARG;
    if (M > MT_MAX_GEMV_ROWS || K > MT_MAX_GEMV_K || N > (int64_t)INT32_MAX)
        return MT_ERR_UNSUPPORTED;
    if (!(std::isfinite(eps) && eps > 0.f)) return MT_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return MT_OK;  // an empty output: nothing to read or write
    if (!X || !gamma || !W || !Y || (op == kLayer && !beta)) return MT_ERR_INVALID_ARG;
    const size_t ybytes = (size_t)M * (size_t)N * 2;
    if (overlap(Y, ybytes, X, (size_t)M * (size_t)K * 2) || overlap(Y, ybytes, gamma, (size_t)K * 2) ||
        overlap(Y, ybytes, op == kLayer ? beta : nullptr, (size_t)K * 2) ||
        overlap(Y, ybytes, W, (size_t)K * (size_t)N * 2))
        return MT_ERR_INVALID_ARG;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return gemv_fail(e);
    const bool vec = (N % 8 == 0) && (((uintptr_t)W & 15u) == 0);
    const bool a16 = (((uintptr_t)X | (uintptr_t)gamma | (uintptr_t)(op == kLayer ? beta : gamma)) &
                      15u) == 0;
    LaunchPlan p;
    int slice = 0;
    if ((e = gemv_plan(op, (int)M, (int)N, (int)K, vec, device, &p, &slice)) != cudaSuccess)
        return gemv_fail(e);
    GemvArgs a{};
    a.X = X;
    a.gamma = gamma;
    a.beta = op == kLayer ? beta : gamma;
    a.W = W;
    a.Y = Y;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.slice = slice;
    a.eps = eps;
    a.xvec = (K % 8 == 0) && a16;
    e = launch_pdl(p, &a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MT_OK : gemv_fail(e);
}

}  // namespace
}  // namespace mt

using namespace mt;

extern "C" mt_status_t mt_fused_rmsnorm_gemv(const void *X, const void *gamma, const void *W,
                                             void *Y, int64_t M, int64_t N, int64_t K, float eps,
                                             mt_stream_t stream) {
    return norm_gemv_impl(kRms, X, gamma, nullptr, W, Y, M, N, K, eps, stream);
}

extern "C" mt_status_t mt_fused_layernorm_gemv(const void *X, const void *gamma, const void *beta,
                                               const void *W, void *Y, int64_t M, int64_t N,
                                               int64_t K, float eps, mt_stream_t stream) {
    return norm_gemv_impl(kLayer, X, gamma, beta, W, Y, M, N, K, eps, stream);
}
