// gemv_api.cu -- launch planning and C entry points of the fused normalization + GEMV
// (include/mt_norm.h documents the contracts; gemv.cuh the kernel).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "gemv.cuh"
#include "launch.cuh"
#include "mt_norm.h"

namespace mt {
namespace {

// Input features per slice at most (two 8-feature chunks per thread build its normalized
// rows).
constexpr int kGemvMaxSlice = kGemvSliceChunks * 8 * kGemvWarps * 32;

// W ring stages per thread (features in flight + 1).
#ifndef MT_GEMV_STAGES
#define MT_GEMV_STAGES 12
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
void gemv_set(int slice, LaunchPlan *p) {
    p->kernel = reinterpret_cast<const void *>(&norm_gemv_kernel<OP, MT, LPF, kGemvStages, VEC>);
    p->smem = gemv_smem<MT, LPF, kGemvStages>(slice);
}

template <int OP, int MT>
void gemv_pick(int lpf, bool vec, int slice, LaunchPlan *p) {
    if (!vec) return gemv_set<OP, MT, 32, false>(slice, p);  // per-element W loads
    if (lpf == 32) return gemv_set<OP, MT, 32, true>(slice, p);
    if (lpf == 16) return gemv_set<OP, MT, 16, true>(slice, p);
    return gemv_set<OP, MT, 8, true>(slice, p);
}

template <int OP>
void gemv_pick_rows(int M, int lpf, bool vec, int slice, LaunchPlan *p) {
    switch (M) {
        case 1: return gemv_pick<OP, 1>(lpf, vec, slice, p);
        case 2: return gemv_pick<OP, 2>(lpf, vec, slice, p);
        case 3: return gemv_pick<OP, 3>(lpf, vec, slice, p);
        case 4: return gemv_pick<OP, 4>(lpf, vec, slice, p);
        default: return gemv_pick<OP, 8>(lpf, vec, slice, p);
    }
}

// Split-K launch shape: tiles of 8 * LPF columns (LPF 32 for N >= 1024, narrower for
// narrow outputs; 32 for per-element loads), and the number of slices (each thread
// keeping at least four features, each slice at most kGemvMaxSlice of them): the fewest
// waves of resident CTAs whose last wave is at least 90% full, else the best-filled grid.
// (Measured on GB300 against always taking the best-filled grid: M = 2, 8192 x 14336
// 52.2 -> 46.7 us, M = 8, 4096 x 4096 28.5 -> 25.4 us; the bench's decode shapes within 1%.)
cudaError_t gemv_plan(int op, int M, int N, int K, bool vec, int device, LaunchPlan *p,
                      int *slice, int *ks, int *ntiles) {
    int sms = 0;
    cudaError_t e = device_sm_count(device, &sms);
    if (e != cudaSuccess) return e;
    const int lpf = !vec ? 32 : N >= 1024 ? 32 : N >= 256 ? 16 : 8;
    const int64_t tiles = (N + 8 * lpf * kGemvCpl - 1) / (8 * lpf * kGemvCpl);
    const int fg = kGemvWarps * (32 / lpf);
    const int64_t kmin = std::max<int64_t>(1, (K + kGemvMaxSlice - 1) / kGemvMaxSlice);
    const int64_t kmax = std::max<int64_t>(kmin, (K + 4 * fg - 1) / (4 * fg));
    auto slice_of = [&](int64_t k) { return (int)(((K + k - 1) / k + 7) / 8 * 8); };
    // resident CTAs (the shared memory differs little with the slice: take the largest)
    if (op == kRms) gemv_pick_rows<kRms>(M, lpf, vec, slice_of(kmin), p);
    else gemv_pick_rows<kLayer>(M, lpf, vec, slice_of(kmin), p);
    int per_sm = 0;
    if ((e = cached_occupancy(p->kernel, kGemvWarps * 32, p->smem, device, &per_sm)) != cudaSuccess)
        return e;
    const int64_t cap = (int64_t)std::max(per_sm, 1) * sms;
    int64_t best_k = kmin;
    double best_fill = -1.0;
    for (int64_t k = kmin; k <= std::min<int64_t>(kmax, 4 * cap); ++k) {
        const int64_t kk = (K + slice_of(k) - 1) / slice_of(k);  // slices actually used
        const int64_t ctas = tiles * kk;
        if (ctas > 8 * cap) break;
        const double fill = (double)ctas / (double)(((ctas + cap - 1) / cap) * cap);
        if (best_fill < 0.9 && fill > best_fill + 1e-9) {
            best_fill = fill;
            best_k = kk;
        }
    }
    const int sl = slice_of(best_k);
    const int64_t k = (K + sl - 1) / sl;
    if (sl > kGemvMaxSlice || tiles * k > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
    if (op == kRms) gemv_pick_rows<kRms>(M, lpf, vec, sl, p);
    else gemv_pick_rows<kLayer>(M, lpf, vec, sl, p);
    p->threads = kGemvWarps * 32;
    p->grid = (int)(tiles * k);
    p->rows_per_cta = M;
    *slice = sl;
    *ks = (int)k;
    *ntiles = (int)tiles;
    // raises the kernel's dynamic shared memory limit to p->smem
    return cached_occupancy(p->kernel, p->threads, p->smem, device, &per_sm);
}

mt_status_t norm_gemv_impl(int op, const void *X, const void *gamma, const void *beta,
                           const void *W, void *Y, int64_t M, int64_t N, int64_t K, float eps,
                           mt_stream_t stream_in) {
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
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_in);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return gemv_fail(e);
    const bool vec = (N % 8 == 0) && (((uintptr_t)W & 15u) == 0);
    const bool a16 = (((uintptr_t)X | (uintptr_t)gamma | (uintptr_t)(op == kLayer ? beta : gamma)) &
                      15u) == 0;
    LaunchPlan p;
    int slice = 0, ks = 0, tiles = 0;
    e = gemv_plan(op, (int)M, (int)N, (int)K, vec, device, &p, &slice, &ks, &tiles);
    if (e != cudaSuccess) return gemv_fail(e);
    // stream-ordered scratch: the statistics, the tile counters, the fp32 partial rows
    const size_t stats_bytes = 256;
    const size_t count_bytes = ((size_t)tiles * sizeof(unsigned) + 255) / 256 * 256;
    const size_t part_bytes = (size_t)ks * (size_t)M * (size_t)N * sizeof(float);
    void *ws = nullptr;
    if ((e = cudaMallocAsync(&ws, stats_bytes + count_bytes + part_bytes, stream)) != cudaSuccess)
        return gemv_fail(e);
    GemvArgs a{};
    a.X = X;
    a.gamma = gamma;
    a.beta = op == kLayer ? beta : gamma;
    a.W = W;
    a.Y = Y;
    a.stats = static_cast<float *>(ws);
    a.count = reinterpret_cast<unsigned *>(static_cast<char *>(ws) + stats_bytes);
    a.part = reinterpret_cast<float *>(static_cast<char *>(ws) + stats_bytes + count_bytes);
    a.tiles = tiles;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.slice = slice;
    a.ks = ks;
    a.eps = eps;
    a.xvec = (K % 8 == 0) && a16;
    LaunchPlan st;
    st.kernel = op == kRms ? reinterpret_cast<const void *>(&gemv_stats_kernel<kRms>)
                           : reinterpret_cast<const void *>(&gemv_stats_kernel<kLayer>);
    st.threads = kGemvStatsThreads;
    st.grid = (int)M;
    e = launch_pdl(st, &a, stream);
    if (e == cudaSuccess) e = launch_pdl(p, &a, stream);
    const cudaError_t fe = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = fe;
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
