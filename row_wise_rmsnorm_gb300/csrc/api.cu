// api.cu -- the C ABI declared in include/mt_norm.h.
//
// Host side only: argument validation (before any CUDA call, so that every
// argument error is reported the same way with or without a GPU), choice of the
// vectorised or scalar kernel, backward workspace sizing, and launches on the
// caller's stream. There is no CPU path: every step of the computation runs in the
// kernels of kernels.cuh.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "launch.cuh"
#include "reduce.cuh"
#include "mt_norm.h"

namespace mt {
namespace {

thread_local int g_last_cuda_error = 0;

mt_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return MT_ERR_CUDA;
}

struct Buf {
    const void *p;
    size_t bytes;
};

bool overlap(const Buf &a, const Buf &b) {
    if (a.p == nullptr || b.p == nullptr || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t x = (uintptr_t)a.p, y = (uintptr_t)b.p;
    return x < y + b.bytes && y < x + a.bytes;
}

// True if an output overlaps an input or another output.
bool any_overlap(std::initializer_list<Buf> outs, std::initializer_list<Buf> ins) {
    for (auto o = outs.begin(); o != outs.end(); ++o) {
        for (const Buf &i : ins)
            if (overlap(*o, i)) return true;
        for (auto o2 = o + 1; o2 != outs.end(); ++o2)
            if (overlap(*o, *o2)) return true;
    }
    return false;
}

mt_status_t check_shape(int64_t N, int64_t D) {
    if (N < 1 || D < 1) return MT_ERR_INVALID_ARG;
    if (D > MT_MAX_COLS || N > (int64_t)INT32_MAX) return MT_ERR_UNSUPPORTED;
    return MT_OK;
}

mt_status_t check_eps(float eps) {
    return (std::isfinite(eps) && eps > 0.f) ? MT_OK : MT_ERR_INVALID_ARG;
}

bool aligned16(std::initializer_list<const void *> ptrs) {
    for (const void *p : ptrs)
        if (p != nullptr && ((uintptr_t)p & 15u) != 0) return false;
    return true;
}

std::mutex g_cache_mu;
std::map<int, int> g_sm_count;
std::map<std::tuple<const void *, int, size_t, int>, int> g_occupancy;

// Every launch carries the programmatic-stream-serialization attribute (see pdl_enter()
// in kernels.cuh).
mt_status_t launch(const LaunchPlan &p, void *arg, cudaStream_t stream) {
    if (p.kernel == nullptr || p.grid < 1) return cuda_fail(cudaErrorInvalidConfiguration);
    void *args[] = {arg};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelExC(&cfg, p.kernel, args);
    if (e != cudaSuccess) return cuda_fail(e);
    return MT_OK;
}

mt_status_t run_forward(int op, const FwdArgs &a, bool vec8, mt_stream_t stream) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e);
    LaunchPlan p;
    e = (op == kRms)     ? fwd_plan_rms(a.N, a.D, vec8, device, &p)
        : (op == kLayer) ? fwd_plan_layer(a.N, a.D, vec8, device, &p)
                         : fwd_plan_add(a.N, a.D, vec8, device, &p);
    if (e != cudaSuccess) return cuda_fail(e);
    FwdArgs copy = a;
    return launch(p, &copy, reinterpret_cast<cudaStream_t>(stream));
}

int num_partial_arrays(int op) { return op == kLayer ? 2 : 1; }

cudaError_t plan_backward(int op, int64_t N, int D, bool vec8, bool has_ds, int device,
                          LaunchPlan *p) {
    switch (op) {
        case kRms: return bwd_plan_rms(N, D, vec8, device, p);
        case kLayer: return bwd_plan_layer(N, D, vec8, device, p);
        default: return bwd_plan_add(N, D, vec8, has_ds, device, p);
    }
}

// One fp32 row of D per persistent CTA, per parameter gradient.
size_t partial_bytes(int op, int rows, int D) {
    const size_t raw = (size_t)num_partial_arrays(op) * (size_t)rows * (size_t)D * sizeof(float);
    return (raw + 255) & ~(size_t)255;
}

// workspace == nullptr with own_ws: allocate stream-ordered scratch here.
mt_status_t run_backward(int op, BwdArgs a, bool vec8, float *dgamma, float *dbeta,
                         void *workspace, size_t ws_bytes, bool own_ws, mt_stream_t stream_in) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_in);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e);
    LaunchPlan p;
    e = plan_backward(op, a.N, a.D, vec8, a.dS != nullptr, device, &p);
    if (e != cudaSuccess) return cuda_fail(e);
    const int prow = p.grid;  // partial rows: one per CTA
    const size_t need = partial_bytes(op, prow, a.D);
    if (own_ws) {
        e = cudaMallocAsync(&workspace, need, stream);
        if (e != cudaSuccess) return cuda_fail(e);
    } else if (ws_bytes < need) {
        return MT_ERR_UNSUPPORTED;
    }
    float *part = static_cast<float *>(workspace);
    a.part_g = part;
    a.part_b = (op == kLayer) ? part + (size_t)prow * (size_t)a.D : nullptr;
    mt_status_t st = launch(p, &a, stream);
    if (st == MT_OK) {
        // Programmatic dependent launch: the reduction is set up while the backward
        // runs and starts reading only after the backward grid has completed. The wide
        // form is used when its 128-column blocks still give one block per SM.
        int sms = 0;
        e = device_sm_count(device, &sms);
        if (e != cudaSuccess) return cuda_fail(e);
        const int arrays = num_partial_arrays(op);
        const bool wide = (a.D % 4 == 0) && ((a.D + 127) / 128) * arrays >= sms;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = wide ? dim3((unsigned)((a.D + 127) / 128), (unsigned)arrays)
                           : dim3((unsigned)((a.D + 31) / 32), (unsigned)arrays);
        cfg.blockDim = dim3(32 * (wide ? kReduceWideWarps : kReduceNarrowWarps));
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const float *cpart = part;
        e = wide ? cudaLaunchKernelEx(&cfg, param_reduce_kernel<4, kReduceWideWarps>, cpart, prow,
                                      a.D, dgamma, dbeta)
                 : cudaLaunchKernelEx(&cfg, param_reduce_kernel<1, kReduceNarrowWarps>, cpart,
                                      prow, a.D, dgamma, dbeta);
        if (e != cudaSuccess) st = cuda_fail(e);
    }
    if (own_ws) {
        e = cudaFreeAsync(workspace, stream);
        if (e != cudaSuccess && st == MT_OK) st = cuda_fail(e);
    }
    return st;
}

}  // namespace

void record_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

cudaError_t device_sm_count(int device, int *sms) {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    auto it = g_sm_count.find(device);
    if (it != g_sm_count.end()) {
        *sms = it->second;
        return cudaSuccess;
    }
    int v = 0;
    cudaError_t e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    g_sm_count[device] = v;
    *sms = v;
    return cudaSuccess;
}

cudaError_t cached_occupancy(const void *kernel, int threads, size_t smem, int device,
                             int *blocks_per_sm) {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    auto key = std::make_tuple(kernel, threads, smem, device);
    auto it = g_occupancy.find(key);
    if (it != g_occupancy.end()) {
        *blocks_per_sm = it->second;
        return cudaSuccess;
    }
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return e;
    if (cur != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
    // Opt in to the dynamic shared memory size whatever it is (the default 48 KB limit
    // counts static shared memory too). The function attribute is only ever raised, so
    // a plan cached earlier with a larger size stays launchable.
    static std::map<std::pair<const void *, int>, size_t> smem_limit;
    size_t &limit = smem_limit[std::make_pair(kernel, device)];
    if (smem > limit) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) limit = smem;
    }
    int v = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, threads, smem);
    if (cur != device) cudaSetDevice(cur);
    if (e != cudaSuccess) return e;
    g_occupancy[key] = v;
    *blocks_per_sm = v;
    return cudaSuccess;
}

}  // namespace mt

using namespace mt;

// ================================================================= RMSNorm ===

extern "C" mt_status_t mt_rmsnorm_forward(const void *X, const void *gamma, void *Y,
                                          float *rstd, int64_t N, int64_t D, float eps,
                                          mt_stream_t stream) {
    if (!X || !gamma || !Y || !rstd) return MT_ERR_INVALID_ARG;
    mt_status_t s = check_shape(N, D);
    if (s != MT_OK) return s;
    if ((s = check_eps(eps)) != MT_OK) return s;
    const size_t act = (size_t)N * (size_t)D * 2, par = (size_t)D * 2, st = (size_t)N * 4;
    if (any_overlap({{Y, act}, {rstd, st}}, {{X, act}, {gamma, par}})) return MT_ERR_INVALID_ARG;
    FwdArgs a{};
    a.X = static_cast<const __half *>(X);
    a.gamma = static_cast<const __half *>(gamma);
    a.Y = static_cast<__half *>(Y);
    a.rstd = rstd;
    a.N = N;
    a.D = (int)D;
    a.eps = eps;
    const bool vec8 = (D % 8 == 0) && aligned16({X, gamma, Y});
    return run_forward(kRms, a, vec8, stream);
}

static mt_status_t rms_backward_impl(const void *X, const void *gamma, const void *dY,
                                     const float *rstd, void *dX, float *dgamma, int64_t N,
                                     int64_t D, void *ws, size_t ws_bytes, bool own_ws,
                                     mt_stream_t stream) {
    if (!X || !gamma || !dY || !rstd || !dX || !dgamma) return MT_ERR_INVALID_ARG;
    mt_status_t s = check_shape(N, D);
    if (s != MT_OK) return s;
    const size_t act = (size_t)N * (size_t)D * 2, par = (size_t)D * 2, st = (size_t)N * 4;
    if (!own_ws && (ws == nullptr || ((uintptr_t)ws & 15u) != 0)) return MT_ERR_INVALID_ARG;
    if (any_overlap({{dX, act}, {dgamma, (size_t)D * 4}, {own_ws ? nullptr : ws, ws_bytes}},
                    {{X, act}, {gamma, par}, {dY, act}, {rstd, st}}))
        return MT_ERR_INVALID_ARG;
    BwdArgs a{};
    a.X = static_cast<const __half *>(X);
    a.gamma = static_cast<const __half *>(gamma);
    a.dY = static_cast<const __half *>(dY);
    a.rstd = rstd;
    a.dX = static_cast<__half *>(dX);
    a.N = N;
    a.D = (int)D;
    const bool vec8 = (D % 8 == 0) && aligned16({X, gamma, dY, dX});
    return run_backward(kRms, a, vec8, dgamma, nullptr, ws, ws_bytes, own_ws, stream);
}

extern "C" mt_status_t mt_rmsnorm_backward(const void *X, const void *gamma, const void *dY,
                                           const float *rstd, void *dX, float *dgamma,
                                           int64_t N, int64_t D, mt_stream_t stream) {
    return rms_backward_impl(X, gamma, dY, rstd, dX, dgamma, N, D, nullptr, 0, true, stream);
}

extern "C" mt_status_t mt_rmsnorm_backward_ws(const void *X, const void *gamma, const void *dY,
                                              const float *rstd, void *dX, float *dgamma,
                                              int64_t N, int64_t D, void *workspace,
                                              size_t workspace_bytes, mt_stream_t stream) {
    return rms_backward_impl(X, gamma, dY, rstd, dX, dgamma, N, D, workspace, workspace_bytes,
                             false, stream);
}

// =============================================================== LayerNorm ===

extern "C" mt_status_t mt_layernorm_forward(const void *X, const void *gamma, const void *beta,
                                            void *Y, float *mean, float *rstd, int64_t N,
                                            int64_t D, float eps, mt_stream_t stream) {
    if (!X || !gamma || !beta || !Y || !mean || !rstd) return MT_ERR_INVALID_ARG;
    mt_status_t s = check_shape(N, D);
    if (s != MT_OK) return s;
    if ((s = check_eps(eps)) != MT_OK) return s;
    const size_t act = (size_t)N * (size_t)D * 2, par = (size_t)D * 2, st = (size_t)N * 4;
    if (any_overlap({{Y, act}, {mean, st}, {rstd, st}}, {{X, act}, {gamma, par}, {beta, par}}))
        return MT_ERR_INVALID_ARG;
    FwdArgs a{};
    a.X = static_cast<const __half *>(X);
    a.gamma = static_cast<const __half *>(gamma);
    a.beta = static_cast<const __half *>(beta);
    a.Y = static_cast<__half *>(Y);
    a.mean = mean;
    a.rstd = rstd;
    a.N = N;
    a.D = (int)D;
    a.eps = eps;
    const bool vec8 = (D % 8 == 0) && aligned16({X, gamma, beta, Y});
    return run_forward(kLayer, a, vec8, stream);
}

static mt_status_t ln_backward_impl(const void *X, const void *gamma, const void *dY,
                                    const float *mean, const float *rstd, void *dX,
                                    float *dgamma, float *dbeta, int64_t N, int64_t D, void *ws,
                                    size_t ws_bytes, bool own_ws, mt_stream_t stream) {
    if (!X || !gamma || !dY || !mean || !rstd || !dX || !dgamma || !dbeta)
        return MT_ERR_INVALID_ARG;
    mt_status_t s = check_shape(N, D);
    if (s != MT_OK) return s;
    const size_t act = (size_t)N * (size_t)D * 2, par = (size_t)D * 2, st = (size_t)N * 4;
    if (!own_ws && (ws == nullptr || ((uintptr_t)ws & 15u) != 0)) return MT_ERR_INVALID_ARG;
    if (any_overlap({{dX, act}, {dgamma, (size_t)D * 4}, {dbeta, (size_t)D * 4},
                     {own_ws ? nullptr : ws, ws_bytes}},
                    {{X, act}, {gamma, par}, {dY, act}, {mean, st}, {rstd, st}}))
        return MT_ERR_INVALID_ARG;
    BwdArgs a{};
    a.X = static_cast<const __half *>(X);
    a.gamma = static_cast<const __half *>(gamma);
    a.dY = static_cast<const __half *>(dY);
    a.mean = mean;
    a.rstd = rstd;
    a.dX = static_cast<__half *>(dX);
    a.N = N;
    a.D = (int)D;
    const bool vec8 = (D % 8 == 0) && aligned16({X, gamma, dY, dX});
    return run_backward(kLayer, a, vec8, dgamma, dbeta, ws, ws_bytes, own_ws, stream);
}

extern "C" mt_status_t mt_layernorm_backward(const void *X, const void *gamma, const void *dY,
                                             const float *mean, const float *rstd, void *dX,
                                             float *dgamma, float *dbeta, int64_t N, int64_t D,
                                             mt_stream_t stream) {
    return ln_backward_impl(X, gamma, dY, mean, rstd, dX, dgamma, dbeta, N, D, nullptr, 0, true,
                            stream);
}

extern "C" mt_status_t mt_layernorm_backward_ws(const void *X, const void *gamma, const void *dY,
                                                const float *mean, const float *rstd, void *dX,
                                                float *dgamma, float *dbeta, int64_t N,
                                                int64_t D, void *workspace,
                                                size_t workspace_bytes, mt_stream_t stream) {
    return ln_backward_impl(X, gamma, dY, mean, rstd, dX, dgamma, dbeta, N, D, workspace,
                            workspace_bytes, false, stream);
}

// ============================================== fused residual add + RMSNorm ===

extern "C" mt_status_t mt_add_rmsnorm_forward(const void *X, const void *R, const void *gamma,
                                              void *S, void *Y, float *rstd, int64_t N,
                                              int64_t D, float eps, mt_stream_t stream) {
    if (!X || !R || !gamma || !S || !Y || !rstd) return MT_ERR_INVALID_ARG;
    mt_status_t s = check_shape(N, D);
    if (s != MT_OK) return s;
    if ((s = check_eps(eps)) != MT_OK) return s;
    const size_t act = (size_t)N * (size_t)D * 2, par = (size_t)D * 2, st = (size_t)N * 4;
    if (any_overlap({{S, act}, {Y, act}, {rstd, st}}, {{X, act}, {R, act}, {gamma, par}}))
        return MT_ERR_INVALID_ARG;
    FwdArgs a{};
    a.X = static_cast<const __half *>(X);
    a.R = static_cast<const __half *>(R);
    a.gamma = static_cast<const __half *>(gamma);
    a.S = static_cast<__half *>(S);
    a.Y = static_cast<__half *>(Y);
    a.rstd = rstd;
    a.N = N;
    a.D = (int)D;
    a.eps = eps;
    const bool vec8 = (D % 8 == 0) && aligned16({X, R, gamma, S, Y});
    return run_forward(kAddRms, a, vec8, stream);
}

static mt_status_t add_backward_impl(const void *S, const void *gamma, const void *dY,
                                     const void *dS, const float *rstd, void *dX, float *dgamma,
                                     int64_t N, int64_t D, void *ws, size_t ws_bytes,
                                     bool own_ws, mt_stream_t stream) {
    if (!S || !gamma || !dY || !rstd || !dX || !dgamma) return MT_ERR_INVALID_ARG;
    mt_status_t s = check_shape(N, D);
    if (s != MT_OK) return s;
    const size_t act = (size_t)N * (size_t)D * 2, par = (size_t)D * 2, st = (size_t)N * 4;
    if (!own_ws && (ws == nullptr || ((uintptr_t)ws & 15u) != 0)) return MT_ERR_INVALID_ARG;
    if (any_overlap({{dX, act}, {dgamma, (size_t)D * 4}, {own_ws ? nullptr : ws, ws_bytes}},
                    {{S, act}, {gamma, par}, {dY, act}, {dS, dS ? act : 0}, {rstd, st}}))
        return MT_ERR_INVALID_ARG;
    BwdArgs a{};
    a.X = static_cast<const __half *>(S);
    a.gamma = static_cast<const __half *>(gamma);
    a.dY = static_cast<const __half *>(dY);
    a.dS = static_cast<const __half *>(dS);
    a.rstd = rstd;
    a.dX = static_cast<__half *>(dX);
    a.N = N;
    a.D = (int)D;
    const bool vec8 = (D % 8 == 0) && aligned16({S, gamma, dY, dS, dX});
    return run_backward(kAddRms, a, vec8, dgamma, nullptr, ws, ws_bytes, own_ws, stream);
}

extern "C" mt_status_t mt_add_rmsnorm_backward(const void *S, const void *gamma, const void *dY,
                                               const void *dS, const float *rstd, void *dX,
                                               float *dgamma, int64_t N, int64_t D,
                                               mt_stream_t stream) {
    return add_backward_impl(S, gamma, dY, dS, rstd, dX, dgamma, N, D, nullptr, 0, true, stream);
}

extern "C" mt_status_t mt_add_rmsnorm_backward_ws(const void *S, const void *gamma,
                                                  const void *dY, const void *dS,
                                                  const float *rstd, void *dX, float *dgamma,
                                                  int64_t N, int64_t D, void *workspace,
                                                  size_t workspace_bytes, mt_stream_t stream) {
    return add_backward_impl(S, gamma, dY, dS, rstd, dX, dgamma, N, D, workspace,
                             workspace_bytes, false, stream);
}

// =============================================================== utilities ===

extern "C" mt_status_t mt_norm_backward_workspace_size(mt_norm_op_t op, int64_t N, int64_t D,
                                                       int device, size_t *bytes) {
    if (bytes == nullptr) return MT_ERR_INVALID_ARG;
    if (op != MT_OP_RMSNORM && op != MT_OP_LAYERNORM && op != MT_OP_ADD_RMSNORM)
        return MT_ERR_INVALID_ARG;
    mt_status_t s = check_shape(N, D);
    if (s != MT_OK) return s;
    if (device < 0) return MT_ERR_INVALID_ARG;
    const int kop = (op == MT_OP_RMSNORM) ? kRms : (op == MT_OP_LAYERNORM) ? kLayer : kAddRms;
    // The largest of the variants a call may take (vectorised or not, with or
    // without dS), so one size fits every call with this op and shape.
    size_t best = 0;
    for (int v = 0; v < 2; ++v) {
        for (int ds = 0; ds < (kop == kAddRms ? 2 : 1); ++ds) {
            if (v == 1 && D % 8 != 0) continue;
            LaunchPlan p;
            cudaError_t e = plan_backward(kop, N, (int)D, v == 1, ds == 1, device, &p);
            if (e != cudaSuccess) return cuda_fail(e);
            const size_t b = partial_bytes(kop, p.grid, (int)D);
            if (b > best) best = b;
        }
    }
    *bytes = best;
    return MT_OK;
}

extern "C" int mt_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" const char *mt_status_string(mt_status_t status) {
    switch (status) {
        case MT_OK: return "MT_OK";
        case MT_ERR_INVALID_ARG: return "MT_ERR_INVALID_ARG: invalid argument";
        case MT_ERR_UNSUPPORTED: return "MT_ERR_UNSUPPORTED: shape or workspace not supported";
        case MT_ERR_CUDA: return "MT_ERR_CUDA: a CUDA call failed (see mt_last_cuda_error)";
    }
    return "unknown mt_status_t";
}

extern "C" int mt_norm_version(void) { return 100; }
