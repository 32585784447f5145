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

// N = 0 is a valid, empty batch (see forward_impl / backward_impl).
mt_status_t check_shape(int64_t N, int64_t D) {
    if (N < 0 || D < 1) return MT_ERR_INVALID_ARG;
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
std::map<std::tuple<const void *, int, size_t, int, int>, int> g_cluster_occupancy;

}  // namespace

// Every launch carries the programmatic-stream-serialization attribute (see pdl_enter()
// in kernels.cuh).
cudaError_t launch_pdl(const LaunchPlan &p, void *arg, cudaStream_t stream) {
    if (p.kernel == nullptr || p.grid < 1) return cudaErrorInvalidConfiguration;
    const cudaError_t h = launch_hook();
    if (h != cudaSuccess) return h;
    void *args[] = {arg};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.cluster > 1) {
        // (a non-portable cluster size was opted into when the plan was made:
        // cached_cluster_occupancy)
        if (p.grid % p.cluster != 0) return cudaErrorInvalidConfiguration;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)p.cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelExC(&cfg, p.kernel, args);
}

namespace {

mt_status_t launch(const LaunchPlan &p, void *arg, cudaStream_t stream) {
    const cudaError_t e = launch_pdl(p, arg, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return MT_OK;
}


// The vector plan for (op, activation type), or kNoVectorPlan.
cudaError_t plan_forward_vec(int op, int xdt, int64_t N, int D, int wdt, LaunchPlan *p) {
#define MT_CASE(OP, XT) \
    if (op == OP && xdt == XT) return fwd_plan_for<OP, XT>(N, D, wdt, p);
    MT_ALL_PLANS(MT_CASE)
#undef MT_CASE
    return kNoVectorPlan;
}

cudaError_t plan_backward_vec(int op, int xdt, int64_t N, int D, int wdt, int gdt, bool has_ds,
                              int device, LaunchPlan *p) {
#define MT_CASE(OP, XT) \
    if (op == OP && xdt == XT) return bwd_plan_for<OP, XT>(N, D, wdt, gdt, has_ds, device, p);
    MT_ALL_PLANS(MT_CASE)
#undef MT_CASE
    return kNoVectorPlan;
}

// The vector kernel when the row layout allows it and the dtype combination has one,
// else the scalar kernel.
cudaError_t plan_forward(int op, int64_t N, int D, bool vec8, int xdt, int wdt, LaunchPlan *p) {
    if (vec8) {
        const cudaError_t e = plan_forward_vec(op, xdt, N, D, wdt, p);
        if (e != kNoVectorPlan) return e;
    }
    *p = LaunchPlan{};
    return fwd_plan_scalar_op(op, N, D, p);
}

cudaError_t plan_backward(int op, int64_t N, int D, bool vec8, int xdt, int wdt, int gdt,
                          bool has_ds, int device, LaunchPlan *p) {
    if (vec8) {
        const cudaError_t e = plan_backward_vec(op, xdt, N, D, wdt, gdt, has_ds, device, p);
        if (e != kNoVectorPlan) return e;
    }
    *p = LaunchPlan{};
    return bwd_plan_scalar_op(op, N, D, has_ds, device, p);
}

mt_status_t run_forward(int op, const FwdArgs &a, bool vec8, mt_stream_t stream) {
    LaunchPlan p;
    const cudaError_t e = plan_forward(op, a.N, a.D, vec8, a.xdt, a.wdt, &p);
    if (e != cudaSuccess) return cuda_fail(e);
    FwdArgs copy = a;
    copy.slice = p.slice;
    copy.ahead = 0;
    if (p.warm) {  // the L2 warm-up distance: the rows of the launch's resident CTAs
        int device = 0, bps = 0, sms = 0;
        cudaError_t q = cudaGetDevice(&device);
        if (q == cudaSuccess) q = cached_occupancy(p.kernel, p.threads, p.smem, device, &bps);
        if (q == cudaSuccess) q = device_sm_count(device, &sms);
        if (q != cudaSuccess) return cuda_fail(q);
        copy.ahead = bps * sms * std::max(p.rows_per_cta, 1);
    }
    return launch(p, &copy, reinterpret_cast<cudaStream_t>(stream));
}

int num_partial_arrays(int op) { return op == kLayer ? 2 : 1; }

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
    e = plan_backward(op, a.N, a.D, vec8, a.xdt, a.wdt, a.gdt, a.dS != nullptr, device, &p);
    if (e != cudaSuccess) return cuda_fail(e);
    const int prow = p.owners();  // partial rows: one per CTA, or per cluster of a split row
    a.slice = p.slice;
    const size_t need = partial_bytes(op, prow, a.D);
    if (own_ws) {
        e = cudaMallocAsync(&workspace, need, stream);
        if (e != cudaSuccess) return cuda_fail(e);
    } else if (ws_bytes < need) {
        return MT_ERR_UNSUPPORTED;
    }
    if (p.waits && (e = device_status_word(device, &a.status)) != cudaSuccess) {
        const mt_status_t fail = cuda_fail(e);
        if (own_ws) cudaFreeAsync(workspace, stream);
        return fail;
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
        e = device_sm_count(device, &sms);  // cached by the plan: cannot fail here
        if (e != cudaSuccess) sms = 1;
        const int arrays = num_partial_arrays(op);
        const bool wide = (a.D % 4 == 0) && ((a.D + 127) / 128) * arrays >= sms;
        // wide blocks of 4 warps when each warp's rows still fit one batch of loads (split rows
        // leave 152 / CL partial rows: 19 for 8-CTA clusters, 38 for 4; measured on GB300:
        // LayerNorm 1024 x 131072 backward 212.5 -> 206.0 us; 8 warps for 76 rows did not pay)
        const int ww = (prow <= 4 * kReduceBatch) ? 4 : kReduceWideWarps;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = wide ? dim3((unsigned)((a.D + 127) / 128), (unsigned)arrays)
                           : dim3((unsigned)((a.D + 31) / 32), (unsigned)arrays);
        cfg.blockDim = dim3(32 * (wide ? ww : kReduceNarrowWarps));
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const float *cpart = part;
        e = launch_hook();
        if (e == cudaSuccess)
            e = !wide ? cudaLaunchKernelEx(&cfg, param_reduce_kernel<1, kReduceNarrowWarps>, cpart,
                                           prow, a.D, dgamma, dbeta)
                : ww == 4 ? cudaLaunchKernelEx(&cfg, param_reduce_kernel<4, 4>, cpart, prow, a.D,
                                               dgamma, dbeta)
                          : cudaLaunchKernelEx(&cfg, param_reduce_kernel<4, kReduceWideWarps>, cpart,
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

}  // namespace mt

// Error bits of the kernels' bounded waits (kErrClusterWait), one word per device that
// loads the library; kernels receive its address (device_status_word) and OR bits in.
static __device__ unsigned g_mt_device_status;

namespace mt {

cudaError_t device_status_word(int device, unsigned **word) {
    static std::mutex mu;
    static std::map<int, unsigned *> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(device);
    if (it != cache.end()) {
        *word = it->second;
        return cudaSuccess;
    }
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return e;
    if (cur != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_mt_device_status);
    if (cur != device) cudaSetDevice(cur);
    if (e != cudaSuccess) return e;
    cache[device] = static_cast<unsigned *>(p);
    *word = static_cast<unsigned *>(p);
    return cudaSuccess;
}

#ifdef MT_TEST_HOOKS
// Test build only (-DMT_TEST_HOOKS, libmt_norm_hooks.so): host-side failure injection.
// mt_test_fail_launch(skip, err) arms a one-shot failure: the launch that comes after
// `skip` further launches returns `err` without launching anything, as a failing
// cudaLaunchKernelEx would. Nothing on the GPU is made to fail.
namespace {
std::mutex g_hook_mu;
int g_hook_skip = -1;  // < 0: disarmed
cudaError_t g_hook_err = cudaSuccess;
}  // namespace

cudaError_t launch_hook() {
    std::lock_guard<std::mutex> lock(g_hook_mu);
    if (g_hook_skip < 0) return cudaSuccess;
    if (g_hook_skip-- > 0) return cudaSuccess;
    return g_hook_err;
}
#else
cudaError_t launch_hook() { return cudaSuccess; }
#endif

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

// Called after cached_occupancy for the same kernel and shape, which has raised the
// kernel's dynamic shared memory limit.
cudaError_t cached_cluster_occupancy(const void *kernel, int threads, size_t smem, int cluster,
                                     int device, int *clusters) {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    auto key = std::make_tuple(kernel, threads, smem, cluster, device);
    auto it = g_cluster_occupancy.find(key);
    if (it != g_cluster_occupancy.end()) {
        *clusters = it->second;
        return cudaSuccess;
    }
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return e;
    if (cur != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int v = 0;
    if (cluster > kMaxCluster) {
        // A non-portable cluster size: the kernel opts in here, once per kernel and
        // device (the attribute persists, so launches need not set it again). A device
        // or driver that refuses the opt-in or the occupancy query for this size cannot
        // run the clusters: that is recorded as 0 resident clusters (the planner then
        // takes the scalar kernel) and the error is cleared, not returned.
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&v, kernel, &cfg);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            v = 0;
            e = cudaSuccess;
        }
    } else {
        e = cudaOccupancyMaxActiveClusters(&v, kernel, &cfg);
    }
    if (cur != device) cudaSetDevice(cur);
    if (e != cudaSuccess) return e;
    g_cluster_occupancy[key] = v;
    *clusters = v;
    return cudaSuccess;
}

}  // namespace mt

using namespace mt;

// ====================================================== generic forward/backward ===

namespace {

bool valid_dtype(int dt) { return dt == kF16 || dt == kBF16 || dt == kF32; }
size_t dtype_bytes(int dt) { return dt == kF32 ? 4 : 2; }

// Forward of `op` with activations of type xdt and gamma/beta of type wdt. Pointers the
// op does not use are ignored.
mt_status_t forward_impl(int op, int xdt, int wdt, const void *X, const void *R,
                         const void *gamma, const void *beta, void *S, void *Y, float *mean,
                         float *rstd, int64_t N, int64_t D, float eps, mt_stream_t stream) {
    const bool ln = op == kLayer, add = op == kAddRms;
    if (!ln) { beta = nullptr; mean = nullptr; }
    if (!add) { R = nullptr; S = nullptr; }
    if (!valid_dtype(xdt) || !valid_dtype(wdt)) return MT_ERR_INVALID_ARG;
    mt_status_t s = check_shape(N, D);
    if (s != MT_OK) return s;
    if ((s = check_eps(eps)) != MT_OK) return s;
    if (N == 0) return MT_OK;  // an empty batch: nothing is read or written
    if (!X || !gamma || !Y || !rstd || (ln && (!beta || !mean)) || (add && (!R || !S)))
        return MT_ERR_INVALID_ARG;
    const size_t act = (size_t)N * (size_t)D * dtype_bytes(xdt);
    const size_t par = (size_t)D * dtype_bytes(wdt), st = (size_t)N * 4;
    if (any_overlap({{S, act}, {Y, act}, {mean, st}, {rstd, st}},
                    {{X, act}, {R, act}, {gamma, par}, {beta, par}}))
        return MT_ERR_INVALID_ARG;
    FwdArgs a{};
    a.X = X;
    a.R = R;
    a.gamma = gamma;
    a.beta = beta;
    a.S = S;
    a.Y = Y;
    a.mean = mean;
    a.rstd = rstd;
    a.N = N;
    a.D = (int)D;
    a.eps = eps;
    a.xdt = xdt;
    a.wdt = wdt;
    const bool vec8 = (D % 8 == 0) && aligned16({X, R, gamma, beta, S, Y});
    return run_forward(op, a, vec8, stream);
}

// Backward of `op`: X (or the saved S) and dX of type xdt, gamma of type wdt, dY/dS of
// type gdt. dS may be NULL (fused op only; ignored otherwise). workspace NULL with
// own_ws: stream-ordered scratch is allocated here.
mt_status_t backward_impl(int op, int xdt, int wdt, int gdt, const void *X, const void *gamma,
                          const void *dY, const void *dS, const float *mean, const float *rstd,
                          void *dX, float *dgamma, float *dbeta, int64_t N, int64_t D,
                          void *ws, size_t ws_bytes, bool own_ws, mt_stream_t stream) {
    const bool ln = op == kLayer, add = op == kAddRms;
    if (!ln) { mean = nullptr; dbeta = nullptr; }
    if (!add) dS = nullptr;
    if (!valid_dtype(xdt) || !valid_dtype(wdt) || !valid_dtype(gdt)) return MT_ERR_INVALID_ARG;
    mt_status_t s = check_shape(N, D);
    if (s != MT_OK) return s;
    if (N == 0) {
        // an empty batch: the parameter gradients are empty sums, 0; nothing else is
        // read or written and no workspace is needed
        if (!dgamma || (ln && !dbeta) || (ln && dgamma == dbeta)) return MT_ERR_INVALID_ARG;
        cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
        cudaError_t e = cudaMemsetAsync(dgamma, 0, (size_t)D * sizeof(float), st);
        if (e == cudaSuccess && ln) e = cudaMemsetAsync(dbeta, 0, (size_t)D * sizeof(float), st);
        return e == cudaSuccess ? MT_OK : cuda_fail(e);
    }
    if (!X || !gamma || !dY || !rstd || !dX || !dgamma || (ln && (!mean || !dbeta)))
        return MT_ERR_INVALID_ARG;
    const size_t act = (size_t)N * (size_t)D * dtype_bytes(xdt);
    const size_t cot = (size_t)N * (size_t)D * dtype_bytes(gdt);
    const size_t par = (size_t)D * dtype_bytes(wdt), st = (size_t)N * 4, grad = (size_t)D * 4;
    if (!own_ws && (ws == nullptr || ((uintptr_t)ws & 15u) != 0)) return MT_ERR_INVALID_ARG;
    if (any_overlap({{dX, act}, {dgamma, grad}, {dbeta, grad}, {own_ws ? nullptr : ws, ws_bytes}},
                    {{X, act}, {gamma, par}, {dY, cot}, {dS, cot}, {mean, st}, {rstd, st}}))
        return MT_ERR_INVALID_ARG;
    BwdArgs a{};
    a.X = X;
    a.gamma = gamma;
    a.dY = dY;
    a.dS = dS;
    a.mean = mean;
    a.rstd = rstd;
    a.dX = dX;
    a.N = N;
    a.D = (int)D;
    a.xdt = xdt;
    a.wdt = wdt;
    a.gdt = gdt;
    const bool vec8 = (D % 8 == 0) && aligned16({X, gamma, dY, dS, dX});
    return run_backward(op, a, vec8, dgamma, dbeta, ws, ws_bytes, own_ws, stream);
}

}  // namespace

// ================================================================= RMSNorm ===

extern "C" mt_status_t mt_rmsnorm_forward(const void *X, const void *gamma, void *Y,
                                          float *rstd, int64_t N, int64_t D, float eps,
                                          mt_stream_t stream) {
    return forward_impl(kRms, kF16, kF16, X, nullptr, gamma, nullptr, nullptr, Y, nullptr, rstd,
                        N, D, eps, stream);
}

extern "C" mt_status_t mt_rmsnorm_backward(const void *X, const void *gamma, const void *dY,
                                           const float *rstd, void *dX, float *dgamma,
                                           int64_t N, int64_t D, mt_stream_t stream) {
    return backward_impl(kRms, kF16, kF16, kF16, X, gamma, dY, nullptr, nullptr, rstd, dX, dgamma,
                         nullptr, N, D, nullptr, 0, true, stream);
}

extern "C" mt_status_t mt_rmsnorm_backward_ws(const void *X, const void *gamma, const void *dY,
                                              const float *rstd, void *dX, float *dgamma,
                                              int64_t N, int64_t D, void *workspace,
                                              size_t workspace_bytes, mt_stream_t stream) {
    return backward_impl(kRms, kF16, kF16, kF16, X, gamma, dY, nullptr, nullptr, rstd, dX, dgamma,
                         nullptr, N, D, workspace, workspace_bytes, false, stream);
}

// =============================================================== LayerNorm ===

extern "C" mt_status_t mt_layernorm_forward(const void *X, const void *gamma, const void *beta,
                                            void *Y, float *mean, float *rstd, int64_t N,
                                            int64_t D, float eps, mt_stream_t stream) {
    return forward_impl(kLayer, kF16, kF16, X, nullptr, gamma, beta, nullptr, Y, mean, rstd, N,
                        D, eps, stream);
}

extern "C" mt_status_t mt_layernorm_backward(const void *X, const void *gamma, const void *dY,
                                             const float *mean, const float *rstd, void *dX,
                                             float *dgamma, float *dbeta, int64_t N, int64_t D,
                                             mt_stream_t stream) {
    return backward_impl(kLayer, kF16, kF16, kF16, X, gamma, dY, nullptr, mean, rstd, dX, dgamma,
                         dbeta, N, D, nullptr, 0, true, stream);
}

extern "C" mt_status_t mt_layernorm_backward_ws(const void *X, const void *gamma, const void *dY,
                                                const float *mean, const float *rstd, void *dX,
                                                float *dgamma, float *dbeta, int64_t N,
                                                int64_t D, void *workspace,
                                                size_t workspace_bytes, mt_stream_t stream) {
    return backward_impl(kLayer, kF16, kF16, kF16, X, gamma, dY, nullptr, mean, rstd, dX, dgamma,
                         dbeta, N, D, workspace, workspace_bytes, false, stream);
}

// ============================================== fused residual add + RMSNorm ===

extern "C" mt_status_t mt_add_rmsnorm_forward(const void *X, const void *R, const void *gamma,
                                              void *S, void *Y, float *rstd, int64_t N,
                                              int64_t D, float eps, mt_stream_t stream) {
    return forward_impl(kAddRms, kF16, kF16, X, R, gamma, nullptr, S, Y, nullptr, rstd, N, D, eps,
                        stream);
}

extern "C" mt_status_t mt_add_rmsnorm_backward(const void *S, const void *gamma, const void *dY,
                                               const void *dS, const float *rstd, void *dX,
                                               float *dgamma, int64_t N, int64_t D,
                                               mt_stream_t stream) {
    return backward_impl(kAddRms, kF16, kF16, kF16, S, gamma, dY, dS, nullptr, rstd, dX, dgamma,
                         nullptr, N, D, nullptr, 0, true, stream);
}

extern "C" mt_status_t mt_add_rmsnorm_backward_ws(const void *S, const void *gamma,
                                                  const void *dY, const void *dS,
                                                  const float *rstd, void *dX, float *dgamma,
                                                  int64_t N, int64_t D, void *workspace,
                                                  size_t workspace_bytes, mt_stream_t stream) {
    return backward_impl(kAddRms, kF16, kF16, kF16, S, gamma, dY, dS, nullptr, rstd, dX, dgamma,
                         nullptr, N, D, workspace, workspace_bytes, false, stream);
}

// ========================================================= explicit dtypes ===

static int op_code(mt_norm_op_t op) {
    return (op == MT_OP_RMSNORM) ? kRms : (op == MT_OP_LAYERNORM) ? kLayer
                                        : (op == MT_OP_ADD_RMSNORM) ? kAddRms : -1;
}

extern "C" mt_status_t mt_norm_forward_ex(mt_norm_op_t op, mt_dtype_t x_dtype, mt_dtype_t w_dtype,
                                          const void *X, const void *R, const void *gamma,
                                          const void *beta, void *S, void *Y, float *mean,
                                          float *rstd, int64_t N, int64_t D, float eps,
                                          mt_stream_t stream) {
    const int kop = op_code(op);
    if (kop < 0) return MT_ERR_INVALID_ARG;
    return forward_impl(kop, (int)x_dtype, (int)w_dtype, X, R, gamma, beta, S, Y, mean, rstd, N,
                        D, eps, stream);
}

extern "C" mt_status_t mt_norm_backward_ex(mt_norm_op_t op, mt_dtype_t x_dtype,
                                           mt_dtype_t w_dtype, mt_dtype_t g_dtype, const void *X,
                                           const void *gamma, const void *dY, const void *dS,
                                           const float *mean, const float *rstd, void *dX,
                                           float *dgamma, float *dbeta, int64_t N, int64_t D,
                                           void *workspace, size_t workspace_bytes,
                                           mt_stream_t stream) {
    const int kop = op_code(op);
    if (kop < 0) return MT_ERR_INVALID_ARG;
    return backward_impl(kop, (int)x_dtype, (int)w_dtype, (int)g_dtype, X, gamma, dY, dS, mean,
                         rstd, dX, dgamma, dbeta, N, D, workspace, workspace_bytes,
                         workspace == nullptr, stream);
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
    if (N == 0) {  // an empty batch needs no workspace
        *bytes = 0;
        return MT_OK;
    }
    const int kop = (op == MT_OP_RMSNORM) ? kRms : (op == MT_OP_LAYERNORM) ? kLayer : kAddRms;
    // The largest of the variants a call may take (vectorised or not, with or without
    // dS, any storage types), so one size fits every call with this op and shape.
    size_t best = 0;
    for (int v = 0; v < 2; ++v) {
        if (v == 1 && D % 8 != 0) continue;
        for (int ds = 0; ds < (kop == kAddRms ? 2 : 1); ++ds) {
            for (int xdt = 0; xdt < 3; ++xdt) {
                for (int wdt = 0; wdt < 3; ++wdt) {
                    for (int gdt = 0; gdt < 3; ++gdt) {
                        LaunchPlan p;
                        cudaError_t e = plan_backward(kop, N, (int)D, v == 1, xdt, wdt, gdt,
                                                      ds == 1, device, &p);
                        if (e != cudaSuccess) return cuda_fail(e);
                        const size_t b = partial_bytes(kop, p.owners(), (int)D);
                        if (b > best) best = b;
                    }
                }
            }
        }
    }
    *bytes = best;
    return MT_OK;
}

extern "C" int mt_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" mt_status_t mt_device_wait_errors(int device, unsigned *flags, int clear) {
    if (flags == nullptr || device < 0) return MT_ERR_INVALID_ARG;
    unsigned *word = nullptr;
    cudaError_t e = device_status_word(device, &word);
    if (e != cudaSuccess) return cuda_fail(e);
    int cur = 0;
    if ((e = cudaGetDevice(&cur)) != cudaSuccess) return cuda_fail(e);
    if (cur != device && (e = cudaSetDevice(device)) != cudaSuccess) return cuda_fail(e);
    e = cudaMemcpy(flags, word, sizeof(unsigned), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && clear) e = cudaMemset(word, 0, sizeof(unsigned));
    if (cur != device) cudaSetDevice(cur);
    return e == cudaSuccess ? MT_OK : cuda_fail(e);
}

#ifdef MT_TEST_HOOKS
extern "C" void mt_test_fail_launch(int skip, int error) {
    std::lock_guard<std::mutex> lock(g_hook_mu);
    g_hook_skip = skip;
    g_hook_err = (cudaError_t)error;
}

// 1 while an injected failure is still armed.
extern "C" int mt_test_failure_armed(void) {
    std::lock_guard<std::mutex> lock(g_hook_mu);
    return g_hook_skip >= 0;
}

// Bytes in use in the memory pool stream-ordered allocations on `device` draw from.
extern "C" int mt_test_pool_used_bytes(int device, unsigned long long *bytes) {
    cudaMemPool_t pool;
    cudaError_t e = cudaDeviceGetMemPool(&pool, device);
    if (e == cudaSuccess) {
        unsigned long long v = 0;  // the attribute is a 64-bit unsigned integer
        e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemCurrent, &v);
        *bytes = (unsigned long long)v;
    }
    return (int)e;
}
#endif

extern "C" const char *mt_status_string(mt_status_t status) {
    switch (status) {
        case MT_OK: return "MT_OK";
        case MT_ERR_INVALID_ARG: return "MT_ERR_INVALID_ARG: invalid argument";
        case MT_ERR_UNSUPPORTED: return "MT_ERR_UNSUPPORTED: shape or workspace not supported";
        case MT_ERR_CUDA: return "MT_ERR_CUDA: a CUDA call failed (see mt_last_cuda_error)";
    }
    return "unknown mt_status_t";
}

extern "C" int mt_norm_version(void) { return 200; }
