// noalloc.cu -- an RMSNorm backward that allocates nothing.
//
// The ordinary backward needs a scratch buffer for its per-CTA dgamma partials:
// mt_rmsnorm_backward allocates it stream-ordered, mt_rmsnorm_backward_ws takes it
// from the caller. Some callers can do neither. A host framework that owns all device
// memory through its own pool may forbid any allocation behind its back (it would
// break the pool's accounting and fragment the heap); a latency-critical loop may not
// tolerate an allocator call at all; and code handed only raw pointers may have no
// allocator it is allowed to use. For them, mt_rmsnorm_backward_noalloc takes the
// scratch from a fixed array compiled into this library.
//
// The array is a file-scope __device__ object of kNoAllocScratchBytes. Every GPU that
// loads the library reserves it until the process exits. Host code may not use the
// array's name as a device address (on the host it names a stand-in object), so the
// first call on each device looks up the array's device address with
// cudaGetSymbolAddress, with that device current, and caches it; make that first call
// before any stream capture begins. All calls share the one array and leave the last
// call's partials in it; nothing in it has to start at zero, because the backward
// writes every partial it later reads. Calls that overlap on the GPU (on different
// streams, or from several threads) race on the array and must not be issued.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "launch.cuh"
#include "mt_norm.h"

namespace {

// Largest partial buffer any RMSNorm shape up to MT_MAX_COLS columns needs on a GB300
// (152 SMs) with the current kernels is under 10 MB; 16 MiB leaves headroom.
constexpr size_t kNoAllocScratchBytes = MT_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

extern "C" mt_status_t mt_rmsnorm_backward_noalloc(const void *X, const void *gamma,
                                                   const void *dY, const float *rstd, void *dX,
                                                   float *dgamma, int64_t N, int64_t D,
                                                   mt_stream_t stream) {
    // Argument errors are reported before any CUDA call, as for every other entry point.
    if (N < 0 || D < 1) return MT_ERR_INVALID_ARG;
    if (D > MT_MAX_COLS || N > (int64_t)INT32_MAX) return MT_ERR_UNSUPPORTED;
    if (N == 0)  // an empty batch: dgamma = 0, no scratch
        return mt_rmsnorm_backward_ws(X, gamma, dY, rstd, dX, dgamma, N, D, nullptr, 0, stream);
    if (!X || !gamma || !dY || !rstd || !dX || !dgamma) return MT_ERR_INVALID_ARG;

    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) {
        mt::record_cuda_error(e);
        return MT_ERR_CUDA;
    }
    if (device < 0 || device >= kMaxDevices) return MT_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_scratch_addr[device] == nullptr) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) {
                mt::record_cuda_error(e);
                return MT_ERR_CUDA;
            }
            g_scratch_addr[device] = p;
        }
        scratch = g_scratch_addr[device];
    }
    // The _ws entry point checks that the partials fit: a shape whose partials exceed
    // kNoAllocScratchBytes returns MT_ERR_UNSUPPORTED without launching anything.
    return mt_rmsnorm_backward_ws(X, gamma, dY, rstd, dX, dgamma, N, D, scratch,
                                  kNoAllocScratchBytes, stream);
}
