// ops_scalar.cu -- the scalar fallback kernels (any alignment, any width, storage types
// chosen at run time) for every op.
#include "launch.cuh"

namespace mt {

cudaError_t fwd_plan_scalar_op(int op, int64_t N, int D, LaunchPlan *p) {
    switch (op) {
        case kRms: return fwd_plan_scalar<kRms>(N, D, p);
        case kLayer: return fwd_plan_scalar<kLayer>(N, D, p);
        default: return fwd_plan_scalar<kAddRms>(N, D, p);
    }
}

cudaError_t bwd_plan_scalar_op(int op, int64_t N, int D, bool has_ds, int device, LaunchPlan *p) {
    switch (op) {
        case kRms: return bwd_plan_scalar<kRms, false>(N, D, device, p);
        case kLayer: return bwd_plan_scalar<kLayer, false>(N, D, device, p);
        default:
            return has_ds ? bwd_plan_scalar<kAddRms, true>(N, D, device, p)
                          : bwd_plan_scalar<kAddRms, false>(N, D, device, p);
    }
}

}  // namespace mt
