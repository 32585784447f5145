// ops_add.cu -- fused residual-add + RMSNorm kernel instantiations.
#include "launch.cuh"

namespace mt {
cudaError_t fwd_plan_add(int64_t N, int D, bool vec8, int device, LaunchPlan *p) {
    return fwd_plan<kAddRms>(N, D, vec8, device, p);
}
cudaError_t bwd_plan_add(int64_t N, int D, bool vec8, bool has_ds, int device, LaunchPlan *p) {
    return has_ds ? bwd_plan<kAddRms, true>(N, D, vec8, device, p)
                  : bwd_plan<kAddRms, false>(N, D, vec8, device, p);
}
}  // namespace mt
