// ops_rms.cu -- RMSNorm kernel instantiations (forward and backward).
#include "launch.cuh"

namespace mt {
cudaError_t fwd_plan_rms(int64_t N, int D, bool vec8, int device, LaunchPlan *p) {
    return fwd_plan<kRms>(N, D, vec8, device, p);
}
cudaError_t bwd_plan_rms(int64_t N, int D, bool vec8, int device, LaunchPlan *p) {
    return bwd_plan<kRms, false>(N, D, vec8, device, p);
}
}  // namespace mt
