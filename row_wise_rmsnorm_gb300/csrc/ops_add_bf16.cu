// ops_add_bf16.cu -- fused residual-add + RMSNorm vector kernels with bf16 activations (every parameter
// and cotangent type the plans cover), one translation unit so they compile in parallel.
#define MT_PLANS_TU
#include "launch.cuh"

namespace mt {
MT_INSTANTIATE_PLANS(kAddRms, kBF16)
}  // namespace mt
