// ops_rms_f32.cu -- RMSNorm vector kernels with fp32 activations (every parameter
// and cotangent type the plans cover), one translation unit so they compile in parallel.
#define MT_PLANS_TU
#include "launch.cuh"

namespace mt {
MT_INSTANTIATE_PLANS(kRms, kF32)
}  // namespace mt
