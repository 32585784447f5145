// ops_layer_f16.cu -- LayerNorm vector kernels with fp16 activations (every parameter
// and cotangent type the plans cover), one translation unit so they compile in parallel.
#define MT_PLANS_TU
#include "launch.cuh"

namespace mt {
MT_INSTANTIATE_PLANS(kLayer, kF16)
}  // namespace mt
