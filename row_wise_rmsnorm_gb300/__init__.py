"""GB300 (sm_103a) row-wise normalization: RMSNorm, LayerNorm and fused residual-add +
RMSNorm, forward and backward, behind the C ABI of include/mt_norm.h.

The package holds the CUDA kernels and the C ABI (csrc/), the build step (build.py)
and a thin ctypes binding (_binding.py) with the C entry points' names plus
allocating convenience wrappers. PyTorch is used only for device memory and streams.
"""
from ._binding import (  # noqa: F401
    EXPORTED,
    MT_ERR_CUDA,
    MT_ERR_INVALID_ARG,
    MT_ERR_UNSUPPORTED,
    MT_MAX_COLS,
    MT_NOALLOC_SCRATCH_BYTES,
    MT_OK,
    MT_OP_ADD_RMSNORM,
    MT_OP_LAYERNORM,
    MT_OP_RMSNORM,
    MtNormError,
    add_rmsnorm_backward,
    add_rmsnorm_forward,
    layernorm_backward,
    layernorm_forward,
    library_path,
    load,
    mt_add_rmsnorm_backward,
    mt_add_rmsnorm_backward_ws,
    mt_add_rmsnorm_forward,
    mt_last_cuda_error,
    mt_layernorm_backward,
    mt_layernorm_backward_ws,
    mt_layernorm_forward,
    mt_norm_backward_workspace_size,
    mt_norm_version,
    mt_rmsnorm_backward,
    mt_rmsnorm_backward_noalloc,
    mt_rmsnorm_backward_ws,
    mt_rmsnorm_forward,
    mt_status_string,
    rmsnorm_backward,
    rmsnorm_forward,
)
