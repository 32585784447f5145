"""GB300 (sm_103a) row-wise normalization: RMSNorm, LayerNorm and fused residual-add +
RMSNorm, forward and backward, behind the C ABI of include/mt_norm.h.

The package holds the CUDA kernels and the C ABI (csrc/), the build step (build.py)
and a thin ctypes binding (_binding.py) with the C entry points' names plus
allocating convenience wrappers. PyTorch is used only for device memory and streams.

The package's names are the binding's public ones, bound here at import: the C entry
points (mt_*), the header's constants (MT_*), the allocating wrappers (rmsnorm_forward,
...), EXPORTED, MtNormError, load and library_path.
"""
import types as _types

from . import _binding

globals().update({n: v for n, v in vars(_binding).items()
                  if not n.startswith("_") and not isinstance(v, _types.ModuleType)
                  and n != "annotations"})
