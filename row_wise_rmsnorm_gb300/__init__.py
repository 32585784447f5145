"""GB300 (sm_103a) row-wise normalization: RMSNorm, LayerNorm and fused residual-add +
RMSNorm, forward and backward, behind the C ABI of include/mt_norm.h.

The package holds the CUDA kernels and the C ABI (csrc/), the build step (build.py)
and a thin ctypes binding (_binding.py) with the C entry points' names plus
allocating convenience wrappers. PyTorch is used only for device memory and streams.

The package's names are the binding's public ones: the C entry points (mt_*), the
header's constants (MT_*), the allocating wrappers (rmsnorm_forward, ...), EXPORTED,
MtNormError, load and library_path.
"""
import types as _types

from . import _binding


def __getattr__(name):
    if not name.startswith("_"):
        value = getattr(_binding, name, _binding)
        if value is not _binding and not isinstance(value, _types.ModuleType):
            return value
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")


def __dir__():
    return sorted(set(globals()) | {n for n in dir(_binding) if not n.startswith("_")
                                    and not isinstance(getattr(_binding, n), _types.ModuleType)})
