"""GB300-native batched decode sampler.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/vt_sampler.h``); ``sampler`` is a thin
ctypes binding over it.  ``workloads`` makes seeded synthetic inputs.

The binding is imported lazily, so that ``workloads`` can be used without the
built library; touching ``Sampler`` (or anything from ``sampler``) loads the
library and raises if it has not been built.
"""

__all__ = ["Sampler", "VtError", "DTYPE_F32", "DTYPE_BF16", "library_path", "build"]


def __getattr__(name):
    if name in ("Sampler", "VtError", "DTYPE_F32", "DTYPE_BF16", "library_path"):
        from . import sampler
        return getattr(sampler, name)
    if name == "build":
        from ._build import build
        return build
    raise AttributeError(name)
