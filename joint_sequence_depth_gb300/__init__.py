"""MoDA (Mixture-of-Depths Attention) for one GB300: a C-ABI CUDA library and its binding.

The compute path lives in ``csrc/`` (hand-written sm_103a kernels behind the
C ABI of ``include/moda.h``).  ``binding`` marshals torch CUDA tensors into
those calls; it loads ``libmoda.so`` on first use and raises if it is missing.
"""

__all__ = ["moda_fwd", "moda_bwd", "moda_bwd_workspace_bytes", "library_path"]


def __getattr__(name):
    if name in __all__:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
