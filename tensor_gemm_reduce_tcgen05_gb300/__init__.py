"""Fused GEMM + reduce-scatter for GB300 (sm_103a).

The compute path is the C-ABI library ``libgemm_rs.so`` built from
``csrc/``.  ``binding`` loads it with ctypes and marshals arguments only.
Import ``binding`` (or call :func:`load`) to use it.  Importing this package
does not load any CUDA code.
"""

__all__ = ["load"]


def load():
    """Load the CUDA library and return the binding module.  Raises if the
    library has not been built."""
    from . import binding
    binding.lib()
    return binding
