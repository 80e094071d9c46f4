"""GB300-native NVFP4 / MXFP4 W4A4 linear layer with residual activation
compensation: a C-ABI CUDA library (``libnvfp4w4a4.so``, sm_103a) and a thin
ctypes binding.  Importing the package does not load the library; the first
call of a binding does, and raises if the library has not been built."""

from .workloads import SPECS, WORKLOADS  # noqa: F401


def __getattr__(name):
    # lazy: the binding loads the CUDA library on first use
    from . import binding
    return getattr(binding, name)
