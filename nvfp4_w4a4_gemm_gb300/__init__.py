"""GB300-native NVFP4 / MXFP4 W4A4 linear layer with residual activation
compensation: a C-ABI CUDA library (``libnvfp4w4a4.so``, sm_103a) and a thin
ctypes binding (:mod:`nvfp4_w4a4_gemm_gb300.binding`).  Importing the package
does not load the library; the first call of a binding does, and raises if
the library has not been built (``python -m nvfp4_w4a4_gemm_gb300.build``)."""

import importlib

from .workloads import SPECS, WORKLOADS  # noqa: F401

_SUBMODULES = ("binding", "build", "workloads")


def __getattr__(name):
    if name in _SUBMODULES:
        return importlib.import_module(f"{__name__}.{name}")
    if name.startswith("_"):
        raise AttributeError(name)
    # binding functions (nvfp4_quantize, w4a4_gemm_comp, ...) at package level
    return getattr(importlib.import_module(f"{__name__}.binding"), name)
