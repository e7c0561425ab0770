"""B300-native CSA + HCA hybrid compressed attention.

The compute path is the CUDA library ``libcsa.so`` (sm_103a kernels behind a
C ABI declared in ``include/csa.h``); this package is a thin ctypes binding
over it.  There is no CPU fallback: calling any op without the built library
or without a CUDA device raises.
"""
__version__ = "0.1.0"
