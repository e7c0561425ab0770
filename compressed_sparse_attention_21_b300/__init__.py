"""B300-native CSA + HCA hybrid compressed attention.

The compute path is the CUDA library ``libcsa.so`` (sm_103a kernels behind the
C ABI declared in ``include/csa.h``); this package is a thin ctypes binding
over it.  There is no CPU fallback: any op raises if the library is missing
or the tensors are not on a CUDA device.
"""
from ._lib import (CSA_SKIP_COMPRESS, CsaError, Hybrid, Layout, attend_workspace_size,
                   check_device_error, csa_compress, hca_compress, hca_dense_attend,
                   index_workspace_size, lightning_index_topk, load, sparse_mqa_attend,
                   timing_enable, timing_read, timing_reset)

__version__ = "0.1.0"

__all__ = ["CSA_SKIP_COMPRESS", "CsaError", "Hybrid", "Layout", "attend_workspace_size",
           "check_device_error", "csa_compress", "hca_compress", "hca_dense_attend",
           "index_workspace_size", "lightning_index_topk", "load", "sparse_mqa_attend",
           "timing_enable", "timing_read", "timing_reset"]
