"""Sink + short-window KV-cache attention for one GPU (sm_103a, B300).

The compute path is the CUDA library ``libsinkwin.so`` (C ABI in
``include/kvc.h``); this package only marshals arguments to it.  Importing the
package loads the library and fails if it has not been built.
"""

from ._abi import (KVC_BF16, KVC_FP4, KVC_OK, KVC_EINVAL, KVC_ESTATE, KVC_ECUDA,  # noqa: F401
                   KVC_ETIMEOUT, KVC_EUNSUPPORTED, KvcError, lib, status_string)
from .cache import KVCache, gemm_fp4, gemm_fp4_ws_bytes, quant_fp4  # noqa: F401

lib()  # load now: no silent fallback exists
