"""GB300-native exact attention: fa_fwd / fa_bwd over a C-ABI CUDA library.

Importing the package is cheap; the shared library (``libfa.so``) is loaded
on first use and the import fails loudly when it is missing.  There is no
CPU fallback.
"""
from .binding import (  # noqa: F401
    FaError,
    fa_bwd,
    fa_bwd_strided,
    fa_bwd_varlen,
    fa_bwd_workspace_bytes,
    fa_decode_workspace_bytes,
    fa_device_status,
    fa_fwd,
    fa_fwd_decode,
    fa_fwd_fp8,
    fa_fwd_strided,
    fa_fwd_varlen,
    library,
    status_string,
)
