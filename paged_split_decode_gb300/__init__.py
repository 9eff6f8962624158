"""GB300-native paged split-K decode attention.

The computation lives in libpdecode.so (CUDA kernels for sm_103a behind the C
ABI of include/pdecode.h); this package is its thin Python binding plus the
seeded synthetic workload generator. Build the library with
``paged_split_decode_gb300.build.build()``.
"""
from .binding import (DecodeError, decode_paged, decode_paged_combine, dims_of, get_workspace,
                      grid_ctas, load, make_dims, status_str, workspace_bytes)

__all__ = ["DecodeError", "decode_paged", "decode_paged_combine", "dims_of", "get_workspace",
           "grid_ctas", "load", "make_dims", "status_str", "workspace_bytes"]
