"""GB300-native paged split-K decode attention.

The computation lives in libpdecode.so (CUDA kernels for sm_103a behind the C
ABI of include/pdecode.h); this package is its thin Python binding plus the
seeded synthetic workload generator. Build the library with
``paged_split_decode_gb300.build.build()``.
"""
from .binding import (DEVERR_BLOCK_ID, DEVERR_QUERY_START, DEVERR_SEQ_LEN, DEVERR_SLOT,
                      DEVERR_TIMEOUT, DecodeError, decode_paged, decode_paged_combine,
                      decode_paged_varlen, dims_of, get_workspace, grid_ctas, load,
                      make_dims, status_str, workspace_bytes, write_kv_cache)

__all__ = ["DEVERR_BLOCK_ID", "DEVERR_QUERY_START", "DEVERR_SEQ_LEN", "DEVERR_SLOT",
           "DEVERR_TIMEOUT", "DecodeError", "decode_paged", "decode_paged_combine",
           "decode_paged_varlen", "dims_of", "get_workspace", "grid_ctas", "load",
           "make_dims", "status_str", "workspace_bytes", "write_kv_cache"]
