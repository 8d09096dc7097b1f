"""MLA decode over a paged, compressed latent KV cache on one B300 (sm_103a).

The compute runs in libmla.so (hand-written CUDA); this package is its ctypes
binding plus a convenience wrapper for one decode step."""
from ._lib import (MLAError, MlaParams, make_params, mla_absorb_q, mla_cache_append, mla_decode,  # noqa: F401
                   mla_decode_num_splits, mla_decode_workspace_size, mla_out_proj, mla_rope_q,
                   mla_split_kv_combine, mla_workspace_offsets, mla_workspace_status, status_string,
                   MLA_APPEND_RMSNORM, MLA_APPEND_ROPE, LIB_PATH)
from .decoder import MLADecodeStep  # noqa: F401
