"""MLA decode over a paged, compressed latent KV cache on one B300 (sm_103a).

The compute runs in libmla.so (hand-written CUDA); this package is its ctypes
binding plus a convenience wrapper for one decode step.  The library is
loaded on first use of any binding name; if it has not been built that use
raises ImportError (there is no CPU fallback).  `python -m
mla_latent_kv_66_b300.build` compiles it in-tree.
"""
_BINDINGS = ("MLAError", "MlaParams", "make_params", "mla_absorb_q", "mla_cache_append", "mla_decode",
             "mla_decode_num_splits", "mla_decode_workspace_size", "mla_out_proj", "mla_rope_q",
             "mla_split_kv_combine", "mla_workspace_offsets", "mla_workspace_status", "status_string",
             "mla_multi_token_expand", "mla_decode_static", "mla_decode_static_status",
             "mla_workspace_query_offsets", "KV_DTYPES", "mla_combine_out_proj",
             "MLA_APPEND_RMSNORM", "MLA_APPEND_ROPE", "LIB_PATH")


def __getattr__(name):
    if name in _BINDINGS:
        from . import _lib
        return getattr(_lib, name)
    if name == "MLADecodeStep":
        from .decoder import MLADecodeStep
        return MLADecodeStep
    raise AttributeError(name)
