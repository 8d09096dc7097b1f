"""ctypes binding of libmla.so.  Argument marshalling only: every step runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.

The functions carry the C names (mla_absorb_q, mla_decode, ...) and take
torch tensors; a non-OK status raises MLAError.  If libmla.so is missing the
import fails: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla.so")

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA = 0, 1, 2, 3
MLA_ERR_PAGE_OOB, MLA_ERR_WORKSPACE, MLA_ERR_SEQ_LEN, MLA_ERR_TIMEOUT = 4, 5, 6, 7
MLA_KV_BF16, MLA_KV_E4M3, MLA_KV_E4M3_MMA, MLA_KV_E4M3_MMA1 = 0, 1, 2, 3
# kv_dtype names: the cache format, and for E4M3 how mla_decode multiplies it
KV_DTYPES = {"bf16": MLA_KV_BF16, "e4m3": MLA_KV_E4M3, "e4m3_mma": MLA_KV_E4M3_MMA, "e4m3_mma1": MLA_KV_E4M3_MMA1}
MLA_OUT_F32, MLA_OUT_BF16 = 0, 1
MLA_APPEND_RMSNORM, MLA_APPEND_ROPE = 1, 2


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


class MlaParams(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("kv_lora_rank", ctypes.c_int),
                ("rope_dim", ctypes.c_int), ("nope_dim", ctypes.c_int), ("v_dim", ctypes.c_int),
                ("page_size", ctypes.c_int), ("max_pages_per_seq", ctypes.c_int),
                ("num_pages", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("kv_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int)]


def make_params(B, H, max_pages_per_seq, num_pages, kv_dtype="bf16", out_dtype="f32",
                softmax_scale=None) -> MlaParams:
    return MlaParams(B, H, 512, 64, 128, 128, 64, max_pages_per_seq, num_pages,
                     1.0 / math.sqrt(192.0) if softmax_scale is None else softmax_scale,
                     KV_DTYPES[kv_dtype],
                     MLA_OUT_BF16 if out_dtype == "bf16" else MLA_OUT_F32)


_P = ctypes.c_void_p
_SIGS = {
    "mla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mla_version": (ctypes.c_int, []),
    "mla_decode_num_splits": (ctypes.c_int, [ctypes.POINTER(MlaParams), ctypes.c_int]),
    "mla_decode_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(MlaParams), ctypes.c_int]),
    "mla_workspace_offsets": (None, [ctypes.POINTER(MlaParams), ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "mla_workspace_query_offsets": (None, [ctypes.POINTER(MlaParams), ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_size_t)]),
    "mla_absorb_q": (ctypes.c_int, [ctypes.POINTER(MlaParams), _P, _P, _P, _P]),
    "mla_decode": (ctypes.c_int, [ctypes.POINTER(MlaParams), _P, _P, _P, _P, _P, _P, _P, ctypes.c_int,
                                  _P, ctypes.c_size_t, _P, _P, _P]),
    "mla_split_kv_combine": (ctypes.c_int, [ctypes.POINTER(MlaParams), _P, ctypes.c_size_t, ctypes.c_int,
                                            _P, _P, _P]),
    "mla_out_proj": (ctypes.c_int, [ctypes.POINTER(MlaParams), _P, _P, _P, _P]),
    "mla_combine_out_proj": (ctypes.c_int, [ctypes.POINTER(MlaParams), _P, ctypes.c_size_t, ctypes.c_int, _P, _P,
                                            _P, _P, _P, _P]),
    "mla_cache_append": (ctypes.c_int, [ctypes.POINTER(MlaParams), _P, _P, _P, ctypes.c_int, ctypes.c_int,
                                        _P, _P, _P, _P]),
    "mla_rope_q": (ctypes.c_int, [ctypes.POINTER(MlaParams), _P, _P, _P, _P]),
    "mla_workspace_status": (ctypes.c_int, [_P, ctypes.c_int, _P]),
    "mla_multi_token_expand": (ctypes.c_int, [ctypes.POINTER(MlaParams), ctypes.c_int, _P, _P, _P, _P, _P]),
    "mla_decode_static": (ctypes.c_int, [ctypes.POINTER(MlaParams), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "mla_decode_static_status": (ctypes.c_int, [ctypes.c_int, _P]),
    "mla_selftest_bounded_wait": (ctypes.c_int, [_P, _P]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m mla_latent_kv_66_b300.build` (there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(s: int) -> str:
    return lib.mla_status_string(int(s)).decode()


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(st, where):
    if st != MLA_OK:
        raise MLAError(st, where)


def mla_decode_num_splits(p: MlaParams, num_splits: int = 0) -> int:
    return lib.mla_decode_num_splits(ctypes.byref(p), num_splits)


def mla_decode_workspace_size(p: MlaParams, num_splits: int = 0) -> int:
    return lib.mla_decode_workspace_size(ctypes.byref(p), num_splits)


def mla_workspace_offsets(p: MlaParams, num_splits: int = 0):
    arr = (ctypes.c_size_t * 5)()
    lib.mla_workspace_offsets(ctypes.byref(p), num_splits, arr)
    return list(arr)


def mla_workspace_query_offsets(p: MlaParams, num_splits: int = 0):
    arr = (ctypes.c_size_t * 2)()
    lib.mla_workspace_query_offsets(ctypes.byref(p), num_splits, arr)
    return list(arr)


def mla_absorb_q(p, q_nope, w_uk, q_lat, stream=None):
    _check(lib.mla_absorb_q(ctypes.byref(p), _ptr(q_nope), _ptr(w_uk), _ptr(q_lat), _stream(stream)),
           "mla_absorb_q")


def mla_decode(p, q_lat, q_pe, ckv, kpe, kv_scale, page_table, seq_lens, num_splits, workspace,
               o_lat, lse=None, stream=None):
    _check(lib.mla_decode(ctypes.byref(p), _ptr(q_lat), _ptr(q_pe), _ptr(ckv), _ptr(kpe), _ptr(kv_scale),
                          _ptr(page_table), _ptr(seq_lens), num_splits, _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _ptr(o_lat), _ptr(lse),
                          _stream(stream)), "mla_decode")


def mla_split_kv_combine(p, workspace, num_splits, o_lat, lse=None, stream=None):
    _check(lib.mla_split_kv_combine(ctypes.byref(p), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), num_splits,
                                    _ptr(o_lat), _ptr(lse), _stream(stream)), "mla_split_kv_combine")


def mla_out_proj(p, o_lat, w_uv, out, stream=None):
    _check(lib.mla_out_proj(ctypes.byref(p), _ptr(o_lat), _ptr(w_uv), _ptr(out), _stream(stream)),
           "mla_out_proj")


def mla_combine_out_proj(p, workspace, num_splits, seq_lens, o_lat, w_uv, out, lse=None, stream=None):
    _check(lib.mla_combine_out_proj(ctypes.byref(p), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), num_splits, _ptr(seq_lens),
                                    _ptr(o_lat), _ptr(lse), _ptr(w_uv), _ptr(out), _stream(stream)),
           "mla_combine_out_proj")


def mla_cache_append(p, kv_rows, slots, positions, flags, ckv, kpe, kv_scale=None, stream=None):
    T = kv_rows.shape[0]
    _check(lib.mla_cache_append(ctypes.byref(p), _ptr(kv_rows), _ptr(slots), _ptr(positions), T, flags,
                                _ptr(ckv), _ptr(kpe), _ptr(kv_scale), _stream(stream)), "mla_cache_append")


def mla_rope_q(p, q_pe_raw, seq_lens, q_pe, stream=None):
    _check(lib.mla_rope_q(ctypes.byref(p), _ptr(q_pe_raw), _ptr(seq_lens), _ptr(q_pe), _stream(stream)),
           "mla_rope_q")


def mla_workspace_status(workspace, clear=False, stream=None) -> int:
    return lib.mla_workspace_status(_ptr(workspace), 1 if clear else 0, _stream(stream))


def mla_decode_static(p, q_lat, q_pe, ckv, kpe, kv_scale, page_table, seq_lens, o_lat, lse=None, stream=None):
    """Decode + split-KV combine with the library's fixed internal scratch
    (for callers that may not allocate device memory)."""
    _check(lib.mla_decode_static(ctypes.byref(p), _ptr(q_lat), _ptr(q_pe), _ptr(ckv), _ptr(kpe), _ptr(kv_scale),
                                 _ptr(page_table), _ptr(seq_lens), _ptr(o_lat), _ptr(lse), _stream(stream)),
           "mla_decode_static")


def mla_decode_static_status(clear=False, stream=None) -> int:
    """Error word of mla_decode_static's fixed scratch (synchronises the stream)."""
    return lib.mla_decode_static_status(1 if clear else 0, _stream(stream))


def mla_multi_token_expand(p, q_len, page_table, seq_lens, page_table_out, seq_lens_out, stream=None):
    """Rows b*q_len + i of the causal multi-token decode: page-table row b and
    length seq_lens[b] - q_len + 1 + i (p.B = number of sequences)."""
    _check(lib.mla_multi_token_expand(ctypes.byref(p), q_len, _ptr(page_table), _ptr(seq_lens), _ptr(page_table_out),
                                      _ptr(seq_lens_out), _stream(stream)), "mla_multi_token_expand")


def mla_selftest_bounded_wait(workspace, stream=None):
    _check(lib.mla_selftest_bounded_wait(_ptr(workspace), _stream(stream)), "mla_selftest_bounded_wait")
