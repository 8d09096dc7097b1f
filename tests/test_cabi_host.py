"""Host-only checks of the C ABI (no GPU needed): the library loads, exports
every entry point declared in include/mla.h, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import mla_latent_kv_66_b300 as mla
from mla_latent_kv_66_b300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 12
    raw = ctypes.CDLL(L.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings():
    for s in range(8):
        assert mla.status_string(s) and mla.status_string(s) != "unknown status"
    assert mla.status_string(99) == "unknown status"


def test_workspace_layout_matches_the_documented_formula():
    p = L.make_params(B=7, H=128, max_pages_per_seq=10, num_pages=70)
    G = 5
    assert L.mla_decode_num_splits(p, G) == G
    up = lambda x: (x + 255) // 256 * 256
    rec = 256
    seq = up(rec + 2 * G * 16)
    lse = up(seq + (7 + 1) * 4)
    po = up(lse + 2 * G * 128 * 4)
    total = up(po + 2 * G * 128 * 512 * 2)
    assert L.mla_workspace_offsets(p, G) == [0, rec, seq, lse, po]
    assert L.mla_decode_workspace_size(p, G) == total


def test_workspace_query_region_of_the_8bit_decode():
    G, up = 5, (lambda x: (x + 255) // 256 * 256)
    base = L.mla_decode_workspace_size(L.make_params(7, 128, 10, 70, "e4m3"), G)
    for kv in ("e4m3_mma", "e4m3_mma1"):
        p = L.make_params(B=7, H=128, max_pages_per_seq=10, num_pages=70, kv_dtype=kv)
        codes = base
        scale = up(codes + 7 * 128 * 2 * 576)
        assert L.mla_workspace_query_offsets(p, G) == [codes, scale]
        assert L.mla_decode_workspace_size(p, G) == up(scale + 7 * 128 * 4)
        # the rest of the layout is the one of the other kv_dtypes
        assert L.mla_workspace_offsets(p, G) == L.mla_workspace_offsets(L.make_params(7, 128, 10, 70), G)
    for kv in ("bf16", "e4m3"):
        assert L.mla_workspace_query_offsets(L.make_params(7, 128, 10, 70, kv), G) == [0, 0]


def _call_decode(p, ws_bytes=1 << 30, G=4, scale=None, nulls=()):
    fake = ctypes.c_void_p(0x1000)
    args = [fake] * 7
    for i in nulls:
        args[i] = None
    return L.lib.mla_decode(ctypes.byref(p) if p is not None else None, args[0], args[1], args[2],
                            args[3], scale, args[4], args[5], G, args[6], ws_bytes, fake, None, None)


def test_host_argument_checks_return_before_any_launch():
    p = L.make_params(B=2, H=128, max_pages_per_seq=4, num_pages=8)
    assert _call_decode(None) == L.MLA_ERR_INVALID_ARG
    assert _call_decode(p, nulls=(0,)) == L.MLA_ERR_INVALID_ARG
    assert _call_decode(p, ws_bytes=16) == L.MLA_ERR_WORKSPACE
    assert _call_decode(p, G=-1) == L.MLA_ERR_INVALID_ARG
    # bf16 cache with a scale pointer is a contradiction, an E4M3 cache without one too
    assert _call_decode(p, scale=ctypes.c_void_p(0x2000)) == L.MLA_ERR_INVALID_ARG
    for kv in ("e4m3", "e4m3_mma", "e4m3_mma1"):
        assert _call_decode(L.make_params(B=2, H=128, max_pages_per_seq=4, num_pages=8, kv_dtype=kv)) == \
            L.MLA_ERR_INVALID_ARG
    bad = L.make_params(B=2, H=128, max_pages_per_seq=4, num_pages=8)
    bad.kv_dtype = 4
    assert _call_decode(bad) == L.MLA_ERR_INVALID_ARG
    # the kernels move 16 bytes at a time: an unaligned tensor is refused
    fake, odd = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1008)
    for i in range(3):
        args = [fake] * 3
        args[i] = odd
        assert L.lib.mla_decode(ctypes.byref(p), args[0], args[1], fake, fake, None, fake, fake, 4, args[2],
                                1 << 30, fake, None, None) == L.MLA_ERR_INVALID_ARG
    assert L.lib.mla_split_kv_combine(ctypes.byref(p), fake, 1 << 30, 4, odd, None, None) == L.MLA_ERR_INVALID_ARG
    f = L.lib.mla_combine_out_proj
    assert f(ctypes.byref(p), fake, 1 << 30, 4, fake, odd, None, fake, fake, None) == L.MLA_ERR_INVALID_ARG
    assert f(ctypes.byref(p), fake, 1 << 30, 4, fake, fake, None, None, fake, None) == L.MLA_ERR_INVALID_ARG
    assert f(ctypes.byref(p), fake, 1 << 30, 4, None, fake, None, fake, fake, None) == L.MLA_ERR_INVALID_ARG
    assert f(ctypes.byref(p), fake, 16, 4, fake, fake, None, fake, fake, None) == L.MLA_ERR_WORKSPACE
    assert f(ctypes.byref(p), None, 1 << 30, 4, fake, fake, None, fake, fake, None) == L.MLA_ERR_WORKSPACE
    bad = L.make_params(B=2, H=128, max_pages_per_seq=4, num_pages=8)
    bad.kv_lora_rank = 256
    assert _call_decode(bad) == L.MLA_ERR_UNSUPPORTED
    bad = L.make_params(B=2, H=24, max_pages_per_seq=4, num_pages=8)
    assert _call_decode(bad) == L.MLA_ERR_UNSUPPORTED
    bad = L.make_params(B=0, H=128, max_pages_per_seq=4, num_pages=8)
    assert _call_decode(bad) == L.MLA_ERR_INVALID_ARG
    bad = L.make_params(B=2, H=128, max_pages_per_seq=4, num_pages=8, softmax_scale=float("nan"))
    assert _call_decode(bad) == L.MLA_ERR_INVALID_ARG
    fake = ctypes.c_void_p(0x1000)
    assert L.lib.mla_absorb_q(ctypes.byref(p), None, fake, fake, None) == L.MLA_ERR_INVALID_ARG
    odd8 = ctypes.c_void_p(0x1008)
    for i in range(3):  # q_nope, w_uk, q_lat: 16-byte alignment
        args = [fake] * 3
        args[i] = odd8
        assert L.lib.mla_absorb_q(ctypes.byref(p), *args, None) == L.MLA_ERR_INVALID_ARG
    assert L.lib.mla_out_proj(ctypes.byref(p), fake, None, fake, None) == L.MLA_ERR_INVALID_ARG
    assert L.lib.mla_cache_append(ctypes.byref(p), fake, fake, fake, -1, 3, fake, fake, None, None) \
        == L.MLA_ERR_INVALID_ARG
    assert L.lib.mla_cache_append(ctypes.byref(p), fake, fake, fake, 4, 8, fake, fake, None, None) \
        == L.MLA_ERR_INVALID_ARG
    assert L.lib.mla_workspace_status(None, 0, None) == L.MLA_ERR_INVALID_ARG


def test_python_binding_refuses_host_tensors():
    import torch
    p = L.make_params(B=1, H=16, max_pages_per_seq=1, num_pages=1)
    x = torch.zeros(1, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mla.mla_absorb_q(p, x, x, x)
