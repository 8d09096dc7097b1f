"""The allocation-free decode entry point, mla_decode_static.

It exists for callers that are handed device buffers but may not allocate
any (a plugin inside a runtime that owns all device memory, or a path where
cudaMalloc's possible device synchronisation is not allowed): its scratch is
a fixed array inside the library.  These tests call it through the C ABI and
check it against the workspace entry points (mla_decode followed by
mla_split_kv_combine with a caller-allocated workspace) on two calls in a
row with different inputs, so a call that read the previous call's leftovers
would fail.  This file sorts last so that a run stopping at its first failure
has already run every other test.
"""
import numpy as np
import pytest
import torch

import mla_inputs as mi
from mla_latent_kv_66_b300 import _lib as L
from oracle import mla_oracle as O

from helpers import bf16_dev, i32_dev, tol_ok, to_f64, upload_cache

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-2, 1e-3


def _inputs(lens, H, seed, kv="bf16"):
    w = mi.Workload("static", B=len(lens), H=H, L=0, ragged=(1, 2), seed=seed, pages="permuted")
    inp = mi.make_inputs(w, with_kv=False)
    inp["seq_lens"] = np.asarray(lens, np.int32)
    inp["page_table"], inp["num_pages"] = mi.page_layout(w, inp["seq_lens"])
    inp["kv_raw"] = {b: mi.kv_rows(w, b, int(lens[b])) for b in range(len(lens))}
    cache = O.build_cache(inp, "bf16" if kv == "bf16" else "e4m3")
    dev = dict(
        p=L.make_params(len(lens), H, inp["page_table"].shape[1], inp["num_pages"], kv),
        q_lat=bf16_dev(O.f64_to_bf16(O.absorb_q(inp["q_nope"], inp["w_uk"]))),
        q_pe=bf16_dev(O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])),
        table=i32_dev(inp["page_table"]), lens=i32_dev(inp["seq_lens"]))
    dev["ckv"], dev["kpe"], dev["sc"] = upload_cache(cache)
    return dev


def _with_workspace(d):
    p = d["p"]
    G = L.mla_decode_num_splits(p, 0)
    ws = torch.zeros(L.mla_decode_workspace_size(p, G), dtype=torch.uint8, device="cuda")
    o = torch.empty(p.B, p.H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(p.B, p.H, dtype=torch.float32, device="cuda")
    L.mla_decode(p, d["q_lat"], d["q_pe"], d["ckv"], d["kpe"], d["sc"], d["table"], d["lens"], G, ws, o, lse)
    L.mla_split_kv_combine(p, ws, G, o, lse)
    return o, lse


def _static(d):
    p = d["p"]
    o = torch.full((p.B, p.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.B, p.H), float("nan"), dtype=torch.float32, device="cuda")
    L.mla_decode_static(p, d["q_lat"], d["q_pe"], d["ckv"], d["kpe"], d["sc"], d["table"], d["lens"], o, lse)
    return o, lse


@pytest.mark.parametrize("kv", ["e4m3", "e4m3_mma"])
def test_static_scratch_with_an_e4m3_cache(kv):
    """The E4M3 caches through the fixed scratch (the tensor-core mode keeps
    its E4M3 query there too): bit-equal to the workspace entry points."""
    for d in (_inputs([1500, 64, 1, 300], H=128, seed=33, kv=kv), _inputs([900, 2500], H=128, seed=34, kv=kv)):
        o_ref, lse_ref = _with_workspace(d)
        o, lse = _static(d)
        torch.cuda.synchronize()
        assert L.mla_decode_static_status() == L.MLA_OK
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse, lse_ref)


def test_static_scratch_matches_the_workspace_entry_point_on_two_calls():
    """For these batches the fixed scratch holds the automatic partition
    count, so both entry points run the same kernels on the same schedule
    and must agree bit for bit; a stale partial from the previous call would
    show up as a difference.  (The branch that lowers the partition count
    until the workspace fits is reached only by batches of millions of
    sequences, and is covered here only by the rejection case below.)"""
    cases = [_inputs([2000, 64, 1, 777, 130], H=128, seed=31),
             _inputs([4096, 3000, 65], H=128, seed=32)]
    for d in cases:
        o_ref, lse_ref = _with_workspace(d)
        o, lse = _static(d)
        torch.cuda.synchronize()
        assert L.mla_decode_static_status() == L.MLA_OK
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse, lse_ref)
        ok, err, bound = tol_ok(to_f64(o), to_f64(o_ref), TOL_REL, TOL_ABS)
        assert ok, (err, bound)


def test_static_scratch_reports_device_side_errors():
    """A sequence length outside [1, max_pages*64] is skipped by the kernels
    and recorded in the scratch's error word, which the status call reads
    (and clears); the next call starts from a clear word."""
    d = _inputs([300, 100], H=16, seed=33)
    bad = dict(d)
    bad["lens"] = i32_dev(np.array([0, 100], np.int32))
    _static(bad)
    assert L.mla_decode_static_status(clear=True) == L.MLA_ERR_SEQ_LEN
    assert L.mla_decode_static_status() == L.MLA_OK
    _static(bad)
    _static(d)  # a good call clears the word when it starts
    assert L.mla_decode_static_status() == L.MLA_OK


def test_static_scratch_rejects_a_batch_too_large_for_it():
    # nine million sequences need 36 MB of page offsets alone, more than the
    # fixed 32 MiB scratch even with a single KV partition: the call is
    # refused on the host before anything is launched or dereferenced
    p = L.make_params(B=9_000_000, H=128, max_pages_per_seq=1, num_pages=1)
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(L.MLAError) as e:
        L.mla_decode_static(p, x, x, x, x, None, t, t, x, None)
    assert e.value.status == L.MLA_ERR_WORKSPACE
