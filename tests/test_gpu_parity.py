"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs.

Tolerances (the contract for this path): bf16 cache
max|out - ref| <= 1e-2 * max|ref| + 1e-3; FP8 cache: the bf16 bound against
the oracle run on the decoded E4M3 cache, and <= 5e-2 * max|ref| against the
oracle run on the unquantised bf16 cache; page-table and split indexing
bit-exact.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import mla_inputs as mi
import mla_latent_kv_66_b300 as mla
from mla_latent_kv_66_b300 import _lib as L
from oracle import mla_oracle as O

from helpers import (bf16_bits, bf16_dev, i32_dev, reference_partition, sample_pairs, tol_ok,
                     to_f64, upload_cache)

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-2, 1e-3


def small_inputs(lens, H=16, seed=21, pages="permuted"):
    w = mi.Workload("t", B=len(lens), H=H, L=0, ragged=(1, 2), seed=seed, pages=pages)
    inp = mi.make_inputs(w, with_kv=False)
    inp["seq_lens"] = np.asarray(lens, np.int32)
    inp["page_table"], inp["num_pages"] = mi.page_layout(w, inp["seq_lens"])
    inp["kv_raw"] = {b: mi.kv_rows(w, b, int(lens[b])) for b in range(len(lens))}
    return inp


def garbage(inp, nan_tail=False):
    g = mi.garbage_pool_bits(inp["workload"], inp["num_pages"], 512), \
        mi.garbage_pool_bits(inp["workload"], inp["num_pages"], 64)
    if nan_tail:
        g = tuple(np.where(np.arange(x.shape[1])[None, :, None] % 2 == 1, np.uint16(0x7FC0), x) for x in g)
    return g


def run_gpu(inp, cache, q_pe_bits, num_splits, q_lat_bits=None, out_dtype="f32"):
    w = inp["workload"]
    B, H = len(inp["seq_lens"]), w.H
    table = inp["page_table"]
    p = L.make_params(B, H, table.shape[1], inp["num_pages"], cache["kv_dtype"], out_dtype)
    G = L.mla_decode_num_splits(p, num_splits)
    ws = torch.zeros(L.mla_decode_workspace_size(p, G), dtype=torch.uint8, device="cuda")
    ckv, kpe, sc = upload_cache(cache)
    qn, wuk, wuv = bf16_dev(inp["q_nope"]), bf16_dev(inp["w_uk"]), bf16_dev(inp["w_uv"])
    qpe = bf16_dev(q_pe_bits)
    tab, lens = i32_dev(table), i32_dev(inp["seq_lens"])
    q_lat = torch.empty(B, H, 512, dtype=torch.bfloat16, device="cuda")
    L.mla_absorb_q(p, qn, wuk, q_lat)
    q_used = bf16_dev(q_lat_bits) if q_lat_bits is not None else q_lat
    o_lat = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    L.mla_decode(p, q_used, qpe, ckv, kpe, sc, tab, lens, G, ws, o_lat, lse)
    L.mla_split_kv_combine(p, ws, G, o_lat, lse)
    out = torch.empty(B, H, 128, dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32, device="cuda")
    L.mla_out_proj(p, o_lat, wuv, out)
    torch.cuda.synchronize()
    st = L.mla_workspace_status(ws)
    return dict(q_lat=q_lat, o_lat=o_lat, lse=lse, out=out, ws=ws, p=p, G=G, status=st)


def oracle_all(inp, cache, q_pe_bits, pairs=None):
    return O.decode_reference(cache, inp, q_pe_bits, pairs)


# ------------------------------------------------------------------ tiny workload, every output
def test_tiny_workload_end_to_end_all_heads():
    inp = mi.make_inputs(mi.WORKLOADS["tiny"])
    cache = O.build_cache(inp, garbage=garbage(inp))
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    r = run_gpu(inp, cache, qpe, num_splits=0)
    assert r["status"] == 0
    ref, lse_ref = oracle_all(inp, cache, qpe)
    got = to_f64(r["out"]).reshape(-1, 128)
    ok, err, bound = tol_ok(got, ref, TOL_REL, TOL_ABS)
    assert ok, (err, bound)
    # intermediates: q_lat within one bf16 rounding of the fp64 absorption
    qref = O.absorb_q(inp["q_nope"], inp["w_uk"])
    qgot = to_f64(r["q_lat"])
    assert np.all(np.abs(qgot - qref) <= 2.0 ** -8 * np.abs(qref) + 1e-6 * np.abs(qref).max())
    assert np.allclose(to_f64(r["lse"]).reshape(-1), lse_ref, rtol=0, atol=1e-3)


@pytest.mark.parametrize("splits", [1, 3, 8, 64])
def test_decode_kernel_on_exact_q_lat(splits):
    inp = small_inputs([700, 64, 1, 130, 65])
    cache = O.build_cache(inp, garbage=garbage(inp))
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    qlat_ref = O.absorb_q(inp["q_nope"], inp["w_uk"])
    qlat_bits = O.f64_to_bf16(qlat_ref)
    r = run_gpu(inp, cache, qpe, splits, q_lat_bits=qlat_bits)
    assert r["status"] == 0
    qp = O.bf16_to_f64(qpe)
    ql = O.bf16_to_f64(qlat_bits)
    got = to_f64(r["o_lat"])
    for b in range(len(inp["seq_lens"])):
        n = int(inp["seq_lens"][b])
        c, kp = O.gather_sequence(cache, inp["page_table"], b, n)
        for h in range(inp["workload"].H):
            o_ref, lse_ref = O.latent_attention(c, kp, ql[b, h], qp[b, h])
            ok, err, bound = tol_ok(got[b, h], o_ref, TOL_REL, TOL_ABS)
            assert ok, (b, h, err, bound)
            assert abs(float(r["lse"][b, h]) - lse_ref) < 1e-3


def test_one_token_context_returns_the_cached_latent_exactly():
    inp = small_inputs([1, 1, 1])
    cache = O.build_cache(inp, garbage=garbage(inp))
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    r = run_gpu(inp, cache, qpe, 2)
    for b in range(3):
        pg = inp["page_table"][b, 0]
        c0 = cache["ckv"][pg, 0]
        for h in range(16):
            assert np.array_equal(bf16_bits(r["o_lat"][b, h]), c0)


def test_garbage_and_nan_past_sequence_end_are_ignored():
    inp = small_inputs([70, 5, 127])
    cache = O.build_cache(inp, garbage=garbage(inp, nan_tail=True))
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    r = run_gpu(inp, cache, qpe, 4)
    ref, _ = oracle_all(inp, cache, qpe)
    got = to_f64(r["out"]).reshape(-1, 128)
    assert np.all(np.isfinite(got))
    assert tol_ok(got, ref, TOL_REL, TOL_ABS)[0]


@pytest.mark.parametrize("gain", [4, 8, 16])
def test_sharp_softmax_at_large_logits(gain):
    """Peaked softmax rows: the query scaled by 4, 8 or 16 (exact in bf16),
    so the logits have standard deviation 4-16 and the log2-domain scores
    reach about 7 times the gain (past 100 at 16), where the rounding of the
    partial scores the two CTAs of a cluster exchange matters most.  The
    decode on exact q_lat against the oracle's absorbed attention (every head
    of every sequence, output and LSE), and the whole path against the
    non-absorbed oracle, at the bf16 bound."""
    inp = small_inputs([700, 64, 1, 130, 4096], H=128, seed=25)
    g = O.f64_to_bf16(float(gain) * O.bf16_to_f64(inp["q_nope"]))
    inp["q_nope"] = g
    inp["q_pe_raw"] = O.f64_to_bf16(float(gain) * O.bf16_to_f64(inp["q_pe_raw"]))
    cache = O.build_cache(inp, garbage=garbage(inp))
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    qlat_bits = O.f64_to_bf16(O.absorb_q(inp["q_nope"], inp["w_uk"]))
    for splits in (1, 9):
        r = run_gpu(inp, cache, qpe, splits, q_lat_bits=qlat_bits)
        assert r["status"] == 0
        qp, ql = O.bf16_to_f64(qpe), O.bf16_to_f64(qlat_bits)
        got = to_f64(r["o_lat"])
        peak = 0.0
        for b in range(len(inp["seq_lens"])):
            n = int(inp["seq_lens"][b])
            c, kp = O.gather_sequence(cache, inp["page_table"], b, n)
            s_max = np.max(np.abs(c @ ql[b].T + kp @ qp[b].T)) / math.sqrt(192.0) * math.log2(math.e)
            peak = max(peak, s_max)
            for h in range(128):
                o_ref, lse_ref = O.latent_attention(c, kp, ql[b, h], qp[b, h])
                ok, err, bound = tol_ok(got[b, h], o_ref, TOL_REL, TOL_ABS)
                assert ok, (gain, splits, b, h, err, bound)
                assert abs(float(r["lse"][b, h]) - lse_ref) < 1e-3 * max(1.0, abs(lse_ref)), (b, h)
        assert peak > 6 * gain  # the scores really are large
    r = run_gpu(inp, cache, qpe, 0)
    ref, _ = oracle_all(inp, cache, qpe, [(b, h) for b in range(5) for h in (0, 31, 77, 127)])
    got = np.stack([to_f64(r["out"][b, h]) for b in range(5) for h in (0, 31, 77, 127)])
    ok, err, bound = tol_ok(got, ref, TOL_REL, TOL_ABS)
    assert ok, (gain, err, bound)


# ------------------------------------------------------------------ split indexing, bit-exact
@pytest.mark.parametrize("lens,G", [([700, 64, 1, 130, 65], 7), ([4096] * 3, 5), ([64] * 9, 4),
                                    ([3000, 10, 2000], 64), ([1, 2, 3], 8)])
def test_split_records_match_the_documented_partition(lens, G):
    inp = small_inputs(lens)
    cache = O.build_cache(inp)
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    r = run_gpu(inp, cache, qpe, G)
    offs = L.mla_workspace_offsets(r["p"], G)
    raw = r["ws"].cpu().numpy()
    rec = raw[offs[1]: offs[1] + 2 * G * 16].view(np.int32).reshape(2 * G, 4)
    start = raw[offs[2]: offs[2] + (len(lens) + 1) * 4].view(np.int32)
    ref_rec, ref_start = reference_partition(inp["seq_lens"].tolist(), inp["page_table"].shape[1], G)
    assert np.array_equal(start, np.array(ref_start, np.int32))
    assert [tuple(x) for x in rec.tolist()] == ref_rec


def test_page_permutation_is_bit_exact_for_a_fixed_schedule():
    inp = small_inputs([300, 129, 64], pages="contiguous")
    cache = O.build_cache(inp, garbage=garbage(inp))
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    r1 = run_gpu(inp, cache, qpe, 5)
    perm = np.random.default_rng(4).permutation(inp["num_pages"]).astype(np.int32)
    inv = np.argsort(perm)
    moved = dict(cache)
    moved["ckv"], moved["kpe"] = cache["ckv"][inv], cache["kpe"][inv]
    inp2 = dict(inp)
    inp2["page_table"] = np.where(inp["page_table"] >= 0, perm[np.maximum(inp["page_table"], 0)], -1)
    r2 = run_gpu(inp2, moved, qpe, 5)
    assert torch.equal(r1["o_lat"].view(torch.int16), r2["o_lat"].view(torch.int16))
    assert torch.equal(r1["out"], r2["out"])


def test_split_counts_agree_within_tolerance():
    inp = small_inputs([2000, 777])
    cache = O.build_cache(inp)
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    a = to_f64(run_gpu(inp, cache, qpe, 1)["out"])
    b = to_f64(run_gpu(inp, cache, qpe, 41)["out"])
    assert tol_ok(b, a, TOL_REL, TOL_ABS)[0]


def test_combine_with_many_partials_per_sequence():
    """More than 32 partials per sequence, some from empty worker ranges, in a
    batch large enough for the grouped combine (one warp per head merging the
    partials 32 at a time with a running maximum): sampled (sequence, head)
    pairs against the oracle on exact q_lat, every output against the
    unsplit run."""
    lens = [4096 - 61 * b for b in range(19)]
    inp = small_inputs(lens, H=128, seed=23)
    cache = O.build_cache(inp)
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    qlat_bits = O.f64_to_bf16(O.absorb_q(inp["q_nope"], inp["w_uk"]))
    pages = int(sum((n + 63) // 64 for n in lens))
    r = run_gpu(inp, cache, qpe, 2 * pages, q_lat_bits=qlat_bits)  # every other worker range is empty
    assert r["status"] == 0 and r["G"] == 2 * pages
    whole = run_gpu(inp, cache, qpe, 1, q_lat_bits=qlat_bits)
    assert whole["status"] == 0
    got, ref_whole = to_f64(r["o_lat"]), to_f64(whole["o_lat"])
    assert tol_ok(got.reshape(-1, 512), ref_whole.reshape(-1, 512), TOL_REL, TOL_ABS)[0]
    assert np.allclose(to_f64(r["lse"]), to_f64(whole["lse"]), rtol=0, atol=1e-3)
    qp, ql = O.bf16_to_f64(qpe), O.bf16_to_f64(qlat_bits)
    for b in (0, 9, 18):
        c, kp = O.gather_sequence(cache, inp["page_table"], b, lens[b])
        for h in (0, 5, 64, 127):
            o_ref, lse_ref = O.latent_attention(c, kp, ql[b, h], qp[b, h])
            ok, err, bound = tol_ok(got[b, h], o_ref, TOL_REL, TOL_ABS)
            assert ok, (b, h, err, bound)
            assert abs(float(r["lse"][b, h]) - lse_ref) < 1e-3


# ------------------------------------------------------------------ device-side error word
def test_out_of_range_page_and_bad_length_set_the_error_word():
    inp = small_inputs([200, 100])
    cache = O.build_cache(inp)
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    bad = dict(inp)
    bad["page_table"] = inp["page_table"].copy()
    bad["page_table"][0, 1] = inp["num_pages"] + 5
    r = run_gpu(bad, cache, qpe, 3)
    assert r["status"] == L.MLA_ERR_PAGE_OOB
    assert L.mla_workspace_status(r["ws"], clear=True) == L.MLA_ERR_PAGE_OOB
    assert L.mla_workspace_status(r["ws"]) == 0
    bad = dict(inp)
    bad["seq_lens"] = np.array([0, 100], np.int32)
    r = run_gpu(bad, cache, qpe, 3)
    assert r["status"] == L.MLA_ERR_SEQ_LEN
    # the valid sequence is still decoded correctly
    ref, _ = oracle_all(inp, cache, qpe, [(1, h) for h in range(16)])
    assert tol_ok(to_f64(r["out"][1]), ref, TOL_REL, TOL_ABS)[0]


def test_host_rejects_bad_arguments_with_an_error():
    p = L.make_params(1, 16, 1, 1)
    x = torch.zeros(1, 16, 128, dtype=torch.bfloat16, device="cuda")
    bad = L.make_params(1, 16, 1, 1)
    bad.rope_dim = 32
    with pytest.raises(mla.MLAError):
        L.mla_absorb_q(bad, x, x, x)
    with pytest.raises(mla.MLAError):
        L.mla_out_proj(p, x, x, None)


# ------------------------------------------------------------------ bounded waits
def test_a_wait_that_never_completes_ends_with_a_timeout_status():
    """The library's bounded mbarrier wait on a barrier nothing completes:
    after its limit the kernel records MLA_ERR_TIMEOUT and returns, and the
    context stays usable (a decode runs correctly right after)."""
    import time
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    L.mla_selftest_bounded_wait(ws)
    assert L.mla_workspace_status(ws) == L.MLA_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 1.5
    inp = small_inputs([130, 64])
    cache = O.build_cache(inp)
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    r = run_gpu(inp, cache, qpe, 2)
    assert r["status"] == 0
    ref, _ = oracle_all(inp, cache, qpe)
    assert tol_ok(to_f64(r["out"]).reshape(-1, 128), ref, TOL_REL, TOL_ABS)[0]


# ------------------------------------------------------------------ combine fused into the out-projection
@pytest.mark.parametrize("lens,G,H", [([700, 64, 1, 130, 65, 2000], 7, 16), ([4096] * 32, 0, 128),
                                      ([1500] * 40, 64, 128)])
def test_combine_fused_into_out_projection(lens, G, H):
    """mla_combine_out_proj against mla_split_kv_combine + mla_out_proj on the
    same decode: bit-exact (out, o_lat, lse) where the separate combine takes
    its grouped form (B * ceil(H/8) >= 2 x SMs), within rounding otherwise;
    and against the oracle."""
    inp = small_inputs(lens, H=H, seed=29)
    cache = O.build_cache(inp, garbage=garbage(inp))
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    B = len(lens)
    table = inp["page_table"]
    p = L.make_params(B, H, table.shape[1], inp["num_pages"])
    G = L.mla_decode_num_splits(p, G)
    ws = torch.zeros(L.mla_decode_workspace_size(p, G), dtype=torch.uint8, device="cuda")
    ckv, kpe, sc = upload_cache(cache)
    q_lat = torch.empty(B, H, 512, dtype=torch.bfloat16, device="cuda")
    L.mla_absorb_q(p, bf16_dev(inp["q_nope"]), bf16_dev(inp["w_uk"]), q_lat)
    o_a = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse_a = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    L.mla_decode(p, q_lat, bf16_dev(qpe), ckv, kpe, sc, i32_dev(table), i32_dev(inp["seq_lens"]), G, ws, o_a, lse_a)
    o_b, lse_b = o_a.clone(), lse_a.clone()
    wuv = bf16_dev(inp["w_uv"])
    out_a = torch.empty(B, H, 128, dtype=torch.float32, device="cuda")
    out_b = torch.full((B, H, 128), float("nan"), dtype=torch.float32, device="cuda")
    L.mla_split_kv_combine(p, ws, G, o_a, lse_a)
    L.mla_out_proj(p, o_a, wuv, out_a)
    L.mla_combine_out_proj(p, ws, G, i32_dev(inp["seq_lens"]), o_b, wuv, out_b, lse_b)
    torch.cuda.synchronize()
    assert L.mla_workspace_status(ws) == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if B * ((H + 7) // 8) >= 2 * sms:
        assert torch.equal(o_a, o_b) and torch.equal(lse_a, lse_b) and torch.equal(out_a, out_b)
    else:
        assert tol_ok(to_f64(out_b), to_f64(out_a), 1e-2, 1e-3)[0]
        assert tol_ok(to_f64(o_b), to_f64(o_a), 1e-2, 1e-3)[0]
        assert np.allclose(to_f64(lse_b), to_f64(lse_a), atol=1e-4)
    pairs = sample_pairs(B, H, 3, 3, seed=7)
    ref, lse_ref = O.decode_reference(cache, inp, qpe, pairs)
    got = np.stack([to_f64(out_b[b, h]) for b, h in pairs])
    ok, err, bound = tol_ok(got, ref, TOL_REL, TOL_ABS)
    assert ok, (err, bound)
    assert np.allclose([float(lse_b[b, h]) for b, h in pairs], lse_ref, atol=1e-3)


def test_batch_larger_than_one_gemm_tile():
    """B = 300 short sequences through the decode step: the absorption
    (batch tiles of up to 256) and the fused combine + out-projection (tiles
    of up to 128) each run several batch tiles; sampled outputs of every
    tile against the oracle."""
    rng = np.random.default_rng(41)
    lens = rng.integers(1, 300, size=300).tolist()
    inp = small_inputs(lens, H=16, seed=43)
    cache = O.build_cache(inp, garbage=garbage(inp))
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    B, table = len(lens), inp["page_table"]
    step = mla.MLADecodeStep(B, 16, table.shape[1], inp["num_pages"])
    out = step(bf16_dev(inp["q_nope"]), bf16_dev(qpe), bf16_dev(inp["w_uk"]), bf16_dev(inp["w_uv"]),
               *upload_cache(cache), i32_dev(table), i32_dev(inp["seq_lens"]))
    torch.cuda.synchronize()
    assert step.status() == 0
    pairs = [(b, h) for b in (0, 127, 128, 200, 255, 256, 299) for h in (0, 9, 15)]
    ref, _ = O.decode_reference(cache, inp, qpe, pairs)
    got = np.stack([to_f64(out[b, h]) for b, h in pairs])
    ok, err, bound = tol_ok(got, ref, TOL_REL, TOL_ABS)
    assert ok, (err, bound)


# ------------------------------------------------------------------ FP8 cache
def test_fp8_cache_small():
    inp = small_inputs([300, 64, 1, 129])
    cache8 = O.build_cache(inp, "e4m3", garbage=garbage(inp))
    cache = O.build_cache(inp, garbage=garbage(inp))
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    r = run_gpu(inp, cache8, qpe, 3, out_dtype="bf16")
    assert r["status"] == 0
    got = to_f64(r["out"]).reshape(-1, 128)
    ref8, _ = oracle_all(inp, cache8, qpe)
    assert tol_ok(got, ref8, TOL_REL, TOL_ABS)[0]
    ref, _ = oracle_all(inp, cache, qpe)
    assert tol_ok(got, ref, 5e-2)[0]


# ------------------------------------------------------------------ cache write and query RoPE
def test_cache_append_bf16_and_rope_q():
    inp = small_inputs([300, 70])
    w = inp["workload"]
    rows = np.concatenate([inp["kv_raw"][b] for b in range(2)])
    slots = np.concatenate([inp["page_table"][b, np.arange(n) // 64] * 64 + np.arange(n) % 64
                            for b, n in enumerate(inp["seq_lens"])]).astype(np.int32)
    pos = np.concatenate([np.arange(n) for n in inp["seq_lens"]]).astype(np.int32)
    p = L.make_params(2, w.H, inp["page_table"].shape[1], inp["num_pages"])
    ckv = torch.zeros(inp["num_pages"], 64, 512, dtype=torch.bfloat16, device="cuda")
    kpe = torch.zeros(inp["num_pages"], 64, 64, dtype=torch.bfloat16, device="cuda")
    L.mla_cache_append(p, bf16_dev(rows), i32_dev(slots), i32_dev(pos), 3, ckv, kpe)
    ref = O.build_cache(inp)
    got_c, got_k = bf16_bits(ckv), bf16_bits(kpe)
    for g, r_ in ((got_c, ref["ckv"]), (got_k, ref["kpe"])):
        d = np.abs(g.astype(np.int32) - r_.astype(np.int32))
        assert d.max() <= 1 and np.mean(d == 0) > 0.999
    qraw = bf16_dev(inp["q_pe_raw"])
    q = torch.empty_like(qraw)
    L.mla_rope_q(p, qraw, i32_dev(inp["seq_lens"]), q)
    d = np.abs(bf16_bits(q).astype(np.int32) - O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"]).astype(np.int32))
    assert d.max() <= 1 and np.mean(d == 0) > 0.999


def test_fp8_encoding_is_bit_exact_on_identical_rows():
    inp = small_inputs([333])
    ref = O.build_cache(inp)  # bf16 cache rows (normalised, rotated)
    n = 333
    t = np.arange(n)
    pg, sl = inp["page_table"][0, t // 64], t % 64
    rows = np.concatenate([ref["ckv"][pg, sl], ref["kpe"][pg, sl]], axis=1)
    # add some extreme rows: zeros, tiny, huge, ties
    extra = np.zeros((3, 576), np.uint16)
    extra[1, :] = O.f64_to_bf16(np.full(576, 1e-30))
    extra[2, :] = O.f64_to_bf16(np.linspace(-3e4, 3e4, 576))
    rows = np.concatenate([rows, extra])
    codes_ref, scale_ref = O.quantize_rows_e4m3(rows)
    T = rows.shape[0]
    npages = (T + 63) // 64
    p = L.make_params(1, 16, npages, npages, "e4m3")
    ckv = torch.zeros(npages, 64, 512, dtype=torch.uint8, device="cuda")
    kpe = torch.zeros(npages, 64, 64, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(npages, 64, dtype=torch.float32, device="cuda")
    L.mla_cache_append(p, bf16_dev(rows), i32_dev(np.arange(T)), i32_dev(np.zeros(T)), 0, ckv, kpe, sc)
    got = np.concatenate([ckv.cpu().numpy().reshape(-1, 512)[:T], kpe.cpu().numpy().reshape(-1, 64)[:T]], 1)
    assert np.array_equal(got, codes_ref)
    assert np.array_equal(sc.cpu().numpy().reshape(-1)[:T], scale_ref)


def _append_e4m3(rows):
    T = rows.shape[0]
    npages = (T + 63) // 64
    p = L.make_params(1, 16, npages, npages, "e4m3")
    ckv = torch.zeros(npages, 64, 512, dtype=torch.uint8, device="cuda")
    kpe = torch.zeros(npages, 64, 64, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(npages, 64, dtype=torch.float32, device="cuda")
    L.mla_cache_append(p, bf16_dev(rows), i32_dev(np.arange(T)), i32_dev(np.zeros(T)), 0, ckv, kpe, sc)
    codes = np.concatenate([ckv.cpu().numpy().reshape(-1, 512)[:T], kpe.cpu().numpy().reshape(-1, 64)[:T]], 1)
    return codes, sc.cpu().numpy().reshape(-1)[:T]


def test_fp8_encoder_on_every_finite_bf16_pattern():
    """Every finite bf16 bit pattern through the GPU's E4M3 cache encoder,
    bit-exact against the oracle's: (a) in rows whose largest magnitude is
    448, so the scale is exactly 1 and the code is E4M3(v) itself (every
    pattern with |v| <= 448, subnormals included); (b) all finite patterns
    sorted by magnitude, 576 to a row, so the scales run from subnormal to
    the bf16 maximum over 448; (c) the same patterns in a seeded shuffle."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = pats[(pats & 0x7F80) != 0x7F80]
    vals = O.bf16_to_f64(finite)
    in_range = finite[np.abs(vals) <= 448.0]
    marker = O.f64_to_bf16(np.array([448.0]))[0]
    n_per = 575
    k = (len(in_range) + n_per - 1) // n_per
    a = np.full((k, 576), marker, np.uint16)
    flat = a[:, :n_per].reshape(-1)
    flat[: len(in_range)] = in_range
    a[:, :n_per] = flat.reshape(k, n_per)
    order = np.argsort(np.abs(vals), kind="stable")
    srt = finite[order]
    pad = (-len(srt)) % 576
    b_rows = np.concatenate([srt, srt[:pad]]).reshape(-1, 576)
    shuf = finite[np.random.default_rng(41).permutation(len(finite))]
    c_rows = np.concatenate([shuf, shuf[:(-len(shuf)) % 576]]).reshape(-1, 576)
    rows = np.concatenate([a, b_rows, c_rows])
    codes, scale = _append_e4m3(rows)
    codes_ref, scale_ref = O.quantize_rows_e4m3(rows)
    assert np.array_equal(scale, scale_ref)
    assert np.all(scale[:k] == 1.0)
    bad = np.argwhere(codes != codes_ref)
    assert bad.size == 0, (bad[:5], rows[tuple(bad[0])], codes[tuple(bad[0])], codes_ref[tuple(bad[0])])
    # every in-range pattern was encoded with scale 1: its code is E4M3(v)
    assert np.array_equal(codes[:k, :n_per].reshape(-1)[: len(in_range)],
                          O.f32_to_e4m3(O.bf16_to_f64(in_range).astype(np.float32)))


# ------------------------------------------------------------------ several query tokens per sequence
def multi_inputs(lens, T, H=16, seed=27):
    w = mi.Workload("m", B=len(lens), H=H, L=0, ragged=(1, 2), seed=seed, pages="permuted", q_len=T)
    inp = mi.make_inputs(w, with_kv=False)
    inp["seq_lens"] = np.asarray(lens, np.int32)
    inp["page_table"], inp["num_pages"] = mi.page_layout(w, inp["seq_lens"])
    inp["kv_raw"] = {b: mi.kv_rows(w, b, int(lens[b])) for b in range(len(lens))}
    return inp


def run_multi(inp, cache, q_pe_bits, T, num_splits=0):
    B, H = len(inp["seq_lens"]), inp["workload"].H
    table = inp["page_table"]
    step = mla.MLADecodeStep(B, H, table.shape[1], inp["num_pages"], cache["kv_dtype"], num_splits=num_splits,
                             q_len=T)
    ckv, kpe, sc = upload_cache(cache)
    out = step(bf16_dev(inp["q_nope"]), bf16_dev(q_pe_bits), bf16_dev(inp["w_uk"]), bf16_dev(inp["w_uv"]),
               ckv, kpe, sc, i32_dev(table), i32_dev(inp["seq_lens"]))
    torch.cuda.synchronize()
    return step, out


def test_multi_token_decode_against_the_oracle():
    """Three query tokens per sequence with a causal mask, through the row
    expansion and the decode step: every (sequence, token, head) against the
    oracle, including a sequence exactly as long as the query block; the
    expanded page table and lengths bit-exact; the GPU query rotation at the
    expanded lengths within one bf16 ulp of the oracle's."""
    T = 3
    lens = [3, 70, 200, 64]
    inp = multi_inputs(lens, T)
    cache = O.build_cache(inp, garbage=garbage(inp))
    qpe = O.rope_q_multi_bf16(inp["q_pe_raw"], inp["seq_lens"], T)
    for splits in (0, 5):
        step, out = run_multi(inp, cache, qpe, T, splits)
        assert step.status() == 0
        ref, _ = O.decode_multi_reference(cache, inp, qpe, T)
        got = to_f64(out).reshape(-1, 128)
        ok, err, bound = tol_ok(got, ref, TOL_REL, TOL_ABS)
        assert ok, (splits, err, bound)
        # the LSE against the absorbed attention on the GPU's own q_lat, over
        # each row's visible tokens (a one-token row's LSE is a single score,
        # so the bf16 rounding of q_lat would dominate a comparison with the
        # non-absorbed oracle)
        ql, qp = to_f64(step.q_lat).reshape(len(lens), T, 16, 512), O.bf16_to_f64(qpe)
        glse = to_f64(step.lse).reshape(len(lens), T, 16)
        for b, n in enumerate(lens):
            c, kp = O.gather_sequence(cache, inp["page_table"], b, n)
            for i in range(T):
                vis = n - T + 1 + i
                for h in range(16):
                    _, lse_ref = O.latent_attention(c[:vis], kp[:vis], ql[b, i, h], qp[b, i, h])
                    assert abs(glse[b, i, h] - lse_ref) < 1e-3, (splits, b, i, h)
    table, rows_lens = step.table_rows.cpu().numpy(), step.lens_rows.cpu().numpy()
    assert np.array_equal(table, np.repeat(inp["page_table"], T, axis=0))
    assert np.array_equal(rows_lens, np.array([n - T + 1 + i for n in lens for i in range(T)], np.int32))
    p = L.make_params(len(lens) * T, 16, inp["page_table"].shape[1], inp["num_pages"])
    q = torch.empty(len(lens) * T, 16, 64, dtype=torch.bfloat16, device="cuda")
    L.mla_rope_q(p, bf16_dev(inp["q_pe_raw"].reshape(-1, 16, 64)), step.lens_rows, q)
    d = np.abs(bf16_bits(q).astype(np.int32) - qpe.reshape(-1, 16, 64).astype(np.int32))
    assert d.max() <= 1 and np.mean(d == 0) > 0.999


def test_multi_token_sequence_shorter_than_the_query_block_is_reported():
    T = 4
    inp = multi_inputs([2, 100], T)
    cache = O.build_cache(inp)
    qpe = O.rope_q_multi_bf16(inp["q_pe_raw"], np.maximum(inp["seq_lens"], T), T)
    step, out = run_multi(inp, cache, qpe, T)
    assert step.status() == L.MLA_ERR_SEQ_LEN
    # the valid sequence is still decoded correctly
    ref, _ = O.decode_multi_reference(cache, inp, qpe, T, [(1, i, h) for i in range(T) for h in range(16)])
    assert tol_ok(to_f64(out[1]).reshape(-1, 128), ref, TOL_REL, TOL_ABS)[0]


# ------------------------------------------------------------------ full-size workloads, sampled
def build_gpu_cache(inp, kv_dtype):
    """Write the whole workload's cache with the GPU append kernel."""
    w = inp["workload"]
    table, lens = inp["page_table"], inp["seq_lens"]
    npg = inp["num_pages"]
    p = L.make_params(w.B, w.H, table.shape[1], npg, kv_dtype)
    if kv_dtype == "e4m3":
        ckv = torch.full((npg, 64, 512), 0x44, dtype=torch.uint8, device="cuda")
        kpe = torch.full((npg, 64, 64), 0x44, dtype=torch.uint8, device="cuda")
        sc = torch.ones(npg, 64, dtype=torch.float32, device="cuda")
    else:
        ckv = torch.full((npg, 64, 512), 3.0, dtype=torch.bfloat16, device="cuda")
        kpe = torch.full((npg, 64, 64), 3.0, dtype=torch.bfloat16, device="cuda")
        sc = None
    for b in range(w.B):
        n = int(lens[b])
        t = np.arange(n)
        slots = (table[b, t // 64].astype(np.int64) * 64 + t % 64).astype(np.int32)
        L.mla_cache_append(p, bf16_dev(mi.kv_rows(w, b, n)), i32_dev(slots), i32_dev(t),
                           3, ckv, kpe, sc)
    return ckv, kpe, sc


def oracle_sampled(w, pairs, kv_dtype=None):
    """fp64 oracle on a compact sub-problem holding only the sampled sequences
    (the result does not depend on where pages sit in the pool).  kv_dtype
    overrides the workload's cache storage (the E4M3 workload's oracle is run
    on the decoded E4M3 cache and on the unquantised bf16 cache)."""
    seqs = sorted({b for b, _ in pairs})
    full = mi.make_inputs(w, seqs=seqs)
    lens = full["seq_lens"][seqs]
    npg = (lens + 63) // 64
    table = np.full((len(seqs), int(npg.max())), -1, np.int32)
    k = 0
    for i, n in enumerate(npg):
        table[i, :n] = np.arange(k, k + n)
        k += int(n)
    sub = {"workload": dataclasses.replace(w, B=len(seqs)), "seq_lens": lens, "page_table": table,
           "num_pages": k, "q_nope": full["q_nope"][seqs], "q_pe_raw": full["q_pe_raw"][seqs],
           "w_uk": full["w_uk"], "w_uv": full["w_uv"],
           "kv_raw": {i: full["kv_raw"][b] for i, b in enumerate(seqs)}}
    cache = O.build_cache(sub, kv_dtype or w.kv_dtype)
    qpe = O.rope_q_bf16(sub["q_pe_raw"], sub["seq_lens"])
    return O.decode_reference(cache, sub, qpe, [(seqs.index(b), h) for b, h in pairs])


def test_full_size_multi_token_sampled():
    """Two query tokens per sequence at the DeepSeek-V2 layer shape (B=32,
    H=128, L=4096): sampled (sequence, token, head) triples against the
    oracle, which computes each one by one."""
    w = mi.WORKLOADS["mtp2"]
    T = w.q_len
    inp = mi.make_inputs(w, with_kv=False)
    ckv, kpe, sc = build_gpu_cache(inp, w.kv_dtype)
    table = inp["page_table"]
    step = mla.MLADecodeStep(w.B, w.H, table.shape[1], inp["num_pages"], q_len=T)
    lens = i32_dev(inp["seq_lens"])
    tab = i32_dev(table)
    rows_table, rows_lens = step.expand_rows(tab, lens)
    p = L.make_params(w.B * T, w.H, table.shape[1], inp["num_pages"])
    qpe = torch.empty(w.B * T, w.H, 64, dtype=torch.bfloat16, device="cuda")
    L.mla_rope_q(p, bf16_dev(inp["q_pe_raw"].reshape(-1, w.H, 64)), rows_lens, qpe)
    out = step(bf16_dev(inp["q_nope"]), qpe, bf16_dev(inp["w_uk"]), bf16_dev(inp["w_uv"]), ckv, kpe, sc, tab, lens)
    torch.cuda.synchronize()
    assert step.status() == 0
    rng = np.random.default_rng(w.seed)
    triples = [(int(b), int(i), int(h)) for b in sorted(rng.choice(w.B, 3, replace=False))
               for i in range(T) for h in sorted(rng.choice(w.H, 2, replace=False))]
    seqs = sorted({b for b, _, _ in triples})
    full = mi.make_inputs(w, seqs=seqs)
    npg = (full["seq_lens"][seqs] + 63) // 64
    sub_table = np.full((len(seqs), int(npg.max())), -1, np.int32)
    k = 0
    for r_, n in enumerate(npg):
        sub_table[r_, :n] = np.arange(k, k + n)
        k += int(n)
    sub = {"workload": dataclasses.replace(w, B=len(seqs)), "seq_lens": full["seq_lens"][seqs],
           "page_table": sub_table, "num_pages": k, "q_nope": full["q_nope"][seqs],
           "q_pe_raw": full["q_pe_raw"][seqs], "w_uk": full["w_uk"], "w_uv": full["w_uv"],
           "kv_raw": {r_: full["kv_raw"][b] for r_, b in enumerate(seqs)}}
    cache = O.build_cache(sub)
    ref, _ = O.decode_multi_reference(cache, sub, O.rope_q_multi_bf16(sub["q_pe_raw"], sub["seq_lens"], T), T,
                                      [(seqs.index(b), i, h) for b, i, h in triples])
    got = np.stack([to_f64(out[b, i, h]) for b, i, h in triples])
    ok, err, bound = tol_ok(got, ref, TOL_REL, TOL_ABS)
    assert ok, (err, bound)


@pytest.mark.parametrize("name,n_seq,n_head", [("v2_layer", 3, 3), ("long_ctx", 1, 3),
                                               ("ragged", 3, 2), ("fp8_batch", 2, 2)])
def test_full_size_workloads_sampled(name, n_seq, n_head):
    w = mi.WORKLOADS[name]
    inp = mi.make_inputs(w, with_kv=False)
    ckv, kpe, sc = build_gpu_cache(inp, w.kv_dtype)
    B, H = w.B, w.H
    table = inp["page_table"]
    p = L.make_params(B, H, table.shape[1], inp["num_pages"], w.kv_dtype, w.out_dtype)
    step = mla.MLADecodeStep(B, H, table.shape[1], inp["num_pages"], w.kv_dtype, w.out_dtype, w.splits)
    lens = i32_dev(inp["seq_lens"])
    qpe = torch.empty(B, H, 64, dtype=torch.bfloat16, device="cuda")
    L.mla_rope_q(p, bf16_dev(inp["q_pe_raw"]), lens, qpe)
    out = step(bf16_dev(inp["q_nope"]), qpe, bf16_dev(inp["w_uk"]), bf16_dev(inp["w_uv"]),
               ckv, kpe, sc, i32_dev(table), lens)
    torch.cuda.synchronize()
    assert step.status() == 0
    pairs = sample_pairs(B, H, n_seq, n_head, seed=w.seed)
    ref, lse_ref = oracle_sampled(w, pairs)
    got = np.stack([to_f64(out[b, h]) for b, h in pairs])
    # bf16 cache: the oracle on the same cache.  E4M3 cache: the oracle on
    # the decoded E4M3 values at the bf16 bound (the kernel's arithmetic),
    # and on the unquantised cache at 5e-2 (the quantisation itself)
    ok, err, bound = tol_ok(got, ref, TOL_REL, TOL_ABS)
    assert ok, (name, err, bound)
    glse = np.array([float(step.lse[b, h]) for b, h in pairs])
    assert np.allclose(glse, lse_ref, atol=2e-3)
    if w.kv_dtype == "e4m3":
        ref_bf, lse_bf = oracle_sampled(w, pairs, "bf16")
        ok, err, bound = tol_ok(got, ref_bf, 5e-2)
        assert ok, (name, "unquantised", err, bound)
        assert np.allclose(glse, lse_bf, atol=2e-2)
