"""GPU parity of the 8-bit tensor-core decode: the E4M3 cache multiplied as
codes (tcgen05 kind::f8f6f4), the query and the probabilities as E4M3 terms
(MLA_KV_E4M3_MMA: two terms each; MLA_KV_E4M3_MMA1: one), against the fp64
oracle on the same seeded inputs.

Bounds:
- the E4M3 query the decode keeps in its workspace: bit-exact against the
  oracle's quantisation (the same fp32 decisions);
- two terms: the bf16 bound, max|got - ref| <= 1e-2 max|ref| + 1e-3, against
  the oracle on the decoded E4M3 cache (both for o_lat from exact inputs and
  for the whole path's output) -- two E4M3 terms carry about 8 significant
  bits, the rounding left in the query and in P is 2^-8 relative at most;
- one term and two: the FP8 bound, 5e-2 max|ref|, against the oracle on the
  unquantised bf16 cache;
- one term against the decoded E4M3 cache: the FP8 bound, 5e-2 max|ref| +
  1e-3 (one E4M3 rounding, up to 2^-4 relative, on each query value and each
  probability; measured 3.0-3.4% of max|ref| at unit-variance logits).
"""
import math

import numpy as np
import pytest
import torch

import mla_inputs as mi
import mla_latent_kv_66_b300 as mla
from mla_latent_kv_66_b300 import _lib as L
from oracle import mla_oracle as O

from helpers import bf16_dev, i32_dev, sample_pairs, tol_ok, to_f64, upload_cache

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-2, 1e-3
TOL_FP8 = 5e-2
TOL_ONE_TERM = 5e-2


def small_inputs(lens, H=16, seed=31, pages="permuted"):
    w = mi.Workload("t8", B=len(lens), H=H, L=0, ragged=(1, 2), seed=seed, pages=pages)
    inp = mi.make_inputs(w, with_kv=False)
    inp["seq_lens"] = np.asarray(lens, np.int32)
    inp["page_table"], inp["num_pages"] = mi.page_layout(w, inp["seq_lens"])
    inp["kv_raw"] = {b: mi.kv_rows(w, b, int(lens[b])) for b in range(len(lens))}
    return inp


def garbage_codes(inp):
    """Pool pages start as E4M3 NaN codes (0x7F) with NaN scales: a slot past
    a sequence's end must never reach the result."""
    npg = inp["num_pages"]
    return (np.full((npg, 64, 512), 0x7F, np.uint8), np.full((npg, 64, 64), 0x7F, np.uint8),
            np.full((npg, 64), np.nan, np.float32))


def upload_with_garbage(inp, cache8):
    gc, gk, gs = garbage_codes(inp)
    t = np.concatenate([np.arange(n) for n in inp["seq_lens"]])
    b_of = np.concatenate([np.full(n, b) for b, n in enumerate(inp["seq_lens"])])
    pg, sl = inp["page_table"][b_of, t // 64], t % 64
    gc[pg, sl], gk[pg, sl], gs[pg, sl] = cache8["ckv"][pg, sl], cache8["kpe"][pg, sl], cache8["scale"][pg, sl]
    return (torch.from_numpy(gc).cuda(), torch.from_numpy(gk).cuda(), torch.from_numpy(gs).cuda())


def run(inp, cache8, q_pe_bits, kv, num_splits, q_lat_bits=None, out_dtype="f32", garbage=True):
    w = inp["workload"]
    B, H = len(inp["seq_lens"]), w.H
    table = inp["page_table"]
    p = L.make_params(B, H, table.shape[1], inp["num_pages"], kv, out_dtype)
    G = L.mla_decode_num_splits(p, num_splits)
    ws = torch.zeros(L.mla_decode_workspace_size(p, G), dtype=torch.uint8, device="cuda")
    ckv, kpe, sc = upload_with_garbage(inp, cache8) if garbage else upload_cache(cache8)
    q_lat = torch.empty(B, H, 512, dtype=torch.bfloat16, device="cuda")
    L.mla_absorb_q(p, bf16_dev(inp["q_nope"]), bf16_dev(inp["w_uk"]), q_lat)
    q_used = bf16_dev(q_lat_bits) if q_lat_bits is not None else q_lat
    o_lat = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    L.mla_decode(p, q_used, bf16_dev(q_pe_bits), ckv, kpe, sc, i32_dev(table), i32_dev(inp["seq_lens"]), G, ws,
                 o_lat, lse)
    L.mla_split_kv_combine(p, ws, G, o_lat, lse)
    out = torch.empty(B, H, 128, dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32, device="cuda")
    L.mla_out_proj(p, o_lat, bf16_dev(inp["w_uv"]), out)
    torch.cuda.synchronize()
    qoff, soff = L.mla_workspace_query_offsets(p, G)
    codes = ws[qoff: qoff + B * H * 2 * 576].view(B, H, 2, 576).cpu().numpy()
    scale = ws[soff: soff + B * H * 4].view(torch.float32).view(B, H).cpu().numpy()
    return dict(q_lat=q_lat, o_lat=o_lat, lse=lse, out=out, status=L.mla_workspace_status(ws), codes=codes,
                scale=scale)


# ------------------------------------------------------------------ the E4M3 query, bit-exact
@pytest.mark.parametrize("kv,terms", [("e4m3_mma", 2), ("e4m3_mma1", 1)])
def test_query_codes_are_bit_exact(kv, terms):
    inp = small_inputs([130, 64, 1], H=32)
    cache8 = O.build_cache(inp, "e4m3")
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    ql = O.absorb_q(inp["q_nope"], inp["w_uk"])
    # edge rows: all zero; tiny values (subnormal codes); huge and mixed magnitudes
    ql[0, 0], qpe[0, 0] = 0.0, 0
    ql[0, 1] *= 1e-6
    ql[1, 2, ::7] *= 1e4
    qlat_bits = O.f64_to_bf16(ql)
    r = run(inp, cache8, qpe, kv, 2, q_lat_bits=qlat_bits, garbage=False)
    assert r["status"] == 0
    codes, scale = O.quantize_query_e4m3(qlat_bits, qpe, terms)
    assert np.array_equal(r["scale"], scale)
    assert np.array_equal(r["codes"][:, :, :terms], codes)
    assert r["scale"][0, 0] == 1.0 and not r["codes"][0, 0, :terms].any()


# ------------------------------------------------------------------ small problems, every output
@pytest.mark.parametrize("splits", [1, 3, 16])
def test_two_term_decode_on_exact_inputs(splits):
    """o_lat and LSE of every head against the oracle's absorbed attention on
    the decoded E4M3 cache with the dequantised two-term query; the whole
    path against the non-absorbed oracle on the decoded cache (bf16 bound)
    and on the unquantised cache (FP8 bound).  Pool slots past every
    sequence end hold NaN codes and NaN scales."""
    inp = small_inputs([700, 64, 1, 130, 65, 2000])
    cache8 = O.build_cache(inp, "e4m3")
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    qlat_bits = O.f64_to_bf16(O.absorb_q(inp["q_nope"], inp["w_uk"]))
    r = run(inp, cache8, qpe, "e4m3_mma", splits, q_lat_bits=qlat_bits)
    assert r["status"] == 0
    codes, scale = O.quantize_query_e4m3(qlat_bits, qpe, 2)
    qdl, qdp = O.dequantize_query(codes, scale)
    got = to_f64(r["o_lat"])
    assert np.all(np.isfinite(got))
    for b in range(len(inp["seq_lens"])):
        c, kp = O.gather_sequence(cache8, inp["page_table"], b, int(inp["seq_lens"][b]))
        for h in range(16):
            o_ref, lse_ref = O.latent_attention(c, kp, qdl[b, h], qdp[b, h])
            ok, err, bound = tol_ok(got[b, h], o_ref, TOL_REL, TOL_ABS)
            assert ok, (splits, b, h, err, bound)
            assert abs(float(r["lse"][b, h]) - lse_ref) < 2e-3, (b, h)
    r = run(inp, cache8, qpe, "e4m3_mma", splits)
    got = to_f64(r["out"]).reshape(-1, 128)
    ref8, _ = O.decode_reference(cache8, inp, qpe)
    ok, err, bound = tol_ok(got, ref8, TOL_REL, TOL_ABS)
    assert ok, ("decoded", err, bound)
    ref, _ = O.decode_reference(O.build_cache(inp), inp, qpe)
    ok, err, bound = tol_ok(got, ref, TOL_FP8)
    assert ok, ("unquantised", err, bound)


def test_one_term_decode():
    inp = small_inputs([700, 64, 1, 130, 65, 2000])
    cache8 = O.build_cache(inp, "e4m3")
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    r = run(inp, cache8, qpe, "e4m3_mma1", 5)
    assert r["status"] == 0
    got = to_f64(r["out"]).reshape(-1, 128)
    ref8, _ = O.decode_reference(cache8, inp, qpe)
    ok, err, bound = tol_ok(got, ref8, TOL_ONE_TERM, TOL_ABS)
    assert ok, ("decoded", err, bound)
    ref, _ = O.decode_reference(O.build_cache(inp), inp, qpe)
    ok, err, bound = tol_ok(got, ref, TOL_FP8)
    assert ok, ("unquantised", err, bound)


@pytest.mark.parametrize("gain", [4, 16])
def test_two_term_sharp_softmax_at_large_logits(gain):
    """The query scaled by 4 or 16: peaked softmax rows, log2-domain scores
    past 6 x gain.  o_lat of every head against the absorbed attention with
    the dequantised query on the decoded cache, at the bf16 bound."""
    inp = small_inputs([700, 64, 1, 4096], H=128, seed=33)
    inp["q_nope"] = O.f64_to_bf16(float(gain) * O.bf16_to_f64(inp["q_nope"]))
    inp["q_pe_raw"] = O.f64_to_bf16(float(gain) * O.bf16_to_f64(inp["q_pe_raw"]))
    cache8 = O.build_cache(inp, "e4m3")
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    qlat_bits = O.f64_to_bf16(O.absorb_q(inp["q_nope"], inp["w_uk"]))
    r = run(inp, cache8, qpe, "e4m3_mma", 7, q_lat_bits=qlat_bits)
    assert r["status"] == 0
    qdl, qdp = O.dequantize_query(*O.quantize_query_e4m3(qlat_bits, qpe, 2))
    got = to_f64(r["o_lat"])
    peak = 0.0
    for b in range(len(inp["seq_lens"])):
        c, kp = O.gather_sequence(cache8, inp["page_table"], b, int(inp["seq_lens"][b]))
        peak = max(peak, np.max(np.abs(c @ qdl[b].T + kp @ qdp[b].T)) / math.sqrt(192.0) * math.log2(math.e))
        for h in range(128):
            o_ref, lse_ref = O.latent_attention(c, kp, qdl[b, h], qdp[b, h])
            ok, err, bound = tol_ok(got[b, h], o_ref, TOL_REL, TOL_ABS)
            assert ok, (gain, b, h, err, bound)
            assert abs(float(r["lse"][b, h]) - lse_ref) < 2e-3 * max(1.0, abs(lse_ref)), (b, h)
    assert peak > 6 * gain


def test_two_query_tokens_on_the_8bit_tensor_cores():
    """Several query tokens per sequence (causal) with the E4M3 cache on the
    8-bit tensor cores, through the decode step object: every output against
    the oracle on the decoded E4M3 cache (bf16 bound)."""
    T, lens = 2, [2, 70, 300, 129]
    w = mi.Workload("m8", B=len(lens), H=16, L=0, ragged=(1, 2), seed=37, pages="permuted", q_len=T)
    inp = mi.make_inputs(w, with_kv=False)
    inp["seq_lens"] = np.asarray(lens, np.int32)
    inp["page_table"], inp["num_pages"] = mi.page_layout(w, inp["seq_lens"])
    inp["kv_raw"] = {b: mi.kv_rows(w, b, int(lens[b])) for b in range(len(lens))}
    cache8 = O.build_cache(inp, "e4m3")
    qpe = O.rope_q_multi_bf16(inp["q_pe_raw"], inp["seq_lens"], T)
    step = mla.MLADecodeStep(len(lens), 16, inp["page_table"].shape[1], inp["num_pages"], "e4m3_mma", q_len=T)
    ckv, kpe, sc = upload_with_garbage(inp, cache8)
    out = step(bf16_dev(inp["q_nope"]), bf16_dev(qpe), bf16_dev(inp["w_uk"]), bf16_dev(inp["w_uv"]), ckv, kpe, sc,
               i32_dev(inp["page_table"]), i32_dev(inp["seq_lens"]))
    torch.cuda.synchronize()
    assert step.status() == 0
    ref, _ = O.decode_multi_reference(cache8, inp, qpe, T)
    ok, err, bound = tol_ok(to_f64(out).reshape(-1, 128), ref, TOL_REL, TOL_ABS)
    assert ok, (err, bound)


# ------------------------------------------------------------------ full size, sampled
def test_full_size_fp8_batch_on_the_8bit_tensor_cores():
    """B=128, H=128, L=8192, E4M3 cache written by the GPU append kernel,
    through the decode step object (the bench's path): sampled heads against
    the oracle on the decoded E4M3 cache (bf16 bound) and on the unquantised
    cache (FP8 bound)."""
    import dataclasses
    w = dataclasses.replace(mi.WORKLOADS["fp8_batch"], kv_dtype="e4m3_mma")
    inp = mi.make_inputs(w, with_kv=False)
    table, lens_np = inp["page_table"], inp["seq_lens"]
    npg = inp["num_pages"]
    p = L.make_params(w.B, w.H, table.shape[1], npg, w.kv_dtype, w.out_dtype)
    ckv = torch.full((npg, 64, 512), 0x7F, dtype=torch.uint8, device="cuda")
    kpe = torch.full((npg, 64, 64), 0x7F, dtype=torch.uint8, device="cuda")
    sc = torch.ones(npg, 64, dtype=torch.float32, device="cuda")
    for b in range(w.B):
        n = int(lens_np[b])
        t = np.arange(n)
        slots = (table[b, t // 64].astype(np.int64) * 64 + t % 64).astype(np.int32)
        L.mla_cache_append(p, bf16_dev(mi.kv_rows(w, b, n)), i32_dev(slots), i32_dev(t), 3, ckv, kpe, sc)
    step = mla.MLADecodeStep(w.B, w.H, table.shape[1], npg, w.kv_dtype, w.out_dtype, w.splits)
    lens = i32_dev(lens_np)
    qpe = torch.empty(w.B, w.H, 64, dtype=torch.bfloat16, device="cuda")
    L.mla_rope_q(p, bf16_dev(inp["q_pe_raw"]), lens, qpe)
    out = step(bf16_dev(inp["q_nope"]), qpe, bf16_dev(inp["w_uk"]), bf16_dev(inp["w_uv"]), ckv, kpe, sc,
               i32_dev(table), lens)
    torch.cuda.synchronize()
    assert step.status() == 0
    pairs = sample_pairs(w.B, w.H, 2, 3, seed=w.seed)
    seqs = sorted({b for b, _ in pairs})
    full = mi.make_inputs(w, seqs=seqs)
    sl = full["seq_lens"][seqs]
    npg_s = (sl + 63) // 64
    st = np.full((len(seqs), int(npg_s.max())), -1, np.int32)
    k = 0
    for i, n in enumerate(npg_s):
        st[i, :n] = np.arange(k, k + n)
        k += int(n)
    sub = {"workload": dataclasses.replace(w, B=len(seqs)), "seq_lens": sl, "page_table": st, "num_pages": k,
           "q_nope": full["q_nope"][seqs], "q_pe_raw": full["q_pe_raw"][seqs], "w_uk": full["w_uk"],
           "w_uv": full["w_uv"], "kv_raw": {i: full["kv_raw"][b] for i, b in enumerate(seqs)}}
    sub_pairs = [(seqs.index(b), h) for b, h in pairs]
    qpe_s = O.rope_q_bf16(sub["q_pe_raw"], sub["seq_lens"])
    got = np.stack([to_f64(out[b, h]) for b, h in pairs])
    ref8, _ = O.decode_reference(O.build_cache(sub, "e4m3"), sub, qpe_s, sub_pairs)
    ok, err, bound = tol_ok(got, ref8, TOL_REL, TOL_ABS)
    assert ok, ("decoded", err, bound)
    ref, _ = O.decode_reference(O.build_cache(sub), sub, qpe_s, sub_pairs)
    ok, err, bound = tol_ok(got, ref, TOL_FP8)
    assert ok, ("unquantised", err, bound)
