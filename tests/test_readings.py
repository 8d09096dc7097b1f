"""Measured consequences of two storage choices of the boundary, on the
oracle alone (no GPU): o_lat (mla_decode / mla_split_kv_combine output) and
the split-KV partial results are bf16, where an fp32 latent would be the
plainest reading of the pages' value path.  Both cost one bf16 rounding
(2^-9 relative) of a normalised latent; after the W_UV projection the
change of the output stays below 2^-8 of max|out|, well inside the 1e-2
bound of the bf16 path, at unit-variance logits and at sharp softmax rows
(query scaled by 4 and 16)."""
import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as O


def _inputs(gain, lens=(700, 130, 4096), H=16, seed=21):
    w = mi.Workload("r", B=len(lens), H=H, L=0, ragged=(1, 2), seed=seed, pages="permuted")
    inp = mi.make_inputs(w, with_kv=False)
    inp["seq_lens"] = np.asarray(lens, np.int32)
    inp["page_table"], inp["num_pages"] = mi.page_layout(w, inp["seq_lens"])
    inp["kv_raw"] = {b: mi.kv_rows(w, b, int(lens[b])) for b in range(len(lens))}
    inp["q_nope"] = O.f64_to_bf16(gain * O.bf16_to_f64(inp["q_nope"]))
    inp["q_pe_raw"] = O.f64_to_bf16(gain * O.bf16_to_f64(inp["q_pe_raw"]))
    return inp


def bf16(x):
    return O.bf16_to_f64(O.f64_to_bf16(x))


@pytest.mark.parametrize("gain", [1, 4, 16])
def test_bf16_latent_and_bf16_partials_move_the_output_by_less_than_2_pow_minus_8(gain):
    inp = _inputs(gain)
    cache = O.build_cache(inp)
    qpe = O.rope_q_bf16(inp["q_pe_raw"], inp["seq_lens"])
    out, olat, _ = O.decode_absorbed(cache, inp, qpe)
    ql = O.absorb_q(inp["q_nope"], inp["w_uk"])
    qp = O.bf16_to_f64(qpe)
    wuv = O.bf16_to_f64(inp["w_uv"])
    H = inp["workload"].H
    got_lat, got_split = [], []
    for b, n in enumerate(inp["seq_lens"]):
        n = int(n)
        cuts = [0, n // 3, (2 * n) // 3, n]
        for h in range(H):
            i = b * H + h
            got_lat.append(O.out_proj(bf16(olat[i]), wuv[h]))
            # three KV splits: each partial normalised and stored in bf16, merged by LSE
            parts = [O.latent_attention_range(cache, inp["page_table"], b, t0, t1, ql[b, h], qp[b, h])
                     for t0, t1 in zip(cuts[:-1], cuts[1:]) if t1 > t0]
            lse = np.array([p[1] for p in parts])
            wt = np.exp(lse - lse.max())
            merged = sum(wk * bf16(p[0]) for wk, p in zip(wt, parts)) / wt.sum()
            got_split.append(O.out_proj(bf16(merged), wuv[h]))
    scale = np.max(np.abs(out))
    assert np.max(np.abs(np.stack(got_lat) - out)) <= 2.0 ** -8 * scale
    assert np.max(np.abs(np.stack(got_split) - out)) <= 2.0 ** -8 * scale
