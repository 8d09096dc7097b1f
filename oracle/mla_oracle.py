"""fp64 CPU oracle for MLA decode over a compressed latent KV cache.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
the benchmark's CPU-baseline leg may import this module.  It shares no code
with the CUDA path: it reads the seeded inputs from ``mla_inputs`` (which
holds no arithmetic of the method) and implements every step itself, in
float64 numpy, on the exact values of the bf16 / E4M3 inputs.

Sources (page titles and sections):
  [P3] mtrt.cn, "DeepSeek-Coder-V2 的 MLA 多头潜在注意力深度解析：512维潜空间
       压缩 KV 缓存": the two-component cache (512-d latent + 64-d k_pe shared
       by all heads), RMSNorm on the latent, kv_b_proj up-projection into
       128-d k_nope and 128-d value per head, RoPE on the 64-d part only,
       the forward-flow list ("源码里的压缩全流程") and the cache-size table.
  [P4] aiboss88.com wiki, "什么是多头潜在注意力", section "工作机制":
       compress -> cache the latent -> up-project back to K and V, the
       decode step reads only the compressed latent.
Readings where the pages are silent (RoPE variant, query position, RMSNorm
gain/eps, FP8 scale) are stated on each function.

Parity status: every function below is pinned by ``tests/test_oracle_pins.py``
against closed forms, invariants, brute force or an independent library
routine; none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

D_LATENT, D_ROPE, D_NOPE, D_V, PAGE = 512, 64, 128, 128, 64
D_QK = D_NOPE + D_ROPE  # 192: per-head query/key width [P3, model config: 128 heads of 192]
ROPE_THETA = 10000.0


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (upper half of an IEEE binary32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values to bfloat16, nearest with ties to even, in one step.

    bfloat16 keeps 7 fraction bits of binary64's 52, so 45 bits are rounded
    away.  Only normal numbers of the binary32 exponent range (and zero) occur
    in this method's data; anything else is rejected.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    a = np.abs(x)
    bad = (a != 0) & ((a < 2.0 ** -126) | ~np.isfinite(a) | (a >= 2.0 ** 128))
    if bad.any():
        raise ValueError("value outside the bf16 normal range")
    b = x.view(np.uint64)
    keep_lsb = (b >> np.uint64(45)) & np.uint64(1)
    r = (b + np.uint64((1 << 44) - 1) + keep_lsb) & ~np.uint64((1 << 45) - 1)
    y = r.view(np.float64).astype(np.float32)  # exact: 8 significant bits
    return (y.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _e4m3_positive_values() -> np.ndarray:
    """Values of the non-negative finite E4M3 codes 0x00..0x7E (OCP FP8 E4M3:
    4 exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is
    NaN).  Exponent field 0 holds the subnormals m/8 * 2^-6."""
    v = np.empty(127, dtype=np.float64)
    for code in range(127):
        e, m = code >> 3, code & 7
        v[code] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return v


E4M3_POS = _e4m3_positive_values()
E4M3_MAX = 448.0


def e4m3_to_f64(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    mag = c & 0x7F
    out = np.where(mag == 0x7F, np.nan, E4M3_POS[np.minimum(mag, 126)])
    return np.where(c & 0x80, -out, out)


def f32_to_e4m3(x) -> np.ndarray:
    """Encode float32 values as E4M3: nearest representable value, ties to the
    even code, magnitudes above 448 saturate to 448 (the "satfinite" rule),
    NaN to 0x7F."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    i = np.searchsorted(E4M3_POS, np.minimum(a, E4M3_MAX), side="right") - 1
    i = np.clip(i, 0, 126)
    j = np.minimum(i + 1, 126)
    lo, hi = E4M3_POS[i], E4M3_POS[j]
    d_lo, d_hi = a - lo, hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (i % 2 == 1))
    code = np.where(pick_hi, j, i)
    code = np.where(a >= E4M3_MAX, 126, code)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


# --------------------------------------------------------------------------
# cache write: RMSNorm on the latent, RoPE on the 64-d key part
# --------------------------------------------------------------------------
def rmsnorm(x) -> np.ndarray:
    """RMSNorm of each row [P3, section "MLA 的两个核心部件": the 512-d latent is
    RMS-normalised before it is cached].
    Reading: gain 1 and eps 0 (the page gives neither): x / sqrt(mean(x^2))."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True))


def rope(x, pos) -> np.ndarray:
    """Rotary position embedding of the 64-d part [P3, section "MLA 的两个核心部件":
    position encoding acts only on the 64-d q_pe / k_pe].  Reading (the pages do not fix the variant): half-split
    pairing, dimension i with i+32, angle pos * theta^(-i/32), theta = 10000,
    rotating each pair counter-clockwise:
        x'_i      = x_i cos(a) - x_{i+32} sin(a)
        x'_{i+32} = x_{i+32} cos(a) + x_i sin(a)
    x: [..., 64]; pos: broadcastable to x[..., 0]."""
    x = np.asarray(x, dtype=np.float64)
    half = D_ROPE // 2
    inv_freq = ROPE_THETA ** (-np.arange(half, dtype=np.float64) / half)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def cache_rows_bf16(kv_raw_bits, positions) -> np.ndarray:
    """Stored bf16 cache rows [n, 576] for raw down-projection rows.

    [P3, forward flow] the down-projection output is split into the 512-d
    latent and the 64-d k_pe; the latent is RMS-normalised, k_pe is rotated
    at its token position, and both are written to the cache in bf16."""
    raw = bf16_to_f64(kv_raw_bits)
    c = rmsnorm(raw[:, :D_LATENT])
    k = rope(raw[:, D_LATENT:], positions)
    return np.concatenate([f64_to_bf16(c), f64_to_bf16(k)], axis=1)


def quantize_rows_e4m3(rows_bf16_bits):
    """FP8 cache rows: one fp32 scale per token over all 576 values.

    Reading of "one fp32 scale per token (scale = rowmax/448)": rowmax is
    max |v| over the token's bf16 cache row (latent and rotated k_pe); the
    scale is rowmax / 448 rounded to fp32 (1 for an all-zero row); each value
    is encoded as E4M3(fp32(v) / scale) with the quotient rounded to fp32.
    These are the decisions that fix each code, taken in fp32 as a kernel
    takes them."""
    v = bf16_to_f64(rows_bf16_bits).astype(np.float32)
    amax = np.max(np.abs(v), axis=1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    scale = np.where(amax == 0, np.float32(1.0), scale).astype(np.float32)
    q = (v / scale[:, None]).astype(np.float32)
    return f32_to_e4m3(q), scale


def quantize_query_e4m3(q_lat_bits, q_pe_bits, terms=2):
    """Query of the 8-bit tensor-core decode: each (b, h) row of its 576
    values (the 512 latent ones, then the 64 rotated RoPE ones) as E4M3
    codes under one fp32 scale.

    [P1, hotdry "DeepSeek-V3.2-Exp 中多头潜在注意力的优化", deployment
    paragraph: FP8 quantisation when serving MLA.]  The page names no
    format; the reading mirrors the cache's per-token rule:
        scale = fp32(max |v|) / 448 in fp32 (1 for an all-zero row)
        y     = fp32(v) / scale in fp32
        hi    = E4M3(y)
        lo    = E4M3(fp32(y - value(hi)))      (terms == 2 only)
    so that v ~ scale * (value(hi) + value(lo)).  y - value(hi) is exact in
    fp32 (hi is y rounded to 4 significant bits).  All decisions are taken in
    fp32, as a kernel takes them.
    Returns codes uint8 [B, H, terms, 576] and scale float32 [B, H]."""
    v = np.concatenate([bf16_to_f64(q_lat_bits), bf16_to_f64(q_pe_bits)], axis=-1).astype(np.float32)
    amax = np.max(np.abs(v), axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    scale = np.where(amax == 0, np.float32(1.0), scale).astype(np.float32)
    y = (v / scale[..., None]).astype(np.float32)
    hi = f32_to_e4m3(y)
    codes = [hi]
    if terms == 2:
        r = (y - e4m3_to_f64(hi).astype(np.float32)).astype(np.float32)
        codes.append(f32_to_e4m3(r))
    return np.stack(codes, axis=-2), scale


def dequantize_query(codes, scale):
    """fp64 value of an E4M3 query (see quantize_query_e4m3): q_lat [..., 512]
    and q_pe [..., 64] = scale * sum of the terms' values."""
    v = np.sum(e4m3_to_f64(codes), axis=-2) * np.asarray(scale, dtype=np.float64)[..., None]
    return v[..., :D_LATENT], v[..., D_LATENT:]


def rope_q_bf16(q_pe_raw_bits, seq_lens) -> np.ndarray:
    """Rotated query key-part [B,H,64] in bf16.  Reading: the decoding token is
    the last cached position, p_q = seq_len - 1 (its own row is in the cache)."""
    q = bf16_to_f64(q_pe_raw_bits)
    pos = (np.asarray(seq_lens, dtype=np.int64) - 1)[:, None]
    return f64_to_bf16(rope(q, pos))


def build_cache(inp: dict, kv_dtype: str = "bf16", garbage=None) -> dict:
    """Write every sequence's rows into the paged pool through the page table
    (slot page_table[b][t // 64] * 64 + t % 64).  ``garbage``: optional
    (ckv_bits, kpe_bits) filler for slots that hold no token."""
    n_pages = int(inp["num_pages"])
    if garbage is None:
        ckv = np.zeros((n_pages, PAGE, D_LATENT), np.uint16)
        kpe = np.zeros((n_pages, PAGE, D_ROPE), np.uint16)
    else:
        ckv, kpe = (np.array(g, dtype=np.uint16, copy=True) for g in garbage)
    table, lens = inp["page_table"], inp["seq_lens"]
    for b, raw in inp["kv_raw"].items():
        n = int(lens[b])
        rows = cache_rows_bf16(raw, np.arange(n))
        t = np.arange(n)
        pg, sl = table[b, t // PAGE], t % PAGE
        ckv[pg, sl] = rows[:, :D_LATENT]
        kpe[pg, sl] = rows[:, D_LATENT:]
    out = {"kv_dtype": kv_dtype, "ckv": ckv, "kpe": kpe, "scale": None}
    if kv_dtype == "e4m3":
        flat = np.concatenate([ckv.reshape(-1, D_LATENT), kpe.reshape(-1, D_ROPE)], axis=1)
        codes, scale = quantize_rows_e4m3(flat)
        out["ckv"] = codes[:, :D_LATENT].reshape(n_pages, PAGE, D_LATENT)
        out["kpe"] = codes[:, D_LATENT:].reshape(n_pages, PAGE, D_ROPE)
        out["scale"] = scale.reshape(n_pages, PAGE)
    return out


def cache_values(cache: dict, pages, slots):
    """Decoded fp64 (latent [n,512], k_pe [n,64]) of the given cache slots."""
    if cache["kv_dtype"] == "e4m3":
        sc = cache["scale"][pages, slots].astype(np.float64)[:, None]
        return e4m3_to_f64(cache["ckv"][pages, slots]) * sc, e4m3_to_f64(cache["kpe"][pages, slots]) * sc
    return bf16_to_f64(cache["ckv"][pages, slots]), bf16_to_f64(cache["kpe"][pages, slots])


def gather_sequence(cache, page_table, b, n, t0=0):
    t = np.arange(t0, n)
    return cache_values(cache, page_table[b, t // PAGE], t % PAGE)


# --------------------------------------------------------------------------
# attention: the non-absorbed definition and the absorbed form
# --------------------------------------------------------------------------
def softmax(s):
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s)
    e = np.exp(s - m)
    return e / np.sum(e), m + math.log(np.sum(e))


def decode_head(c, k_pe, q_nope, q_pe, w_uk_h, w_uv_h):
    """Non-absorbed decode of one head over one sequence's cache, following
    [P3, forward flow]: up-project the cached latent into this head's key and
    value (kv_b_proj), join the no-position key part with the shared rotated
    k_pe, score against the query, softmax, weight the values.

    c [n,512], k_pe [n,64] (rotated), q_nope [128], q_pe [64] (rotated),
    w_uk_h / w_uv_h [128,512].  Returns (out [128], lse, p [n])."""
    k_nope = c @ w_uk_h.T                     # [n,128]  K_h = W_UK,h c_t
    v = c @ w_uv_h.T                          # [n,128]  V_h = W_UV,h c_t
    K = np.concatenate([k_nope, k_pe], axis=1)  # [n,192] shared k_pe for all heads
    Q = np.concatenate([q_nope, q_pe])          # [192]
    s = (K @ Q) / math.sqrt(D_QK)
    p, lse = softmax(s)
    return p @ v, lse, p


def decode_reference(cache, inp, q_pe_rot_bits, pairs=None):
    """Output [len(pairs), 128] (and lse) of the non-absorbed decode for the
    given (b, h) pairs (all pairs when None)."""
    lens, table = inp["seq_lens"], inp["page_table"]
    w = inp["workload"]
    if pairs is None:
        pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    qn, qp = bf16_to_f64(inp["q_nope"]), bf16_to_f64(q_pe_rot_bits)
    wuk, wuv = inp["w_uk"], inp["w_uv"]
    out = np.empty((len(pairs), D_V))
    lse = np.empty(len(pairs))
    seq_cache = {}
    for i, (b, h) in enumerate(pairs):
        if b not in seq_cache:
            seq_cache = {b: gather_sequence(cache, table, b, int(lens[b]))}
        c, kp = seq_cache[b]
        out[i], lse[i], _ = decode_head(c, kp, qn[b, h], qp[b, h],
                                        bf16_to_f64(wuk[h]), bf16_to_f64(wuv[h]))
    return out, lse


def absorb_q(q_nope_bits, w_uk_bits) -> np.ndarray:
    """q_lat[b,h] = W_UK,h^T q_nope[b,h]: the query carried into latent space,
    so that q_nope . (W_UK,h c) = (W_UK,h^T q_nope) . c.  Exact by the
    linearity of kv_b_proj [P3]."""
    qn, w = bf16_to_f64(q_nope_bits), bf16_to_f64(w_uk_bits)
    return np.einsum("bhn,hnk->bhk", qn, w)


def latent_attention(c, k_pe, q_lat, q_pe):
    """Absorbed attention of one head: scores against the 576-d cache row,
    softmax, weighted sum of latents.  Returns (o_lat [512], lse)."""
    s = (c @ q_lat + k_pe @ q_pe) / math.sqrt(D_QK)
    p, lse = softmax(s)
    return p @ c, lse


def out_proj(o_lat, w_uv_h):
    """out = W_UV,h o_lat: the value up-projection applied after attention."""
    return w_uv_h @ o_lat


def decode_absorbed(cache, inp, q_pe_rot_bits, pairs=None):
    """Absorbed fp64 form, used to check the non-absorbed one and to give
    latent intermediates.  Returns (out, o_lat, lse) for the pairs."""
    lens, table, w = inp["seq_lens"], inp["page_table"], inp["workload"]
    if pairs is None:
        pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    qlat = absorb_q(inp["q_nope"], inp["w_uk"])
    qp = bf16_to_f64(q_pe_rot_bits)
    out = np.empty((len(pairs), D_V))
    olat = np.empty((len(pairs), D_LATENT))
    lse = np.empty(len(pairs))
    seq_cache = {}
    for i, (b, h) in enumerate(pairs):
        if b not in seq_cache:
            seq_cache = {b: gather_sequence(cache, table, b, int(lens[b]))}
        c, kp = seq_cache[b]
        olat[i], lse[i] = latent_attention(c, kp, qlat[b, h], qp[b, h])
        out[i] = out_proj(olat[i], bf16_to_f64(inp["w_uv"][h]))
    return out, olat, lse


def latent_attention_range(cache, page_table, b, t0, t1, q_lat, q_pe):
    """Absorbed attention over cached tokens [t0, t1) only: the partial result
    (normalised o_lat and its log-sum-exp) of one KV split."""
    t = np.arange(t0, t1)
    c, kp = cache_values(cache, page_table[b, t // PAGE], t % PAGE)
    return latent_attention(c, kp, q_lat, q_pe)


# --------------------------------------------------------------------------
# several query tokens per sequence (speculative / multi-token decode)
# --------------------------------------------------------------------------
def rope_q_multi_bf16(q_pe_raw_bits, seq_lens, q_len) -> np.ndarray:
    """Rotated key-part of q_len query tokens per sequence, [B,T,H,64] bf16.
    Reading: the T newest tokens of a sequence of n cached tokens are the
    queries, token i at position n - T + i (its own row is in the cache)."""
    q = bf16_to_f64(q_pe_raw_bits)
    pos = (np.asarray(seq_lens, dtype=np.int64)[:, None] - q_len + np.arange(q_len)[None, :])[:, :, None]
    return f64_to_bf16(rope(q, pos))


def decode_multi_reference(cache, inp, q_pe_rot_bits, q_len, pairs=None):
    """Non-absorbed decode of q_len query tokens per sequence with a causal
    mask [P3, forward flow, applied to every new token]: query token i of
    sequence b (position n - T + i) attends to cache tokens 0..n - T + i.
    inp["q_nope"] is [B,T,H,128]; q_pe_rot_bits [B,T,H,64].  pairs: list of
    (b, i, h) (all when None).  Returns (out [len(pairs),128], lse)."""
    lens, table, w = inp["seq_lens"], inp["page_table"], inp["workload"]
    if pairs is None:
        pairs = [(b, i, h) for b in range(len(lens)) for i in range(q_len) for h in range(w.H)]
    qn, qp = bf16_to_f64(inp["q_nope"]), bf16_to_f64(q_pe_rot_bits)
    out = np.empty((len(pairs), D_V))
    lse = np.empty(len(pairs))
    seq_cache = {}
    for k, (b, i, h) in enumerate(pairs):
        if b not in seq_cache:
            seq_cache = {b: gather_sequence(cache, table, b, int(lens[b]))}
        c, kp = seq_cache[b]
        visible = int(lens[b]) - q_len + i + 1
        out[k], lse[k], _ = decode_head(c[:visible], kp[:visible], qn[b, i, h], qp[b, i, h],
                                        bf16_to_f64(inp["w_uk"][h]), bf16_to_f64(inp["w_uv"][h]))
    return out, lse


# --------------------------------------------------------------------------
# cache accounting [P3, cache-size table "每层每 token 缓存"]
# --------------------------------------------------------------------------
def cache_accounting(heads=128, d_k=128, d_v=128, layers=60, tokens=131072, bytes_per=2):
    mha = heads * (d_k + d_v)
    mla = D_LATENT + D_ROPE
    return {
        "mha_values_per_token_layer": mha,
        "mla_values_per_token_layer": mla,
        "mha_total_bytes": mha * layers * tokens * bytes_per,
        "mla_total_bytes": mla * layers * tokens * bytes_per,
        "ratio": mha / mla,
    }
