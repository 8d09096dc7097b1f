"""Seeded synthetic inputs for MLA latent-cache decode.

This module is shared by the fp64 oracle (``oracle/``) and by the CUDA path's
tests and benchmark.  It draws random numbers, rounds them to the storage
dtype and lays out the paged cache bookkeeping (sequence lengths, page
tables).  It holds none of the method's arithmetic: no RMSNorm, no RoPE, no
FP8 quantisation, no attention.  Each side applies those steps itself.

Shapes follow the DeepSeek-V2 / DeepSeek-Coder-V2 MLA dimensions printed on
the mtrt.cn page "DeepSeek-Coder-V2 的 MLA ... 512维潜空间" (config section:
kv_lora_rank 512, qk_rope_head_dim 64, 128 heads of 128 nope + 64 rope, value
head 128).

Draws (one numpy PCG64 stream per tensor, keyed by the workload seed):
  q_nope   [B,H,128]  N(0,1)          -> bf16   ([B,T,H,128] for T query tokens)
  q_pe_raw [B,H,64]   N(0,1) pre-RoPE -> bf16   ([B,T,H,64])
  w_uk     [H,128,512] N(0,1/512)     -> bf16  (head, nope row, latent)
  w_uv     [H,128,512] N(0,1/512)     -> bf16  (head, value row, latent)
  kv_raw   [T,576]    N(0,1)          -> bf16  one row per cached token, the
           output of the KV down-projection before normalisation: 512 latent
           values then 64 pre-RoPE k_pe values.  Rows are in logical order
           (sequence 0 tokens 0..L0-1, then sequence 1, ...); each sequence
           has its own stream so a subset of sequences can be regenerated.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

D_LATENT = 512   # kv_lora_rank
D_ROPE = 64      # qk_rope_head_dim
D_NOPE = 128     # qk_nope_head_dim
D_V = 128        # v_head_dim
D_ROW = D_LATENT + D_ROPE  # 576 cached values per token per layer
PAGE = 64        # tokens per cache page

# stream ids (second word of the numpy seed sequence)
_S_QNOPE, _S_QPE, _S_WUK, _S_WUV, _S_LENS, _S_PERM, _S_KV, _S_POOL = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload (a batch of sequences, one layer)."""
    name: str
    B: int
    H: int
    seed: int
    L: int = 0                   # fixed length for every sequence (0 = ragged)
    ragged: tuple = ()           # (lo, hi) for log-uniform lengths
    pages: str = "contiguous"    # contiguous | permuted | pool
    kv_dtype: str = "bf16"       # bf16 | e4m3 | e4m3_mma | e4m3_mma1 (the last three: one cache format)
    out_dtype: str = "f32"       # f32 | bf16
    splits: int = 0              # KV partitions to request (0 = automatic)
    q_len: int = 1               # query tokens per sequence (the newest positions)

    @property
    def tokens_hint(self) -> int:
        return self.B * self.L if self.L else -1


WORKLOADS = {
    "tiny": Workload("tiny", B=1, H=16, L=512, seed=0),
    "v2_layer": Workload("v2_layer", B=32, H=128, L=4096, seed=1),
    "long_ctx": Workload("long_ctx", B=1, H=128, L=131072, seed=2,
                         pages="permuted", splits=64),
    "ragged": Workload("ragged", B=64, H=128, ragged=(1024, 32768), seed=3,
                       pages="pool"),
    "fp8_batch": Workload("fp8_batch", B=128, H=128, L=8192, seed=4,
                          kv_dtype="e4m3", out_dtype="bf16"),
    # the same E4M3 cache multiplied as codes on the 8-bit tensor cores
    "fp8_mma": Workload("fp8_mma", B=128, H=128, L=8192, seed=4,
                        kv_dtype="e4m3_mma", out_dtype="bf16"),
    # two query tokens per sequence (speculative / multi-token decode)
    "mtp2": Workload("mtp2", B=32, H=128, L=4096, seed=5, q_len=2),
}


def _rng(seed: int, stream: int, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream, sub]))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x)


def seq_lens_for(w: Workload) -> np.ndarray:
    if w.L:
        return np.full(w.B, w.L, dtype=np.int32)
    lo, hi = w.ragged
    u = _rng(w.seed, _S_LENS).uniform(math.log(lo), math.log(hi), size=w.B)
    return np.clip(np.rint(np.exp(u)), lo, hi).astype(np.int32)


def page_layout(w: Workload, seq_lens: np.ndarray):
    """Return (page_table [B, max_pages] int32 with -1 for unused, num_pages)."""
    n_pages = (seq_lens.astype(np.int64) + PAGE - 1) // PAGE
    max_pages = int(n_pages.max())
    B = len(seq_lens)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    if w.pages == "contiguous":
        for b in range(B):
            table[b, : n_pages[b]] = b * max_pages + np.arange(n_pages[b])
        return table, B * max_pages
    total = int(n_pages.sum())
    perm = _rng(w.seed, _S_PERM).permutation(total).astype(np.int32)
    k = 0
    for b in range(B):
        table[b, : n_pages[b]] = perm[k: k + n_pages[b]]
        k += int(n_pages[b])
    return table, total


def kv_rows(w: Workload, b: int, n: int) -> np.ndarray:
    """bf16 bits [n, 576] of the raw KV rows of sequence b (tokens 0..n-1)."""
    return _normal_bf16(_rng(w.seed, _S_KV, b), (n, D_ROW))


def _qshape(w: Workload, d: int):
    return (w.B, w.H, d) if w.q_len == 1 else (w.B, w.q_len, w.H, d)


def make_inputs(w: Workload, seqs=None, with_kv: bool = True) -> dict:
    """Draw every input of workload ``w``.

    seqs: optional list of sequence indices whose raw KV rows are drawn (the
    others are left out, for CPU-side sampling of large workloads).
    """
    lens = seq_lens_for(w)
    table, num_pages = page_layout(w, lens)
    out = {
        "workload": w,
        "seq_lens": lens,
        "page_table": table,
        "num_pages": num_pages,
        "q_nope": _normal_bf16(_rng(w.seed, _S_QNOPE), _qshape(w, D_NOPE)),
        "q_pe_raw": _normal_bf16(_rng(w.seed, _S_QPE), _qshape(w, D_ROPE)),
        "w_uk": _normal_bf16(_rng(w.seed, _S_WUK), (w.H, D_NOPE, D_LATENT), 1.0 / math.sqrt(512.0)),
        "w_uv": _normal_bf16(_rng(w.seed, _S_WUV), (w.H, D_V, D_LATENT), 1.0 / math.sqrt(512.0)),
    }
    if with_kv:
        which = range(w.B) if seqs is None else seqs
        out["kv_raw"] = {int(b): kv_rows(w, int(b), int(lens[b])) for b in which}
    return out


def garbage_pool_bits(w: Workload, num_pages: int, width: int) -> np.ndarray:
    """Finite filler for every cache slot before real rows are written, so a
    kernel that reads past a sequence end sees non-zero data."""
    return _normal_bf16(_rng(w.seed, _S_POOL, width), (num_pages, PAGE, width), 4.0)
