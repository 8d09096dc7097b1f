"""Test helpers: upload seeded inputs, run the CUDA path through the C ABI,
and an independent statement of the documented KV-partition rule."""
import math

import numpy as np
import torch

PAGE = 64


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def u8_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def i32_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def tol_ok(got, ref, rel, abs_=0.0):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = np.max(np.abs(got - ref))
    bound = rel * np.max(np.abs(ref)) + abs_
    return err <= bound, err, bound


def reference_partition(seq_lens, maxp, G):
    """Split records as the header documents them: flattened pages cut into G
    ranges [floor(wP/G), floor((w+1)P/G)); record w = unit holding the range's
    first page, record G+w = unit holding its last page if another unit."""
    npg = [((n + PAGE - 1) // PAGE) if 1 <= n <= maxp * PAGE else 0 for n in seq_lens]
    start = [0]
    for n in npg:
        start.append(start[-1] + n)
    P = start[-1]
    rec = [(-1, 0, 0, 0)] * (2 * G)
    for w in range(G):
        lo, hi = w * P // G, (w + 1) * P // G
        if lo >= hi:
            continue
        for b, n in enumerate(npg):
            sb, se = start[b], start[b] + n
            if n == 0 or se <= lo or sb >= hi:
                continue
            ub, ue = max(lo, sb), min(hi, se)
            r = (b, ub - sb, ue - sb, int(sb < lo or se > hi))
            if ub == lo:
                rec[w] = r
            elif ue == hi:
                rec[G + w] = r
    return rec, start


def upload_cache(cache):
    if cache["kv_dtype"] == "e4m3":
        return u8_dev(cache["ckv"]), u8_dev(cache["kpe"]), torch.from_numpy(cache["scale"]).cuda()
    return bf16_dev(cache["ckv"]), bf16_dev(cache["kpe"]), None


def sample_pairs(B, H, n_seq, n_head, seed):
    rng = np.random.default_rng(seed)
    bs = sorted(rng.choice(B, size=min(n_seq, B), replace=False).tolist())
    return [(b, int(h)) for b in bs for h in sorted(rng.choice(H, size=min(n_head, H), replace=False))]


def scale():
    return 1.0 / math.sqrt(192.0)
