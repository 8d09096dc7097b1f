"""One MLA decode step over a resident paged latent cache, through the C ABI:
absorb the query (W_UK), latent attention with split-KV, then the combine
and the value out-projection (W_UV), fused into one launch by default.
Buffers are allocated once, at construction; a step over fixed input buffers
can be recorded once as a CUDA graph and replayed, which removes the host
launch overhead of the calls."""
from __future__ import annotations

import torch

from . import _lib as L


class MLADecodeStep:
    """q_len > 1: that many query tokens per sequence (the newest cache
    positions, causal); queries are [B,q_len,H,...] and the output
    [B,q_len,H,128].  The page table and lengths passed to a call are the B
    sequences'; the step expands them into B*q_len rows (expand_rows), whose
    lengths are also what mla_rope_q needs to rotate the queries.
    fused=False runs mla_split_kv_combine and mla_out_proj as two launches
    instead of mla_combine_out_proj."""

    def __init__(self, B, H, max_pages_per_seq, num_pages, kv_dtype="bf16", out_dtype="f32",
                 num_splits=0, device="cuda", q_len=1, fused=True):
        rows = B * q_len
        self.q_len = q_len
        self.fused = fused
        self.p_seq = L.make_params(B, H, max_pages_per_seq, num_pages, kv_dtype, out_dtype)
        self.p = L.make_params(rows, H, max_pages_per_seq, num_pages, kv_dtype, out_dtype)
        self.num_splits = L.mla_decode_num_splits(self.p, num_splits)
        if self.num_splits < 1:
            raise L.MLAError(L.MLA_ERR_INVALID_ARG, "MLADecodeStep")
        ws = L.mla_decode_workspace_size(self.p, self.num_splits)
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=device)
        self.q_lat = torch.empty(rows, H, 512, dtype=torch.bfloat16, device=device)
        self.o_lat = torch.empty(rows, H, 512, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(rows, H, dtype=torch.float32, device=device)
        odt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
        self.out = torch.empty(rows, H, 128, dtype=odt, device=device)
        if q_len > 1:
            self.table_rows = torch.empty(rows, max_pages_per_seq, dtype=torch.int32, device=device)
            self.lens_rows = torch.empty(rows, dtype=torch.int32, device=device)

    def expand_rows(self, page_table, seq_lens, stream=None):
        """Page table and lengths of the B*q_len rows (the inputs themselves
        when q_len == 1)."""
        if self.q_len == 1:
            return page_table, seq_lens
        L.mla_multi_token_expand(self.p_seq, self.q_len, page_table, seq_lens, self.table_rows, self.lens_rows,
                                 stream)
        return self.table_rows, self.lens_rows

    def __call__(self, q_nope, q_pe, w_uk, w_uv, ckv, kpe, kv_scale, page_table, seq_lens, stream=None):
        p, G = self.p, self.num_splits
        page_table, seq_lens = self.expand_rows(page_table, seq_lens, stream)
        L.mla_absorb_q(p, q_nope, w_uk, self.q_lat, stream)
        L.mla_decode(p, self.q_lat, q_pe, ckv, kpe, kv_scale, page_table, seq_lens, G,
                     self.workspace, self.o_lat, self.lse, stream)
        if self.fused:
            L.mla_combine_out_proj(p, self.workspace, G, seq_lens, self.o_lat, w_uv, self.out, self.lse, stream)
        else:
            L.mla_split_kv_combine(p, self.workspace, G, self.o_lat, self.lse, stream)
            L.mla_out_proj(p, self.o_lat, w_uv, self.out, stream)
        if self.q_len > 1:
            return self.out.view(-1, self.q_len, *self.out.shape[1:])
        return self.out

    def capture(self, *inputs):
        """Record one step over these input buffers (the arguments of
        __call__, which must stay allocated and at the same addresses) as a
        CUDA graph; replay() then runs it on the current stream."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self(*inputs)  # warm-up outside the capture (first-call set-up)
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self(*inputs)
        return self.graph

    def replay(self):
        self.graph.replay()
        if self.q_len > 1:
            return self.out.view(-1, self.q_len, *self.out.shape[1:])
        return self.out

    def status(self, clear=False):
        return L.mla_workspace_status(self.workspace, clear)
