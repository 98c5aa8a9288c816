"""A paged KV cache with per-page key summaries, kept on one GPU.

PyTorch allocates the buffers; every write into them (prefill, decode append, summary
refresh) and every read for scoring and attention goes through libpsk's kernels.
The layout is vLLM's: K and V are [num_blocks, page_size, H_kv, D] each (the two halves of
[2, num_blocks, page_size, H_kv, D]), plus a block table [B, max_pages] mapping logical
pages to physical blocks (EntmaxKV README, introduction; its PagedKVCache(page_size,
max_seq_len).initialize(k, v, seq_lens) plays the same role).
"""
from __future__ import annotations

import math

import torch

from . import (PSK_F32, Layout, dense_paged_decode, kv_append_and_summarize, make_workspace,
               page_score_select, sparse_paged_decode)


class PagedKVCache:
    def __init__(self, layout: Layout, block_table, b_max: int, device="cuda", junk: float | None = None):
        """layout: geometry; block_table: int32 [B, max_pages] (host or device); b_max: largest
        per-sequence page budget that will be requested. ``junk`` fills the cache before use
        (so slots past seq_len hold a recognisable value); default leaves it uninitialised."""
        self.layout = layout
        self.b_max = int(b_max)
        self.device = torch.device(device)
        dt = torch.float32 if layout.dtype == PSK_F32 else torch.bfloat16
        self.dtype = dt
        L = layout
        alloc = torch.empty if junk is None else (lambda *s, **kw: torch.full(s, junk, **kw))
        self.k_cache = alloc(L.num_blocks, L.page_size, L.num_kv_heads, L.head_dim, dtype=dt, device=self.device)
        self.v_cache = None if L.latent else alloc(L.num_blocks, L.page_size, L.num_kv_heads, L.v_head_dim,
                                                   dtype=dt, device=self.device)
        self.summaries = torch.zeros(L.num_blocks, L.num_kv_heads, 2, L.head_dim, dtype=dt, device=self.device)
        self.block_table = torch.as_tensor(block_table, dtype=torch.int32).to(self.device).contiguous()
        self.seq_lens = torch.zeros(L.batch, dtype=torch.int32, device=self.device)
        self.ws = make_workspace(layout, self.b_max, device=self.device)
        self.scale = 1.0 / math.sqrt(L.head_dim)

    # -------------------------------------------------------------------- writes
    def append(self, k_new, v_new, start_pos, cu_new, max_new: int, stream=None):
        """Append packed tokens (see psk_kv_append_and_summarize); does not touch seq_lens."""
        kv_append_and_summarize(self.layout, k_new, v_new, start_pos, cu_new, max_new, self.k_cache, self.v_cache,
                                self.summaries, self.block_table, self.ws, stream=stream)

    def prefill(self, k, v, lens, stream=None):
        """Write whole prompts: k [sum(lens), H_kv, D], v likewise (None for a latent cache), lens [B]."""
        lens = torch.as_tensor(lens, dtype=torch.int32)
        cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(lens, 0)
        start = torch.zeros(len(lens), dtype=torch.int32, device=self.device)
        self.append(k.to(self.device), None if v is None else v.to(self.device), start, cu.to(self.device),
                    int(lens.max()), stream=stream)
        self.seq_lens.copy_(lens.to(self.device))

    # -------------------------------------------------------------------- reads
    def score_select(self, q, budgets, selected=None, scores_out=None, stream=None):
        L = self.layout
        if selected is None:
            selected = torch.empty(L.batch, L.num_kv_heads, self.b_max, dtype=torch.int32, device=self.device)
        page_score_select(L, q, self.summaries, self.block_table, self.seq_lens, budgets, self.b_max, self.scale,
                          selected, self.ws, scores_out=scores_out, stream=stream)
        return selected

    def sparse_decode(self, q, selected, out=None, stream=None):
        L = self.layout
        if out is None:
            out = torch.empty(L.batch, L.num_q_heads, L.v_head_dim, dtype=self.dtype, device=self.device)
        sparse_paged_decode(L, q, self.k_cache, self.v_cache, self.block_table, self.seq_lens, selected, self.b_max,
                            self.scale, out, self.ws, stream=stream)
        return out

    def dense_decode(self, q, out=None, stream=None):
        L = self.layout
        if out is None:
            out = torch.empty(L.batch, L.num_q_heads, L.v_head_dim, dtype=self.dtype, device=self.device)
        dense_paged_decode(L, q, self.k_cache, self.v_cache, self.block_table, self.seq_lens, self.scale, out,
                           self.ws, stream=stream)
        return out
