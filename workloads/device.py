"""Put a seeded workload on the GPU: tensors from the generator, cache filled through libpsk.

Input plumbing only: the prefill itself runs in the library's append kernel.
"""
from __future__ import annotations

import numpy as np
import torch

from . import Workload


def to_torch(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Host tensor from generator output (fp32 values or bf16 bit patterns), no copy of values."""
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def from_torch(t: torch.Tensor, dtype: str) -> np.ndarray:
    """Inverse of to_torch (result on the host)."""
    t = t.detach().cpu().contiguous()
    if dtype == "f32":
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def layout_of(w: Workload):
    from page_sparse_kv_gb300 import PSK_BF16, PSK_F32, Layout
    return Layout(w.B, w.H_q, w.H_kv, w.D, w.D_v, w.page_size, w.num_blocks, w.max_pages,
                  PSK_F32 if w.dtype == "f32" else PSK_BF16, 1 if w.latent else 0)


def upload(w: Workload, device="cuda", junk: float | None = 1.0e4, group_tokens: int = 1 << 24):
    """A PagedKVCache holding workload ``w`` after its prefill. Sequences are drawn and
    appended in groups of about ``group_tokens`` tokens to bound host memory."""
    from page_sparse_kv_gb300.cache import PagedKVCache
    cache = PagedKVCache(layout_of(w), w.block_table, w.b_max, device=device, junk=junk)
    dev = cache.device
    lens = w.seq_lens.astype(np.int64)
    i = 0
    while i < w.B:
        j, tok = i, 0
        while j < w.B and (j == i or tok + lens[j] <= group_tokens):
            tok += lens[j]
            j += 1
        seqs = list(range(i, j))
        k, v, cu_part = w.packed_prefill(seqs)
        cu = np.zeros(w.B + 1, dtype=np.int32)
        n = np.zeros(w.B, dtype=np.int64)
        n[i:j] = lens[i:j]
        cu[1:] = np.cumsum(n)
        kt = to_torch(k, w.dtype).to(dev)
        vt = None if v is None else to_torch(v, w.dtype).to(dev)
        start = torch.zeros(w.B, dtype=torch.int32, device=dev)
        cache.append(kt, vt, start, torch.from_numpy(cu).to(dev), int(lens[i:j].max()))
        del kt, vt
        i = j
    cache.seq_lens.copy_(torch.from_numpy(w.seq_lens.astype(np.int32)).to(dev))
    return cache


def queries(w: Workload, step: int = 0, device="cuda") -> torch.Tensor:
    return to_torch(w.queries(step), w.dtype).to(device)


def budgets(w: Workload, device="cuda") -> torch.Tensor:
    return torch.from_numpy(w.budgets.astype(np.int32)).to(device)
