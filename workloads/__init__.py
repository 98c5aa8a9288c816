"""Seeded synthetic inputs for page-selective sparse paged decode attention.

This module holds input generation only: shapes, seeds, random draws, the
fp32 -> bf16 storage cast of the drawn values and the physical block layout.
It contains none of the method's arithmetic (no summaries, scores, selection
or attention), so both the CPU oracle and the CUDA path may consume it.

Workloads (shapes follow the five decode configurations the project measures):

  1  tiny GQA, fp32:  B=1, H_q=4, H_kv=1, D=64, page 16, seq 256 (16 pages),
     32 physical blocks, block table = first 16 entries of a seeded permutation
     of range(32); K, V, q ~ N(0,1); budget 4 pages; no append.
  2  Llama-3.1-8B-shaped layer, bf16: B=1, H_q=32, H_kv=8, D=128, page 16,
     context 32768, 8 hot pages per KV head, budget 128 pages, then 64 appended
     decode tokens (fresh k, v ~ N(0,1) and a fresh q each step).
  3  batched ragged, bf16: B=64, same heads, context ~ U[8192, 65536] per
     sequence, 16 hot pages per KV head, one shuffled physical pool, budget
     max(4, ceil(0.05 * pages)).
  4  long context, bf16: B=1, context 1,048,576 (65,536 pages), 32 hot pages
     per KV head at pages 1 + floor(j * (P - 2) / 32), budget 128 pages.
  5  MLA latent, bf16: B=16, H_q=128 over one latent head of 576 dims (value =
     first 512 dims), page 64, context 131072, 8 hot pages, budget 5 % of pages.

Hot pages (the construction quoted with the decode configurations): for a hot
page of KV head h every key of that head is 0.5 * N(0,1) + 2 * u_h, with u_h a
seeded unit vector; every query head of h's group gets q = u_h + 0.3 * N(0,1).
u_h is drawn per (sequence, KV head).

Reproducibility: every draw comes from ``numpy.random.default_rng`` seeded
with a tuple that names what it draws, so a consumer can regenerate one
sequence, or one token chunk of it, without drawing the rest.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

# token chunk granularity of the key/value draws (a multiple of every page size)
CHUNK_TOKENS = 4096

_STREAM_META, _STREAM_K, _STREAM_V, _STREAM_APPEND_K, _STREAM_APPEND_V, _STREAM_APPEND_Q = range(6)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest even) and return the bit patterns as uint16.

    This is the storage cast of the drawn inputs ("drawn as N(0,1) fp32 then cast").
    Inputs are finite by construction, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    t = u >> np.uint32(16)
    t &= np.uint32(1)
    t += np.uint32(0x7FFF)
    t += u
    t >>= np.uint32(16)
    return t.astype(np.uint16)


@dataclass
class Workload:
    """One decode workload: geometry, lengths, budgets, layout and seeds."""

    name: str
    seed: int
    dtype: str                 # "f32" or "bf16" (storage type of q, K, V, summaries, out)
    B: int
    H_q: int
    H_kv: int
    D: int                     # key dim
    D_v: int                   # value dim
    page_size: int
    seq_lens: np.ndarray       # int32 [B], context before any append
    budgets: np.ndarray        # int32 [B], pages per (sequence, KV head)
    n_hot: int
    hot_rule: str              # "random" or "spread"
    appends: int = 0           # decode tokens appended after the prefill (per sequence)
    latent: bool = False       # MLA: one latent head, value = first D_v key dims
    pool_slack: int = 0        # extra physical blocks in the pool beyond what is needed
    block_table: np.ndarray = field(default=None, repr=False)   # int32 [B, max_pages]
    num_blocks: int = 0
    max_pages: int = 0

    def __post_init__(self):
        self.seq_lens = np.asarray(self.seq_lens, dtype=np.int32)
        self.budgets = np.asarray(self.budgets, dtype=np.int32)
        if self.block_table is None:
            self._build_block_table()

    # ---- geometry ------------------------------------------------------------------
    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def final_lens(self) -> np.ndarray:
        return self.seq_lens + self.appends

    def pages(self, lens=None) -> np.ndarray:
        lens = self.seq_lens if lens is None else np.asarray(lens)
        return (lens + self.page_size - 1) // self.page_size

    @property
    def b_max(self) -> int:
        return int(self.budgets.max())

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def storage_np(self):
        return np.float32 if self.dtype == "f32" else np.uint16

    def _build_block_table(self):
        """Shuffled physical pool: every logical page of every sequence (up to its final
        length) gets a distinct physical block drawn from one seeded permutation."""
        cap_pages = self.pages(self.final_lens)
        self.max_pages = int(cap_pages.max())
        need = int(cap_pages.sum())
        if self.num_blocks == 0:
            self.num_blocks = need + self.pool_slack
        rng = np.random.default_rng([self.seed, _STREAM_META, 1 << 20])
        perm = rng.permutation(self.num_blocks).astype(np.int32)
        bt = np.full((self.B, self.max_pages), -1, dtype=np.int32)
        off = 0
        for i in range(self.B):
            n = int(cap_pages[i])
            bt[i, :n] = perm[off:off + n]
            off += n
        self.block_table = bt

    # ---- per-sequence seeded draws ------------------------------------------------
    def _meta_rng(self, i: int, what: int):
        return np.random.default_rng([self.seed, _STREAM_META, i, what])

    def hot_pages(self, i: int) -> np.ndarray:
        """int [H_kv, n_hot] logical hot pages of sequence i, per KV head (from pages 1..P-2)."""
        P = int(self.pages()[i])
        out = np.zeros((self.H_kv, self.n_hot), dtype=np.int64)
        if self.n_hot == 0 or P < 3:
            return out[:, :0]
        inner = P - 2
        n = min(self.n_hot, inner)
        if self.hot_rule == "spread":
            row = 1 + (np.arange(n) * inner) // n
            out = np.tile(row, (self.H_kv, 1))
        else:
            rng = self._meta_rng(i, 1)
            out = np.stack([1 + np.sort(rng.choice(inner, size=n, replace=False))
                            for _ in range(self.H_kv)])
        return out

    def hot_dirs(self, i: int) -> np.ndarray:
        """float32 [H_kv, D] unit vectors u_h of sequence i."""
        rng = self._meta_rng(i, 2)
        u = rng.standard_normal((self.H_kv, self.D)).astype(np.float64)
        u /= np.linalg.norm(u, axis=1, keepdims=True)
        return u.astype(np.float32)

    def _query_f32(self, rng, i: int) -> np.ndarray:
        noise = rng.standard_normal((self.H_q, self.D), dtype=np.float32)
        if self.n_hot == 0:
            return noise
        u = self.hot_dirs(i)
        return np.repeat(u, self.G, axis=0) + np.float32(0.3) * noise

    def query(self, i: int, step: int = 0) -> np.ndarray:
        """Query [H_q, D] (storage dtype) for sequence i; step > 0 is the step-th appended token."""
        if step == 0:
            rng = self._meta_rng(i, 3)
        else:
            rng = np.random.default_rng([self.seed, _STREAM_APPEND_Q, i, step])
        return self._store(self._query_f32(rng, i))

    def queries(self, step: int = 0) -> np.ndarray:
        return np.stack([self.query(i, step) for i in range(self.B)])

    def _store(self, x: np.ndarray) -> np.ndarray:
        return x.astype(np.float32) if self.dtype == "f32" else f32_to_bf16_bits(x)

    def _chunk_f32(self, stream: int, i: int, c: int, n_tok: int) -> np.ndarray:
        rng = np.random.default_rng([self.seed, stream, i, c])
        return rng.standard_normal((n_tok, self.H_kv, self.D if stream == _STREAM_K else self._v_width),
                                   dtype=np.float32)

    @property
    def _v_width(self) -> int:
        return self.D if self.latent else self.D_v

    def keys_f32(self, i: int, t0: int, t1: int) -> np.ndarray:
        """Pre-cast keys of sequence i for tokens [t0, t1), hot pages applied, float32 [n, H_kv, D]."""
        ps = self.page_size
        out = np.empty((t1 - t0, self.H_kv, self.D), dtype=np.float32)
        c0, c1 = t0 // CHUNK_TOKENS, (t1 - 1) // CHUNK_TOKENS
        for c in range(c0, c1 + 1):
            a, z = c * CHUNK_TOKENS, (c + 1) * CHUNK_TOKENS
            blk = self._chunk_f32(_STREAM_K, i, c, CHUNK_TOKENS)
            lo, hi = max(a, t0), min(z, t1)
            out[lo - t0:hi - t0] = blk[lo - a:hi - a]
        hot = self.hot_pages(i)
        if hot.size:
            u = self.hot_dirs(i)
            for h in range(self.H_kv):
                for p in hot[h]:
                    lo, hi = max(p * ps, t0), min((p + 1) * ps, t1)
                    if lo < hi:
                        out[lo - t0:hi - t0, h] = np.float32(0.5) * out[lo - t0:hi - t0, h] + np.float32(2.0) * u[h]
        return out

    def values_f32(self, i: int, t0: int, t1: int) -> np.ndarray:
        """Pre-cast values of sequence i for tokens [t0, t1), float32 [n, H_kv, D_v].
        For a latent (MLA) workload the value is the first D_v dims of the latent key."""
        if self.latent:
            return self.keys_f32(i, t0, t1)[..., :self.D_v]
        out = np.empty((t1 - t0, self.H_kv, self.D_v), dtype=np.float32)
        c0, c1 = t0 // CHUNK_TOKENS, (t1 - 1) // CHUNK_TOKENS
        for c in range(c0, c1 + 1):
            a = c * CHUNK_TOKENS
            blk = self._chunk_f32(_STREAM_V, i, c, CHUNK_TOKENS)
            lo, hi = max(a, t0), min(a + CHUNK_TOKENS, t1)
            out[lo - t0:hi - t0] = blk[lo - a:hi - a]
        return out

    def keys(self, i: int, t0: int = 0, t1: int | None = None) -> np.ndarray:
        """Prefill keys of sequence i (storage dtype) for tokens [t0, t1) (default: its context)."""
        t1 = int(self.seq_lens[i]) if t1 is None else t1
        return self._store(self.keys_f32(i, t0, t1))

    def values(self, i: int, t0: int = 0, t1: int | None = None) -> np.ndarray:
        t1 = int(self.seq_lens[i]) if t1 is None else t1
        return self._store(self.values_f32(i, t0, t1))

    def append_token(self, i: int, step: int):
        """(k_new [H_kv, D], v_new [H_kv, D_v]) of the step-th appended token (step >= 1), storage dtype."""
        rk = np.random.default_rng([self.seed, _STREAM_APPEND_K, i, step])
        k = rk.standard_normal((self.H_kv, self.D), dtype=np.float32)
        if self.latent:
            v = k[:, :self.D_v]
        else:
            rv = np.random.default_rng([self.seed, _STREAM_APPEND_V, i, step])
            v = rv.standard_normal((self.H_kv, self.D_v), dtype=np.float32)
        return self._store(k), self._store(v)

    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    # ---- packed prefill arrays -----------------------------------------------------
    def packed_prefill(self, seqs=None, threads: int | None = None):
        """Packed ragged prefill: (k [T, H_kv, D], v [T, H_kv, D_v] or None for latent,
        cu [len(seqs)+1] int32). Sequences are drawn in parallel threads."""
        seqs = list(range(self.B)) if seqs is None else list(seqs)
        lens = [int(self.seq_lens[i]) for i in seqs]
        cu = np.zeros(len(seqs) + 1, dtype=np.int64)
        cu[1:] = np.cumsum(lens)
        T = int(cu[-1])
        k = np.empty((T, self.H_kv, self.D), dtype=self.storage_np)
        v = None if self.latent else np.empty((T, self.H_kv, self.D_v), dtype=self.storage_np)

        def work(job):
            j, t0, t1 = job
            i = seqs[j]
            base = int(cu[j])
            k[base + t0:base + t1] = self.keys(i, t0, t1)
            if v is not None:
                v[base + t0:base + t1] = self.values(i, t0, t1)

        jobs = []
        for j, n in enumerate(lens):
            for t0 in range(0, n, CHUNK_TOKENS):
                jobs.append((j, t0, min(n, t0 + CHUNK_TOKENS)))
        nthreads = threads or min(32, os.cpu_count() or 1)
        if len(jobs) == 1 or nthreads == 1:
            for jb in jobs:
                work(jb)
        else:
            with ThreadPoolExecutor(nthreads) as ex:
                list(ex.map(work, jobs))
        return k, v, cu.astype(np.int32)


def _budget_frac(P: np.ndarray, frac: float, floor: int) -> np.ndarray:
    # ceil(frac * P) with the stated minimum; computed in integers for frac = 5 %.
    num = int(round(frac * 100))
    return np.maximum(floor, (P * num + 99) // 100).astype(np.int32)


def config(idx: int) -> Workload:
    """The five named decode workloads at their full sizes."""
    if idx == 1:
        return Workload("tiny-gqa-f32", 1001, "f32", B=1, H_q=4, H_kv=1, D=64, D_v=64, page_size=16,
                        seq_lens=[256], budgets=[4], n_hot=0, hot_rule="random", num_blocks=32)
    if idx == 2:
        return Workload("llama8b-layer-b1-32k+64", 1002, "bf16", B=1, H_q=32, H_kv=8, D=128, D_v=128,
                        page_size=16, seq_lens=[32768], budgets=[128], n_hot=8, hot_rule="random",
                        appends=64)
    if idx == 3:
        rng = np.random.default_rng([1003, _STREAM_META, 1 << 21])
        lens = rng.integers(8192, 65536, size=64, endpoint=True).astype(np.int32)
        P = (lens + 15) // 16
        return Workload("batched-ragged-b64-8k..64k-5pct", 1003, "bf16", B=64, H_q=32, H_kv=8, D=128,
                        D_v=128, page_size=16, seq_lens=lens, budgets=_budget_frac(P, 0.05, 4),
                        n_hot=16, hot_rule="random")
    if idx == 4:
        return Workload("long-1m-b1", 1004, "bf16", B=1, H_q=32, H_kv=8, D=128, D_v=128, page_size=16,
                        seq_lens=[1 << 20], budgets=[128], n_hot=32, hot_rule="spread")
    if idx == 5:
        P = np.full(16, 131072 // 64)
        return Workload("mla-b16-128k-5pct", 1005, "bf16", B=16, H_q=128, H_kv=1, D=576, D_v=512,
                        page_size=64, seq_lens=np.full(16, 131072), budgets=_budget_frac(P, 0.05, 4),
                        n_hot=8, hot_rule="random", latent=True)
    raise ValueError(f"unknown workload {idx}")


def reduced(idx: int, seed_offset: int = 0) -> Workload:
    """A reduced-size workload of the same structure as workload ``idx``: several score chunks,
    several decode splits and a ragged tail page, small enough for the oracle to finish in seconds."""
    s = 2000 + idx + seed_offset
    if idx == 1:
        w = config(1)
        w.seed = s
        w._build_block_table()
        return w
    if idx == 2:
        return Workload("llama8b-layer-b1-reduced", s, "bf16", B=1, H_q=32, H_kv=8, D=128, D_v=128,
                        page_size=16, seq_lens=[3000 + 7], budgets=[40], n_hot=8, hot_rule="random",
                        appends=21, pool_slack=9)
    if idx == 3:
        rng = np.random.default_rng([s, _STREAM_META, 1 << 21])
        lens = rng.integers(200, 4100, size=6, endpoint=True).astype(np.int32)
        P = (lens + 15) // 16
        return Workload("batched-ragged-reduced", s, "bf16", B=6, H_q=32, H_kv=8, D=128, D_v=128,
                        page_size=16, seq_lens=lens, budgets=_budget_frac(P, 0.05, 4), n_hot=4,
                        hot_rule="random", pool_slack=13)
    if idx == 4:
        return Workload("long-reduced", s, "bf16", B=1, H_q=32, H_kv=8, D=128, D_v=128, page_size=16,
                        seq_lens=[9000 * 16 + 5], budgets=[128], n_hot=32, hot_rule="spread")
    if idx == 5:
        lens = np.array([64 * 200 + 17, 64 * 57, 64 * 311 + 63])
        P = (lens + 63) // 64
        return Workload("mla-reduced", s, "bf16", B=3, H_q=128, H_kv=1, D=576, D_v=512, page_size=64,
                        seq_lens=lens, budgets=_budget_frac(P, 0.05, 4), n_hot=8, hot_rule="random",
                        latent=True, pool_slack=5)
    raise ValueError(idx)


def prefix(w: Workload, n: int) -> Workload:
    """The first n sequences of workload w (same seeds, so the same per-sequence draws), with a
    physical pool of their own."""
    return Workload(w.name + f"[:{n}]", w.seed, w.dtype, B=n, H_q=w.H_q, H_kv=w.H_kv, D=w.D, D_v=w.D_v,
                    page_size=w.page_size, seq_lens=w.seq_lens[:n], budgets=w.budgets[:n], n_hot=w.n_hot,
                    hot_rule=w.hot_rule, appends=w.appends, latent=w.latent, pool_slack=w.pool_slack)
