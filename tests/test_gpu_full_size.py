"""GPU parity at the full workload sizes, in the launch configuration bench.py times.

The whole batch runs through libpsk exactly as in the benchmark; the fp64 oracle then checks
sampled sequences one by one (every KV head of each): page summaries bit-exact, scores within
the fp32 bound, selected ids exact up to reported near ties, sparse and dense outputs within
the bf16 tolerances. Oracle work is chunked so its fp64 arrays stay a few GB at most.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

from parity import check_output, compare_selection, score_tolerance

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import page_sparse_kv_gb300 as psk  # noqa: E402
from workloads.device import budgets as dev_budgets, from_torch, to_torch, upload  # noqa: E402

PAGE_CHUNK = 4096  # pages per oracle chunk


@pytest.fixture(scope="module", autouse=True)
def _built():
    from page_sparse_kv_gb300.build import build
    build()


def _oracle_summaries_chunked(w, i, n):
    ps = w.page_size
    P = -(-n // ps)
    lo, hi = [], []
    for c0 in range(0, P, PAGE_CHUNK):
        c1 = min(P, c0 + PAGE_CHUNK)
        t0, t1 = c0 * ps, min(n, c1 * ps)
        keys = w.keys(i, t0, t1) if t1 <= int(w.seq_lens[i]) else None
        if keys is None:
            raise AssertionError("chunk past the prefill")
        a, b = O.page_summaries(keys, t1 - t0, ps, w.dtype)
        lo.append(a)
        hi.append(b)
    return np.concatenate(lo), np.concatenate(hi)


def _check_sequences(w, cache, seqs, q_np, sel_np, sc_np, out_np, dense_np, near_budget=0):
    scale = 1.0 / math.sqrt(w.D)
    summ = from_torch(cache.summaries, w.dtype)
    near_total = 0
    for i in seqs:
        n = int(w.seq_lens[i])
        P = -(-n // w.page_size)
        kmin, kmax = _oracle_summaries_chunked(w, i, n)
        blocks = w.block_table[i, :P]
        assert np.array_equal(summ[blocks, :, 0], kmin), f"kmin seq {i}"
        assert np.array_equal(summ[blocks, :, 1], kmax), f"kmax seq {i}"
        s_ref = O.quest_scores(q_np[i], kmin, kmax, w.dtype, scale)
        tol = score_tolerance(q_np[i], kmin, kmax, w.dtype, scale)
        err = np.abs(sc_np[i, :, :P] - s_ref)
        assert np.all(err <= tol), f"seq {i}: score err {err.max():.3e}"
        use = []
        for h in range(w.H_kv):
            ok, near, got, ref = compare_selection(sel_np[i, h], s_ref[h], int(w.budgets[i]))
            assert ok, f"seq {i} head {h}: selection differs beyond near ties"
            near_total += near
            use.append(got)
        keys, vals = w.keys(i), w.values(i)
        ref = O.attend_pages(q_np[i], keys, vals, n, w.page_size, use, w.dtype, scale)
        check_output(out_np[i], ref, w.dtype)
        if dense_np is not None:
            check_output(dense_np[i], O.dense_attention(q_np[i], keys, vals, n, w.page_size, w.dtype, scale), w.dtype)
        del keys, vals
    if near_total:
        print(f"near ties at the cutoff (reported, within 1e-6 relative): {near_total}")
    return near_total


def _run_batch(w, cache, q_np):
    q = to_torch(q_np, w.dtype).cuda()
    scores = torch.full((w.B, w.H_kv, w.max_pages), float("nan"), device="cuda")
    sel = cache.score_select(q, dev_budgets(w), scores_out=scores)
    out = cache.sparse_decode(q, sel)
    dense = cache.dense_decode(q)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    return (sel.cpu().numpy(), scores.cpu().numpy(), from_torch(out.float(), "f32"),
            from_torch(dense.float(), "f32"))


def test_batched_ragged_full_size_sampled():
    """64 sequences, contexts U[8192, 65536], 5 % budgets: the benchmark workload."""
    w = W.config(3)
    cache = upload(w)
    q_np = w.queries()
    sel, sc, out, dense = _run_batch(w, cache, q_np)
    order = np.argsort(w.seq_lens)
    seqs = sorted({int(order[0]), int(order[-1]), 17, 40})
    _check_sequences(w, cache, seqs, q_np, sel, sc, out, dense)
    # every sequence: sink and tail present, count = min(b, P), ascending
    P = (w.seq_lens + 15) // 16
    for i in range(w.B):
        for h in range(w.H_kv):
            row = [int(x) for x in sel[i, h] if x >= 0]
            assert row[0] == 0 and row[-1] == P[i] - 1 and len(row) == min(int(w.budgets[i]), int(P[i]))
            assert row == sorted(set(row))


def test_long_context_full_size():
    """One sequence of 1,048,576 tokens (65,536 pages), budget 128 pages."""
    w = W.config(4)
    cache = upload(w)
    q_np = w.queries()
    sel, sc, out, dense = _run_batch(w, cache, q_np)
    _check_sequences(w, cache, [0], q_np, sel, sc, out, dense)


def test_llama_layer_with_64_appends_full_size():
    """32768-token context, then 64 decode appends each followed by a full step; every step's
    selection and sparse output are checked, the dense output every 16 steps."""
    w = W.config(2)
    cache = upload(w)
    scale = 1.0 / math.sqrt(w.D)
    n0 = int(w.seq_lens[0])
    K = np.empty((n0 + w.appends, w.H_kv, w.D), dtype=w.storage_np)
    V = np.empty((n0 + w.appends, w.H_kv, w.D_v), dtype=w.storage_np)
    K[:n0] = w.keys(0)
    V[:n0] = w.values(0)
    kmin, kmax = O.page_summaries(K, n0, w.page_size, w.dtype)
    kmin, kmax = list(kmin), list(kmax)
    for step in range(1, w.appends + 1):
        k_new, v_new = w.append_token(0, step)
        pos = n0 + step - 1
        cache.append(to_torch(k_new[None], w.dtype).cuda(), to_torch(v_new[None], w.dtype).cuda(),
                     torch.tensor([pos], dtype=torch.int32, device="cuda"),
                     torch.tensor([0, 1], dtype=torch.int32, device="cuda"), 1)
        cache.seq_lens += 1
        K[pos] = k_new
        V[pos] = v_new
        p = pos // w.page_size
        if p == len(kmin):
            kmin.append(k_new.copy())
            kmax.append(k_new.copy())
        else:
            kmin[p], kmax[p] = O.summary_after_append(kmin[p], kmax[p], k_new, pos, w.page_size, w.dtype)
        q_np = w.queries(step)
        q = to_torch(q_np, w.dtype).cuda()
        scores = torch.full((1, w.H_kv, w.max_pages), float("nan"), device="cuda")
        sel = cache.score_select(q, dev_budgets(w), scores_out=scores)
        out = cache.sparse_decode(q, sel)
        dense = cache.dense_decode(q) if step % 16 == 0 else None
        torch.cuda.synchronize()
        n = pos + 1
        P = -(-n // w.page_size)
        lo, hi = np.stack(kmin), np.stack(kmax)
        summ = from_torch(cache.summaries, w.dtype)
        blk = w.block_table[0, p]
        assert np.array_equal(summ[blk, :, 0], lo[p]) and np.array_equal(summ[blk, :, 1], hi[p])
        s_ref = O.quest_scores(q_np[0], lo, hi, w.dtype, scale)
        sc = scores.cpu().numpy()[0, :, :P]
        assert np.all(np.abs(sc - s_ref) <= score_tolerance(q_np[0], lo, hi, w.dtype, scale))
        sel_np = sel.cpu().numpy()[0]
        use = []
        for h in range(w.H_kv):
            ok, near, got, ref = compare_selection(sel_np[h], s_ref[h], int(w.budgets[0]))
            assert ok, f"step {step} head {h}"
            use.append(got)
        check_output(from_torch(out.float(), "f32")[0],
                     O.attend_pages(q_np[0], K, V, n, w.page_size, use, w.dtype, scale), w.dtype)
        if dense is not None:
            check_output(from_torch(dense.float(), "f32")[0],
                         O.dense_attention(q_np[0], K, V, n, w.page_size, w.dtype, scale), w.dtype)
    assert psk.get_device_status(cache.ws) == 0


def test_mla_full_size_sampled():
    """16 sequences of 131072 tokens over one 576-dim latent head, 128 query heads, page 64,
    5 % budget: tcgen05 score and decode; two sequences checked (one also dense)."""
    w = W.config(5)
    cache = upload(w)
    q_np = w.queries()
    sel, sc, out, dense = _run_batch(w, cache, q_np)
    scale = 1.0 / math.sqrt(w.D)
    summ = from_torch(cache.summaries, w.dtype)
    for i in (3, 11):
        n = int(w.seq_lens[i])
        P = -(-n // w.page_size)
        kmin, kmax = _oracle_summaries_chunked(w, i, n)
        blocks = w.block_table[i, :P]
        assert np.array_equal(summ[blocks, :, 0], kmin) and np.array_equal(summ[blocks, :, 1], kmax)
        s_ref = O.quest_scores(q_np[i], kmin, kmax, w.dtype, scale)
        tol = score_tolerance(q_np[i], kmin, kmax, w.dtype, scale)
        assert np.all(np.abs(sc[i, :, :P] - s_ref) <= tol)
        ok, near, got, ref = compare_selection(sel[i, 0], s_ref[0], int(w.budgets[i]))
        assert ok, f"seq {i}: selection differs beyond near ties"
        keys = w.keys(i)
        vals = keys[..., :w.D_v]
        check_output(out[i], O.attend_pages(q_np[i], keys, vals, n, w.page_size, [got], w.dtype, scale), w.dtype)
        if i == 3:
            check_output(dense[i], O.dense_attention(q_np[i], keys, vals, n, w.page_size, w.dtype, scale), w.dtype)
