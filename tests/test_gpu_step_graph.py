"""GPU parity of the decode step exactly as bench.py times it: one CUDA graph in which the decode
append runs on a side stream beside score + select (no scores_out, so the always-kept pages'
summaries are not read), and the sparse decode joins both (page_sparse_kv_gb300.step).

  * The batched workload at full size (64 sequences, 8K-64K tokens, 5 % budgets): the bench's own
    step, which re-appends each sequence's last token in place, replayed several times; sampled
    sequences are then checked against the oracle (summaries bit-exact, selected ids exact up to
    reported near ties, outputs within the bf16 tolerances) and every row's structure.
  * The Llama-3.1-8B-shaped layer at full size with its 64 decode appends done by graph
    replays: each replay takes the step's new token and query, copies the sequence length to the
    append position and advances it inside the graph, so the new token lands in the tail page
    while score + select runs beside it; after every replay the tail page's summary, the selected
    ids and the output are checked against the oracle fed the same tokens.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

from parity import check_output, compare_selection

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import page_sparse_kv_gb300 as psk  # noqa: E402
from page_sparse_kv_gb300.step import DecodeStep, capture  # noqa: E402
from workloads.device import budgets as dev_budgets, from_torch, to_torch, upload  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from page_sparse_kv_gb300.build import build
    build()


def _calls(w, cache, q, k_new, v_new, start, cu, bud, sel, out):
    L = cache.layout

    def append():
        psk.kv_append_and_summarize(L, k_new, v_new, start, cu, 1, cache.k_cache, cache.v_cache, cache.summaries,
                                    cache.block_table, cache.ws)

    def score():
        psk.page_score_select(L, q, cache.summaries, cache.block_table, cache.seq_lens, bud, w.b_max, cache.scale,
                              sel, cache.ws)

    def decode():
        psk.sparse_paged_decode(L, q, cache.k_cache, cache.v_cache, cache.block_table, cache.seq_lens, sel, w.b_max,
                                cache.scale, out, cache.ws)

    return append, score, decode


def test_benchmarked_step_graph_batched_full_size():
    w = W.config(3)
    cache = upload(w)
    dev = cache.device
    B = w.B
    lens = w.seq_lens.astype(np.int64)
    k_last = np.stack([w.keys(i, int(lens[i]) - 1, int(lens[i]))[0] for i in range(B)])
    v_last = np.stack([w.values(i, int(lens[i]) - 1, int(lens[i]))[0] for i in range(B)])
    q_np = w.queries()
    q = to_torch(q_np, w.dtype).to(dev)
    k_new, v_new = to_torch(k_last, w.dtype).to(dev), to_torch(v_last, w.dtype).to(dev)
    start = torch.from_numpy((lens - 1).astype(np.int32)).to(dev)
    cu = torch.arange(B + 1, dtype=torch.int32, device=dev)
    sel = torch.full((B, w.H_kv, w.b_max), -7, dtype=torch.int32, device=dev)
    out = torch.full((B, w.H_q, w.D_v), float("nan"), dtype=cache.dtype, device=dev)
    step = DecodeStep(*_calls(w, cache, q, k_new, v_new, start, cu, dev_budgets(w), sel, out))
    g = capture(step.launch)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    sel_np = sel.cpu().numpy()
    out_np = from_torch(out.float(), "f32")
    summ = from_torch(cache.summaries, w.dtype)
    scale = 1.0 / math.sqrt(w.D)
    order = np.argsort(w.seq_lens)
    for i in sorted({int(order[0]), int(order[-1]), 5, 33}):
        n = int(lens[i])
        P = -(-n // w.page_size)
        keys, vals = w.keys(i), w.values(i)
        kmin, kmax = O.page_summaries(keys, n, w.page_size, w.dtype)
        blocks = w.block_table[i, :P]
        assert np.array_equal(summ[blocks, :, 0], kmin) and np.array_equal(summ[blocks, :, 1], kmax), f"seq {i}"
        s_ref = O.quest_scores(q_np[i], kmin, kmax, w.dtype, scale)
        use = []
        for h in range(w.H_kv):
            ok, _, got, ref = compare_selection(sel_np[i, h], s_ref[h], int(w.budgets[i]))
            assert ok, f"seq {i} head {h}: selected {got[:8]}... vs oracle {ref[:8]}..."
            use.append(got)
        check_output(out_np[i], O.attend_pages(q_np[i], keys, vals, n, w.page_size, use, w.dtype, scale), w.dtype)
        del keys, vals
    Ps = (lens + w.page_size - 1) // w.page_size
    for i in range(B):
        for h in range(w.H_kv):
            row = [int(x) for x in sel_np[i, h] if x >= 0]
            assert row[0] == 0 and row[-1] == Ps[i] - 1 and len(row) == min(int(w.budgets[i]), int(Ps[i]))
            assert row == sorted(set(row)) and np.all(sel_np[i, h, len(row):] == -1)


def test_llama_layer_64_appends_by_graph_replay_full_size():
    w = W.config(2)
    cache = upload(w)
    dev = cache.device
    scale = 1.0 / math.sqrt(w.D)
    n0 = int(w.seq_lens[0])
    K = np.empty((n0 + w.appends, w.H_kv, w.D), dtype=w.storage_np)
    V = np.empty((n0 + w.appends, w.H_kv, w.D_v), dtype=w.storage_np)
    K[:n0] = w.keys(0)
    V[:n0] = w.values(0)
    kmin, kmax = O.page_summaries(K, n0, w.page_size, w.dtype)
    kmin, kmax = list(kmin), list(kmax)
    q = torch.empty(1, w.H_q, w.D, dtype=cache.dtype, device=dev)
    k_new = torch.empty(1, w.H_kv, w.D, dtype=cache.dtype, device=dev)
    v_new = torch.empty(1, w.H_kv, w.D_v, dtype=cache.dtype, device=dev)
    start = torch.zeros(1, dtype=torch.int32, device=dev)
    cu = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    sel = torch.full((1, w.H_kv, w.b_max), -7, dtype=torch.int32, device=dev)
    out = torch.empty(1, w.H_q, w.D_v, dtype=cache.dtype, device=dev)
    step = DecodeStep(*_calls(w, cache, q, k_new, v_new, start, cu, dev_budgets(w), sel, out))

    def advance_and_step():
        # the append position is the length before this token; the length then counts it
        start.copy_(cache.seq_lens)
        cache.seq_lens.add_(1)
        step.launch()

    # capture() runs the step once to warm up: that run is the first append, with step 1's inputs
    k1, v1 = w.append_token(0, 1)
    k_new.copy_(to_torch(k1[None], w.dtype))
    v_new.copy_(to_torch(v1[None], w.dtype))
    q.copy_(to_torch(w.queries(1), w.dtype))
    g = capture(advance_and_step)
    torch.cuda.synchronize()
    for step_i in range(1, w.appends + 1):
        k_t, v_t = w.append_token(0, step_i)
        q_np = w.queries(step_i)
        if step_i > 1:
            k_new.copy_(to_torch(k_t[None], w.dtype))
            v_new.copy_(to_torch(v_t[None], w.dtype))
            q.copy_(to_torch(q_np, w.dtype))
            g.replay()
        torch.cuda.synchronize()
        pos = n0 + step_i - 1
        K[pos], V[pos] = k_t, v_t
        p = pos // w.page_size
        if p == len(kmin):
            kmin.append(k_t.copy())
            kmax.append(k_t.copy())
        else:
            kmin[p], kmax[p] = O.summary_after_append(kmin[p], kmax[p], k_t, pos, w.page_size, w.dtype)
        assert int(cache.seq_lens[0].item()) == pos + 1
        n = pos + 1
        lo, hi = np.stack(kmin), np.stack(kmax)
        summ = from_torch(cache.summaries, w.dtype)
        blk = w.block_table[0, p]
        assert np.array_equal(summ[blk, :, 0], lo[p]) and np.array_equal(summ[blk, :, 1], hi[p]), f"step {step_i}"
        s_ref = O.quest_scores(q_np[0], lo, hi, w.dtype, scale)
        sel_np = sel.cpu().numpy()[0]
        use = []
        for h in range(w.H_kv):
            ok, _, got, ref = compare_selection(sel_np[h], s_ref[h], int(w.budgets[0]))
            assert ok, f"step {step_i} head {h}"
            use.append(got)
        check_output(from_torch(out.float(), "f32")[0],
                     O.attend_pages(q_np[0], K, V, n, w.page_size, use, w.dtype, scale), w.dtype)
    assert psk.get_device_status(cache.ws) == 0
    # the incremental summaries equal a rebuild over every token
    n = n0 + w.appends
    lo, hi = O.page_summaries(K, n, w.page_size, w.dtype)
    P = -(-n // w.page_size)
    summ = from_torch(cache.summaries, w.dtype)
    blocks = w.block_table[0, :P]
    assert np.array_equal(summ[blocks, :, 0], lo) and np.array_equal(summ[blocks, :, 1], hi)
